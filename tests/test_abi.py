"""CPU: the C-ABI library builds, loads and exports every declared symbol;
host-side checks and size queries work without a GPU (no compute calls)."""
import ctypes

import pytest

from block_scaled_moe_expert_gb300 import binding as B
from block_scaled_moe_expert_gb300 import build as BLD


@pytest.fixture(scope="module")
def L():
    BLD.build()
    B._lib = None
    return B.lib()


def test_every_declared_symbol_is_exported(L):
    names = B.header_symbols()
    assert "moe_experts_forward" in names and "moe_prepare_weights" in names
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    assert L.moe_abi_version() == 1
    for code in range(0, 9):
        assert L.moe_status_string(code).decode().startswith("MOE_")
    assert L.moe_status_string(99) == b"MOE_ERR_UNKNOWN"


@pytest.mark.parametrize("fmt,E,H,I", [(0, 8, 4096, 14336), (0, 256, 7168, 2048), (1, 128, 2880, 2880),
                                       (1, 256, 7168, 2048), (0, 8, 256, 128), (2, 128, 2880, 2880),
                                       (2, 256, 7168, 2048)])
def test_sizes_are_consistent(L, fmt, E, H, I):
    n13 = L.moe_prepared_w13_bytes(fmt, E, H, I)
    n2 = L.moe_prepared_w2_bytes(fmt, E, H, I)
    kp1 = -(-H // 128) * 128
    np1 = 2 * (-(-I // 128) * 128)
    kp2 = -(-I // 128) * 128
    np2 = -(-H // 256) * 256
    code13 = E * np1 * (kp1 if fmt == 0 else kp1 // 2)
    code2 = E * np2 * (kp2 if fmt == 0 else kp2 // 2)
    assert code13 <= n13 <= code13 * 1.1 + 2048 and code2 <= n2 <= code2 * 1.1 + 2048
    for T, K in [(1, 8), (128, 8), (4096, 2)]:
        lay = B.MoeLayout()
        assert L.moe_query_workspace_layout(fmt, T, H, I, E, K, ctypes.byref(lay)) == 0
        assert lay.total_bytes == L.moe_workspace_bytes(fmt, T, H, I, E, K)
        offs = sorted([lay.status, lay.counts, lay.offsets, lay.padded_offsets, lay.perm, lay.inv, lay.row_slot,
                       lay.tiles, lay.xq, lay.xsf, lay.act, lay.asf, lay.y])
        assert all(o % 1024 == 0 for o in offs) and len(set(offs)) == len(offs)
        S = T * K
        assert lay.row_capacity >= S and lay.row_capacity % 128 == 0
        assert lay.row_capacity <= S + min(E, S) * 127 + 127
        assert lay.y + 4 * lay.row_capacity * H <= lay.total_bytes
        assert lay.xq_cols == kp1 and lay.act_cols == kp2
        # activation rows: a byte per code, or two e2m1 codes per byte (fmt 2)
        per = 2 if fmt == 2 else 1
        assert lay.xsf >= lay.xq + lay.row_capacity * kp1 // per
        assert lay.asf >= lay.act + lay.row_capacity * kp2 // per
        # monotone in T: a workspace sized for T serves every smaller T
        assert L.moe_workspace_bytes(fmt, T, H, I, E, K) >= L.moe_workspace_bytes(fmt, max(T - 1, 0), H, I, E, K)


@pytest.mark.parametrize("fmt,E,H,I,K", [(0, 8, 200, 128, 2), (0, 8, 256, 192, 2), (1, 8, 250, 128, 2),
                                         (3, 8, 256, 128, 2), (2, 8, 250, 128, 2), (0, 0, 256, 128, 2),
                                         (0, 513, 256, 128, 2),
                                         (0, 8, 64, 128, 2)])
def test_unsupported_shapes_are_refused(L, fmt, E, H, I, K):
    assert L.moe_workspace_bytes(fmt, 16, H, I, E, K) == 0
    assert L.moe_prepared_w13_bytes(fmt, E, H, I) == 0
    st = L.moe_experts_forward(None, None, None, 16, H, I, E, K, fmt, None, None, float("nan"), None, 0, None, None)
    assert st == 2  # MOE_ERR_UNSUPPORTED_SHAPE


def test_argument_checks_before_any_device_call(L):
    nan = float("nan")
    # T < 0, K out of range: invalid argument
    assert L.moe_experts_forward(None, None, None, -1, 256, 128, 8, 2, 0, None, None, nan, None, 0, None, None) == 1
    assert L.moe_experts_forward(None, None, None, 4, 256, 128, 8, 0, 0, None, None, nan, None, 0, None, None) == 1
    assert L.moe_experts_forward(None, None, None, 4, 256, 128, 8, 33, 0, None, None, nan, None, 0, None, None) == 1
    # T == 0: nothing to do, succeeds without touching a device
    assert L.moe_experts_forward(None, None, None, 0, 256, 128, 8, 2, 0, None, None, nan, None, 0, None, None) == 0
    # null pointers with work to do
    assert L.moe_experts_forward(None, None, None, 4, 256, 128, 8, 2, 0, None, None, nan, None, 0, None, None) == 1
    # misaligned pointers
    p = ctypes.c_void_p(0x1001)
    assert L.moe_experts_forward(p, p, p, 4, 256, 128, 8, 2, 0, p, p, nan, p, 1 << 30, p, None) == 5
    # workspace too small
    a = ctypes.c_void_p(0x100000)
    assert L.moe_experts_forward(a, a, a, 4, 256, 128, 8, 2, 0, a, a, nan, a, 16, ctypes.c_void_p(0x200000),
                                 None) == 6
    # the no-allocation forward refuses calls beyond its fixed capacity
    assert L.moe_experts_forward_static(None, None, None, 4096, 7168, 2048, 8, 2, 0, None, None, nan, None,
                                        None) == 6
    assert L.moe_static_workspace_capacity() == 64 << 20
    # ... and checks its arguments in the same order as moe_experts_forward
    assert L.moe_experts_forward_static(None, None, None, 4, 256, 128, 8, 33, 0, None, None, nan, None, None) == 1
    assert L.moe_experts_forward_static(None, None, None, -1, 256, 128, 8, 2, 0, None, None, nan, None, None) == 1
    assert L.moe_experts_forward_static(None, None, None, 4, 200, 128, 8, 2, 0, None, None, nan, None, None) == 2
    assert L.moe_experts_forward_static(None, None, None, 0, 256, 128, 8, 2, 0, None, None, nan, None, None) == 0
    assert L.moe_static_get_device_status(None, None) == 1
    # debug tap: null tap buffer with work to do
    assert L.moe_debug_forward_act_f32(None, None, None, 4, 256, 128, 8, 2, 0, None, None, nan, None, 0, None,
                                       None, 0, None) == 1
    # bounded-wait self-test: null, short or misaligned workspace
    assert L.moe_selftest_wait_timeout(None, 256, None) == 1
    assert L.moe_selftest_wait_timeout(a, 2, None) == 1
    assert L.moe_selftest_wait_timeout(a, 4, None) == 1  # needs the status word and a counter
    assert L.moe_selftest_wait_timeout(ctypes.c_void_p(0x100002), 256, None) == 1
    # prepare (both storages): null / misaligned / unsupported shape
    for fn in (L.moe_prepare_weights, L.moe_prepare_weights_transposed):
        assert fn(0, 8, 256, 128, None, None, None, None, None, 0, None, 0, None) == 1
        assert fn(0, 8, 256, 128, p, p, p, p, p, 1 << 30, p, 1 << 30, None) == 5
        assert fn(0, 8, 200, 128, p, p, p, p, p, 1 << 30, p, 1 << 30, None) == 2


def test_python_refusals_without_gpu():
    import torch
    with pytest.raises(ValueError):
        B.experts_forward(torch.zeros(2, 256), torch.zeros(2, 2, dtype=torch.int32), torch.zeros(2, 2), None)
    with pytest.raises(NotImplementedError):
        B.experts_forward(torch.zeros(2, 256, dtype=torch.bfloat16), None, None, None, activation_scheme="static")


def test_fp4_activation_format_shares_the_fp4_weights(L):
    for E, H, I in [(8, 256, 128), (128, 2880, 2880)]:
        assert L.moe_prepared_w13_bytes(2, E, H, I) == L.moe_prepared_w13_bytes(1, E, H, I) > 0
        assert L.moe_prepared_w2_bytes(2, E, H, I) == L.moe_prepared_w2_bytes(1, E, H, I) > 0
        # the e2m1 activation rows take half the bytes of the e4m3 ones
        assert L.moe_workspace_bytes(2, 4096, H, I, E, 4) < L.moe_workspace_bytes(1, 4096, H, I, E, 4)


def test_python_refuses_fp4_activations_with_fp8_weights():
    with pytest.raises(ValueError):
        B.prepare_weights(dict(fmt="fp8", E=1, H=128, I=128, w13=None, w13_scale=None, w2=None, w2_scale=None),
                          activations="fp4")
    with pytest.raises(ValueError):
        B.prepare_weights(dict(fmt="fp4", E=1, H=128, I=128, w13=None, w13_scale=None, w2=None, w2_scale=None),
                          activations="int8")
