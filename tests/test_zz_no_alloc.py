"""GPU: the forward that allocates nothing (moe_experts_forward_static).

It serves callers that cannot allocate device memory themselves; its scratch
space is a fixed array inside the library. Called twice in a row through the
C ABI, it must agree with moe_experts_forward (caller-provided workspace) on
the same inputs, within the parity tolerances of the other tests. This file
is collected last on purpose.
"""
import ctypes

import pytest
import torch

from tests import parity as P

pytestmark = pytest.mark.gpu

W = P.W
B = P.B

MOE_ERR_WORKSPACE_TOO_SMALL = 6


def _static_call(wl, r, out):
    p = r["prepared"]
    limit = float("nan") if wl.swiglu_limit is None else wl.swiglu_limit
    return B.lib().moe_experts_forward_static(
        r["hidden"].data_ptr(), r["idx"].data_ptr(), r["w"].data_ptr(), wl.T, wl.H, wl.I, wl.E, wl.K,
        B.FMT[p.fmt], p.w13_prep.data_ptr(), p.w2_prep.data_ptr(), ctypes.c_float(limit), out.data_ptr(),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("wl", [W.WORKLOADS["tiny_fp8"], W.WORKLOADS["dsv3_decode_fp4_T1"],
                                W.Workload("fp4_small_clamp", 24, 256, 128, 8, 2, "fp4", "softmax", seed=41,
                                           swiglu_limit=0.3),
                                W.WORKLOADS["dsv3_decode_fp4xfp4_T1"]],
                         ids=lambda w: w.name)
def test_static_workspace_forward_matches_workspace_forward(wl):
    r = P.run_cuda(wl)
    assert B.lib().moe_workspace_bytes(B.FMT[P.lib_fmt(wl)], wl.T, wl.H, wl.I, wl.E, wl.K) <= \
        B.lib().moe_static_workspace_capacity()
    for call in range(2):
        out = torch.full_like(r["out"], float("nan"))
        assert _static_call(wl, r, out) == 0, call
        torch.cuda.synchronize()
        m = P.compare(out, r["out"].double().cpu().numpy())
        assert m["finite"], (call, m)
        assert m["rel_fro"] <= P.REL_FRO and m["max_excess_over_rms"] <= P.MAX_REL_RMS, (call, m)
        # Same kernels on the same inputs: the results are also bit-identical.
        assert torch.equal(out.view(torch.int16), r["out"].view(torch.int16)), call


def test_static_workspace_refuses_oversized_calls():
    wl = W.scaled(W.WORKLOADS["dsv3_decode_fp8"], E=8, H=7168, I=2048, T=4096, K=2)
    need = B.lib().moe_workspace_bytes(B.FMT[wl.fmt], wl.T, wl.H, wl.I, wl.E, wl.K)
    assert need > B.lib().moe_static_workspace_capacity()
    st = B.lib().moe_experts_forward_static(None, None, None, wl.T, wl.H, wl.I, wl.E, wl.K, B.FMT[wl.fmt], None,
                                            None, ctypes.c_float(float("nan")), None, None)
    assert st == MOE_ERR_WORKSPACE_TOO_SMALL


def test_static_forward_flags_are_readable():
    """A static forward with an out-of-range expert id treats the slot as
    skipped and raises MOE_DEV_BAD_EXPERT_ID in the fixed array's status word,
    which moe_static_get_device_status reads (and clears); the output equals
    the workspace forward's on the same ids."""
    wl = W.Workload("static_bad_id", 8, 256, 128, 8, 2, "fp8", "softmax", seed=43)
    r = P.run_cuda(wl)
    idx = r["idx"].clone()
    idx[3, 1] = wl.E + 5          # out of range: skipped and flagged
    ref = B.experts_forward(r["hidden"], idx, r["w"], r["prepared"], wl.swiglu_limit)
    r2 = dict(r, idx=idx)
    out = torch.full_like(r["out"], float("nan"))
    assert _static_call(wl, r2, out) == 0
    assert B.static_device_status() == B.MOE_DEV_BAD_EXPERT_ID
    assert B.static_device_status() == 0     # read and cleared
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # a clean call leaves no flag
    assert _static_call(wl, r, out) == 0
    assert B.static_device_status() == 0
    assert torch.equal(out.view(torch.int16), r["out"].view(torch.int16))
