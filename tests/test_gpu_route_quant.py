"""GPU: routing and input quantization are bit-exact against the oracle.

Runs the forward through the C ABI and reads the routing arrays, the grouped
e4m3 rows and their scale exponents back from the workspace.
"""
import numpy as np
import pytest
import torch

from oracle.routing import route
from tests import parity as P

pytestmark = pytest.mark.gpu


def _check_route_quant(wl, r):
    L = P.B.workspace_layout(wl.fmt, wl.T, wl.H, wl.I, wl.E, wl.K)
    ws = r["ws"]
    S, E = wl.S, wl.E
    idx = r["idx"].cpu().numpy()
    ref = route(idx, E, L.row_align)
    get = lambda name, n: P.ws_region(ws, L, name, torch.int32, n).cpu().numpy()
    assert (get("counts", E) == ref["counts"]).all()
    assert (get("offsets", E + 1) == ref["offsets"]).all()
    assert (get("padded_offsets", E + 1) == ref["padded_offsets"]).all()
    assert (get("perm", S) == ref["perm"]).all()
    inv = get("inv", S)
    assert (inv == ref["inv"]).all()
    M = int(ref["padded_offsets"][E])
    assert (get("row_slot", M) == ref["row_slot"]).all()
    # GEMM work lists: 128-row m-tiles and 32-row chunks per expert, their
    # offsets and the expert owning each
    mtiles = -(-ref["counts"] // 128)
    chunks = -(-ref["counts"] // 32)
    mt_off = np.concatenate([[0], np.cumsum(mtiles)])
    ch_off = np.concatenate([[0], np.cumsum(chunks)])
    n_mt, n_ch = int(mt_off[-1]), int(ch_off[-1])
    Mcap = L.row_capacity
    base = 16 + 2 * (E + 1)
    tiles = get("tiles", base + Mcap // 128 + n_ch)
    assert tiles[0] == n_mt and tiles[1] == n_ch
    assert (tiles[16:16 + E + 1] == mt_off).all()
    assert (tiles[16 + E + 1:base] == ch_off).all()
    assert (tiles[base:base + n_mt] == np.repeat(np.arange(E), mtiles)).all()
    assert (tiles[base + Mcap // 128:] == np.repeat(np.arange(E), chunks)).all()

    codes, exps = P.OM.quantize_hidden(P.bits_of(r["hidden"]))
    valid = np.flatnonzero(ref["inv"] >= 0)
    rows = ref["inv"][valid]
    tok = valid // wl.K
    xq = P.ws_region(ws, L, "xq", torch.uint8, L.row_capacity * L.xq_cols).view(L.row_capacity, L.xq_cols)
    xq = xq.cpu().numpy()
    assert (xq[rows, :wl.H] == codes[tok]).all()
    assert (xq[rows, wl.H:] == 0).all()
    words = P.ws_region(ws, L, "xsf", torch.int32, L.row_capacity * L.x_blocks)
    ex = P.sf_exponents(words, L.row_capacity, L.x_blocks)
    assert (ex[rows] == exps[tok]).all()
    return ref


CASES = [
    P.W.WORKLOADS["tiny_fp8"],
    P.W.scaled(P.W.WORKLOADS["dsv3_decode_fp8"], T=512, H=256, I=128),
    P.W.scaled(P.W.WORKLOADS["gptoss_fp8xfp4"], T=333, H=2880, I=128, E=16),
    P.W.scaled(P.W.WORKLOADS["dsv3_decode_fp4_T1"], H=512, I=256),
    # 256 and 264 slots: the single-CTA routing kernel; FP4 decode batch of
    # 256 slots: the quantization kernel also sets up GEMM2's fused combine
    P.W.scaled(P.W.WORKLOADS["dsv3_decode_fp8"], T=32, H=256, I=128),
    P.W.scaled(P.W.WORKLOADS["dsv3_decode_fp8"], T=33, H=256, I=128),
    P.W.scaled(P.W.WORKLOADS["dsv3_decode_fp4_T32"], H=512, I=256),
    # more than 8192 slots: the multi-CTA routing path (10 and 34 chunks of 1024 slots)
    P.W.scaled(P.W.WORKLOADS["dsv3_decode_fp8"], T=1250, H=256, I=128),
    P.W.scaled(P.W.WORKLOADS["gptoss_fp8xfp4"], T=8500, H=256, I=128, E=128),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: f"{w.name}_T{w.T}_E{w.E}")
def test_route_and_quant_bit_exact(wl):
    r = P.run_cuda(wl)
    _check_route_quant(wl, r)
    assert P.B.device_status(r["ws"]) == 0


@pytest.mark.parametrize("T", [40, 5000])
def test_invalid_ids_are_skipped_and_flagged(T):
    wl = P.W.scaled(P.W.WORKLOADS["tiny_fp8"], T=T)
    idx, w = P.W.make_routing(wl, "cuda")
    idx[3, 1] = wl.E + 5
    idx[7, 0] = -9
    r = P.run_cuda(wl, idx=idx, w=w)
    _check_route_quant(wl, r)
    assert P.B.device_status(r["ws"]) & P.B.MOE_DEV_BAD_EXPERT_ID
    assert P.B.device_status(r["ws"]) == 0  # cleared by the read


def _sweep_hidden():
    """Every finite bf16 value, plus every e4m3 rounding tie at amax 448."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = P.OF.bf16_bits_to_f64(bits)
    fin = bits[np.isfinite(v)]
    pos = P.OF.E4M3_TABLE[:0x7F]
    mids = np.concatenate([(pos[1:] + pos[:-1]) / 2, -(pos[1:] + pos[:-1]) / 2])
    mid_bits = (mids.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert (P.OF.bf16_bits_to_f64(mid_bits) == mids).all()
    rng = np.random.default_rng(0)
    rows = []
    H = 1024
    shuffled = fin[rng.permutation(fin.size)]
    pad = (-shuffled.size) % H
    rows.append(np.concatenate([shuffled, np.zeros(pad, np.uint16)]).reshape(-1, H))
    tie = np.full(((mid_bits.size + 126) // 127) * 128, 0, np.uint16)
    amax_bits = np.uint16(np.float32(448.0).view(np.uint32) >> 16)
    for b in range(tie.size // 128):
        chunk = mid_bits[b * 127:(b + 1) * 127]
        tie[b * 128] = amax_bits
        tie[b * 128 + 1:b * 128 + 1 + chunk.size] = chunk
    tie = np.concatenate([tie, np.zeros((-tie.size) % H, np.uint16)]).reshape(-1, H)
    rows.append(tie)
    return np.concatenate(rows)


def test_quantizer_exhaustive_bf16_sweep():
    hb = _sweep_hidden()
    T, H = hb.shape
    wl = P.W.Workload("sweep", T, H, 128, 2, 1, "fp8", "softmax", seed=77)
    hidden = torch.from_numpy(hb.view(np.int16)).view(torch.bfloat16).cuda()
    idx = (torch.arange(T, dtype=torch.int32, device="cuda") % 2).view(T, 1).contiguous()
    w = torch.ones(T, 1, dtype=torch.float32, device="cuda")
    r = P.run_cuda(wl, hidden=hidden, idx=idx, w=w)
    _check_route_quant(wl, r)


@pytest.mark.parametrize("T,fmt,E", [(9, "fp8", 8), (70, "fp8", 8), (9, "fp4", 8), (40, "fp4", 64)])
def test_duplicate_ids_in_one_token(T, fmt, E):
    """A token may name the same expert twice: each pair is routed on its own
    (the routing kernel; for FP4 decode batches the single launch's own
    routing at T=9, and the fused combine at T=40)."""
    wl = P.W.Workload("dups", T, 256, 128, E, 4, fmt, "softmax", seed=55)
    idx, w = P.W.make_routing(wl, "cuda")
    idx[0] = torch.tensor([3, 3, 3, 5], dtype=torch.int32)
    idx[T - 1] = torch.tensor([-1, 2, 2, -1], dtype=torch.int32)
    idx[T // 2] = -1
    r = P.run_cuda(wl, idx=idx, w=w)
    _check_route_quant(wl, r)
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], None)
    P.assert_close(r["out"], ref, f"dups T={T}")
