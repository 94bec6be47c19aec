"""GPU: the FP4 x FP4 variant (e2m1 activations in 1x32 blocks, both GEMM
operands e2m1) against the oracle run with FP4 activations.

* the input quantization is bit-exact: every valid pair's packed e2m1 codes
  and 1x32 exponents equal the oracle's quantizer on the same bf16 rows;
* the GEMM1 epilogue's requantization is bit-exact on its own fp32 inputs
  (debug tap), codes and exponents;
* the bf16 output meets the method's tolerances against the fp64 oracle on
  tiny, ragged (H = I = 2880), decode and skip-heavy shapes;
* it is a different computation from the e4m3-activation forward on the
  same inputs (the outputs differ), and it replays from a CUDA graph.
"""
import numpy as np
import pytest
import torch

from oracle.routing import route
from tests import parity as P

pytestmark = pytest.mark.gpu

W = P.W
OF = P.OF

CASES = [
    W.Workload("mx_tiny", 16, 256, 128, 8, 2, "fp4", "softmax", seed=41, act_fmt="fp4"),
    W.Workload("mx_ragged_clamp", 100, 2880, 2880, 8, 4, "fp4", "softmax", seed=42, logit_std=1.5,
               swiglu_limit=7.0, act_fmt="fp4"),
    W.Workload("mx_decode_T1", 1, 7168, 2048, 64, 8, "fp4", "zipf_sigmoid", seed=43, act_fmt="fp4"),
    W.Workload("mx_zipf_skips", 300, 512, 384, 16, 4, "fp4", "zipf_sigmoid", seed=44, skip_frac=0.1,
               act_fmt="fp4"),
    W.Workload("mx_ragged_tiles", 333, 1472, 704, 5, 2, "fp4", "softmax", seed=45, act_fmt="fp4"),
]


def _layout(wl):
    return P.B.workspace_layout(P.lib_fmt(wl), wl.T, wl.H, wl.I, wl.E, wl.K)


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_fp4_activation_forward_matches_oracle(wl):
    r = P.run_cuda(wl)
    assert P.B.device_status(r["ws"]) == 0
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], wl.swiglu_limit, act_fmt="fp4")
    m = P.assert_close(r["out"], ref, wl.name)
    print(wl.name, m)


@pytest.mark.parametrize("wl", [CASES[0], CASES[1], CASES[3]], ids=lambda w: w.name)
def test_fp4_input_quantization_bit_exact(wl):
    r = P.run_cuda(wl)
    L = _layout(wl)
    ws = r["ws"]
    assert L.xq_cols % 128 == 0 and L.xq_cols >= wl.H
    ref = route(r["idx"].cpu().numpy(), wl.E, L.row_align)
    inv = P.ws_region(ws, L, "inv", torch.int32, wl.S).cpu().numpy()
    assert (inv == ref["inv"]).all()
    valid = np.flatnonzero(inv >= 0)
    rows, tok = inv[valid], valid // wl.K
    packed = P.ws_region(ws, L, "xq", torch.uint8, L.row_capacity * L.xq_cols // 2)
    packed = packed.view(L.row_capacity, L.xq_cols // 2).cpu().numpy()[rows]
    codes = P.unpack_e2m1(packed, L.xq_cols)
    exps = P.sf_exponents_1x32(P.ws_region(ws, L, "xsf", torch.int32, L.row_capacity * L.x_blocks),
                               L.row_capacity, L.x_blocks)[rows]
    want_c, want_e = P.OM.quantize_hidden(P.bits_of(r["hidden"]), act_fmt="fp4")
    nb = want_e.shape[1]
    assert np.array_equal(codes[:, :wl.H], want_c[tok])
    assert np.array_equal(exps[:, :nb], want_e[tok])
    assert (codes[:, wl.H:] == 0).all() and (exps[:, nb:] == 0).all()


@pytest.mark.parametrize("wl", [CASES[0], CASES[1], CASES[2], CASES[4]], ids=lambda w: w.name)
def test_fp4_requantization_bit_exact_on_the_epilogue_inputs(wl):
    dev = "cuda"
    hidden = W.make_hidden(wl, dev)
    idx, w = W.make_routing(wl, dev)
    prepared = P.B.prepare_weights(W.make_weights(wl, dev), activations="fp4")
    out, act32, ws = P.B.debug_forward_act_f32(hidden, idx, w, prepared, wl.swiglu_limit)
    ref_out = P.B.experts_forward(hidden, idx, w, prepared, wl.swiglu_limit)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    L = _layout(wl)
    inv = P.ws_region(ws, L, "inv", torch.int32, wl.S).cpu().numpy()
    rows = np.sort(inv[inv >= 0])
    packed = P.ws_region(ws, L, "act", torch.uint8, L.row_capacity * L.act_cols // 2)
    codes = P.unpack_e2m1(packed.view(L.row_capacity, L.act_cols // 2).cpu().numpy()[rows], L.act_cols)
    exps = P.sf_exponents_1x32(P.ws_region(ws, L, "asf", torch.int32, L.row_capacity * L.act_blocks),
                               L.row_capacity, L.act_blocks)[rows]
    a = act32.cpu().numpy().astype(np.float64)[rows]
    assert np.isfinite(a).all() and (a[:, wl.I:] == 0).all()
    want_c, want_e = OF.quantize_rows_1x32_e2m1(a[:, :wl.I])
    nb = want_e.shape[1]
    assert np.array_equal(exps[:, :nb], want_e), np.argwhere(exps[:, :nb] != want_e)[:8]
    bad = np.argwhere(codes[:, :wl.I] != want_c)
    assert bad.size == 0, [(int(r), int(c), int(codes[r, c]), int(want_c[r, c]), float(a[r, c])) for r, c in bad[:8]]
    assert (codes[:, wl.I:] == 0).all() and (exps[:, nb:] == 0).all()


def test_fp4_activation_fused_combine_matches_the_combine_kernel():
    """Decode batches of at most 64 slots combine in GEMM2's epilogue; the
    same tokens inside a larger decode batch (120 slots) go through the
    combine kernel: same bits, +0 rows for all-skipped tokens."""
    wl = W.Workload("mx_fused_combine", 10, 320, 192, 64, 4, "fp4", "zipf_sigmoid", seed=48, skip_frac=0.2,
                    act_fmt="fp4")
    idx, w = W.make_routing(wl, "cuda")
    idx[4] = -1
    r = P.run_cuda(wl, idx=idx, w=w)
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], None, act_fmt="fp4")
    P.assert_close(r["out"], ref, "fused combine")
    assert (r["out"][4].view(torch.int16) == 0).all()
    extra = 20
    g = torch.Generator(device="cuda").manual_seed(9)
    hid = torch.cat([r["hidden"], torch.randn(extra, wl.H, generator=g, device="cuda").to(torch.bfloat16)])
    idx2 = torch.cat([idx, torch.randint(0, wl.E, (extra, wl.K), generator=g, device="cuda", dtype=torch.int32)])
    w2 = torch.cat([w, torch.rand(extra, wl.K, generator=g, device="cuda")])
    out = P.B.experts_forward(hid, idx2, w2, r["prepared"])
    assert torch.equal(out[:wl.T].view(torch.int16), r["out"].view(torch.int16))


def test_fp4_activations_change_the_result():
    wl = CASES[3]
    r4 = P.run_cuda(wl)
    r8 = P.run_cuda(W.scaled(wl, act_fmt="fp8"), hidden=r4["hidden"], idx=r4["idx"], w=r4["w"], weights=r4["weights"])
    assert not torch.equal(r4["out"], r8["out"])
    ref8 = P.oracle_out(r8["hidden"], r8["idx"], r8["w"], r8["weights"], wl.swiglu_limit)
    P.assert_close(r8["out"], ref8, "fp8 activations on the same inputs")


def test_fp4_activation_forward_replays_from_a_cuda_graph():
    wl = CASES[3]
    r = P.run_cuda(wl)
    ws = torch.empty_like(r["ws"])
    out = torch.empty_like(r["out"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        P.B.experts_forward(r["hidden"], r["idx"], r["w"], r["prepared"], wl.swiglu_limit, workspace=ws, out=out)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        P.B.experts_forward(r["hidden"], r["idx"], r["w"], r["prepared"], wl.swiglu_limit, workspace=ws, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), r["out"].view(torch.int16))


def _sweep_hidden_fp4():
    """Every finite bf16 value (shuffled, so the blocks' amax vary), then
    blocks holding every e2m1 rounding tie at several scales next to their
    block amax 6 * 2^n."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = OF.bf16_bits_to_f64(bits)
    fin = bits[np.isfinite(v)]
    rng = np.random.default_rng(1)
    H = 1024
    shuffled = fin[rng.permutation(fin.size)]
    rows = [np.concatenate([shuffled, np.zeros((-shuffled.size) % H, np.uint16)]).reshape(-1, H)]
    pos = OF.E2M1_TABLE[:8]
    mids = (pos[1:] + pos[:-1]) / 2
    vals, exact = [], []
    for n in range(-20, 21, 3):
        blk = np.zeros(32)
        blk[0] = 6.0 * 2.0 ** n
        blk[1:1 + mids.size] = mids * 2.0 ** n
        blk[1 + mids.size:1 + 2 * mids.size] = -mids * 2.0 ** n
        ex = np.ones(32, bool)
        blk[1 + 2 * mids.size] = -0.1 * 2.0 ** n  # rounds to -0 (not exact in bf16)
        ex[1 + 2 * mids.size] = False
        vals.append(blk)
        exact.append(ex)
    tie, exact = np.concatenate(vals), np.concatenate(exact)
    tie_bits = (tie.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert (OF.bf16_bits_to_f64(tie_bits)[exact] == tie[exact]).all()
    # the exponent clamps: a block of subnormal bf16 values (n = -127) and one
    # at the top of the bf16 range (n = 126)
    tiny = np.arange(1, 33, dtype=np.uint16)
    huge = np.arange(0x7F7F, 0x7F7F - 32, -1, dtype=np.uint16) | np.tile(np.array([0, 0x8000], np.uint16), 16)
    tie_bits = np.concatenate([tie_bits, tiny, huge])
    tie_bits = np.concatenate([tie_bits, np.zeros((-tie_bits.size) % H, np.uint16)]).reshape(-1, H)
    rows.append(tie_bits)
    return np.concatenate(rows)


def test_fp4_quantizer_exhaustive_bf16_sweep():
    hb = _sweep_hidden_fp4()
    T, H = hb.shape
    wl = W.Workload("sweep_fp4", T, H, 128, 2, 1, "fp4", "softmax", seed=78, act_fmt="fp4")
    hidden = torch.from_numpy(hb.view(np.int16)).view(torch.bfloat16).cuda()
    idx = (torch.arange(T, dtype=torch.int32, device="cuda") % 2).view(T, 1).contiguous()
    w = torch.ones(T, 1, dtype=torch.float32, device="cuda")
    r = P.run_cuda(wl, hidden=hidden, idx=idx, w=w)
    L = _layout(wl)
    inv = P.ws_region(r["ws"], L, "inv", torch.int32, T).cpu().numpy()
    packed = P.ws_region(r["ws"], L, "xq", torch.uint8, L.row_capacity * L.xq_cols // 2)
    codes = P.unpack_e2m1(packed.view(L.row_capacity, L.xq_cols // 2).cpu().numpy()[inv], L.xq_cols)
    exps = P.sf_exponents_1x32(P.ws_region(r["ws"], L, "xsf", torch.int32, L.row_capacity * L.x_blocks),
                               L.row_capacity, L.x_blocks)[inv]
    want_c, want_e = P.OM.quantize_hidden(hb, act_fmt="fp4")
    assert np.array_equal(exps, want_e), np.argwhere(exps != want_e)[:8]
    bad = np.argwhere(codes != want_c)
    assert bad.size == 0, [(int(t), int(c), int(codes[t, c]), int(want_c[t, c]), int(hb[t, c])) for t, c in bad[:8]]
    # the sweep reaches every code, ties and negative zero included, and both exponent ends
    assert set(np.unique(want_c).tolist()) == set(range(16))
    assert want_e.min() == -127 and want_e.max() == 126


def _random_configs(n=8, seed=20241):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        H = int(rng.integers(2, 9)) * 64
        I = int(rng.integers(2, 9)) * 64
        E = int(rng.choice([4, 8, 16, 33, 64]))
        K = int(min(E, rng.choice([1, 2, 4, 8])))
        T = int(rng.choice([1, 3, 17, 64, 150, 300]))
        router = str(rng.choice(["softmax", "zipf_sigmoid"]))
        skip = float(rng.choice([0.0, 0.1]))
        limit = None if rng.random() < 0.5 else float(np.round(rng.uniform(0.1, 5.0), 3))
        out.append(W.Workload(f"mxsweep{i}_T{T}_H{H}_I{I}_E{E}_K{K}", T, H, I, E, K, "fp4", router,
                              seed=4000 + i, skip_frac=skip, swiglu_limit=limit, act_fmt="fp4"))
    return out


@pytest.mark.parametrize("wl", _random_configs(), ids=lambda w: w.name)
def test_fp4_activation_random_configuration_matches_oracle(wl):
    r = P.run_cuda(wl)
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], wl.swiglu_limit, act_fmt="fp4")
    P.assert_close(r["out"], ref, wl.name)
    assert P.B.device_status(r["ws"]) == 0
