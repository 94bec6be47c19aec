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
