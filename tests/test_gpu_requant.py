"""GPU: the GEMM1 epilogue's requantized SwiGLU activations (e4m3 codes and
power-of-two 1x128 exponents in the workspace) against the oracle's.

The GPU requantizes fp32 SwiGLU values and the oracle fp64 ones, so a value
lying on an e4m3 rounding boundary (or an amax on an exponent boundary) may
round the other way: the check is that almost every byte and exponent agree
and that the rest differ by one e4m3 step (or one exponent) only. Columns
past I (the K padding of GEMM2) must hold zero codes.
"""
import numpy as np
import pytest
import torch

from oracle import formats as OF
from tests import parity as P

pytestmark = pytest.mark.gpu

W = P.W

CASES = [
    W.Workload("fp8_ragged", 200, 512, 384, 4, 2, "fp8", "softmax", seed=11),
    W.Workload("fp8_clamp", 160, 256, 256, 8, 2, "fp8", "softmax", seed=12, swiglu_limit=0.3),
    W.Workload("fp4_gptoss_like", 96, 2880, 2880, 8, 4, "fp4", "softmax", seed=15, logit_std=1.5,
               swiglu_limit=7.0),
    W.Workload("fp4_decode_mode", 24, 512, 320, 32, 8, "fp4", "zipf_sigmoid", seed=27),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_requantized_activations_match_the_oracle(wl):
    r = P.run_cuda(wl)
    _, taps = P.OM.experts_forward(P.bits_of(r["hidden"]), r["idx"].cpu().numpy(), r["w"].cpu().numpy(),
                                   P.oracle_weights(r["weights"]), wl.swiglu_limit, return_taps=True)
    L = P.B.workspace_layout(wl.fmt, wl.T, wl.H, wl.I, wl.E, wl.K)
    S = wl.T * wl.K
    inv = P.ws_region(r["ws"], L, "inv", torch.int32, S).cpu().numpy()
    act = P.ws_region(r["ws"], L, "act", torch.uint8, L.row_capacity * L.act_cols)
    act = act.view(L.row_capacity, L.act_cols).cpu().numpy()
    words = P.ws_region(r["ws"], L, "asf", torch.int32, L.row_capacity * L.act_blocks)
    exps = P.sf_exponents(words, L.row_capacity, L.act_blocks)

    g_codes, r_codes, g_exp, r_exp = [], [], [], []
    for (t, k), (aq, ae) in taps["act"].items():
        row = inv[t * wl.K + k]
        assert row >= 0
        g_codes.append(act[row, :wl.I])
        r_codes.append(np.asarray(aq, dtype=np.uint8))
        assert (act[row, wl.I:] == 0).all()
        g_exp.append(exps[row, :len(ae)])
        r_exp.append(np.asarray(ae))
    g_codes, r_codes = np.stack(g_codes), np.stack(r_codes)
    g_exp, r_exp = np.stack(g_exp).astype(np.int64), np.stack(r_exp).astype(np.int64)

    # exponents: equal almost everywhere, off by one at most
    assert np.abs(g_exp - r_exp).max() <= 1
    assert (g_exp == r_exp).mean() >= 0.999, (g_exp == r_exp).mean()
    # codes where the block exponents agree: equal almost everywhere, and a
    # differing byte is the neighbouring e4m3 value of the same sign
    same = np.repeat(g_exp == r_exp, 128, axis=1)[:, :wl.I]
    eq = (g_codes == r_codes)
    assert eq[same].mean() >= 0.999, eq[same].mean()
    d = ~eq & same
    if d.any():
        gs, rs = g_codes[d] >> 7, r_codes[d] >> 7
        gm, rm = (g_codes[d] & 0x7F).astype(np.int64), (r_codes[d] & 0x7F).astype(np.int64)
        assert ((np.abs(gm - rm) <= 1) & ((gs == rs) | (gm + rm <= 1))).all()
    # values where the exponents differ (amax on a boundary): within one e4m3 step
    if (~same).any():
        gv = OF.E4M3_TABLE[g_codes] * np.ldexp(1.0, np.repeat(g_exp, 128, axis=1)[:, :wl.I])
        rv = OF.E4M3_TABLE[r_codes] * np.ldexp(1.0, np.repeat(r_exp, 128, axis=1)[:, :wl.I])
        scale = np.maximum(np.abs(gv), np.abs(rv))[~same]
        assert (np.abs(gv - rv)[~same] <= scale / 8 + 1e-30).all()


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_requantization_is_bit_exact_on_the_epilogue_inputs(wl):
    """The epilogue's requantization is the 1x128 rule itself: applied by the
    oracle's quantizer to the fp32 SwiGLU values the epilogue quantized (read
    through the debug tap; fp32 values are exact in fp64), it must give the
    same e4m3 codes and the same exponents, bit for bit, on every valid row."""
    dev = "cuda"
    hidden = W.make_hidden(wl, dev)
    idx, w = W.make_routing(wl, dev)
    prepared = P.B.prepare_weights(W.make_weights(wl, dev))
    out, act32, ws = P.B.debug_forward_act_f32(hidden, idx, w, prepared, wl.swiglu_limit)
    ref_out = P.B.experts_forward(hidden, idx, w, prepared, wl.swiglu_limit)
    torch.cuda.synchronize()
    # the tap changes nothing else
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))

    L = P.B.workspace_layout(wl.fmt, wl.T, wl.H, wl.I, wl.E, wl.K)
    inv = P.ws_region(ws, L, "inv", torch.int32, wl.T * wl.K).cpu().numpy()
    rows = np.sort(inv[inv >= 0])
    assert len(rows) == int((idx >= 0).sum())
    act = P.ws_region(ws, L, "act", torch.uint8, L.row_capacity * L.act_cols)
    act = act.view(L.row_capacity, L.act_cols).cpu().numpy()[rows]
    words = P.ws_region(ws, L, "asf", torch.int32, L.row_capacity * L.act_blocks)
    exps = P.sf_exponents(words, L.row_capacity, L.act_blocks)[rows]
    a = act32.cpu().numpy().astype(np.float64)[rows]
    assert np.isfinite(a).all()
    assert (a[:, wl.I:] == 0).all()
    codes, e = OF.quantize_rows_1x128(a[:, :wl.I])
    assert np.array_equal(exps[:, :e.shape[1]], e), np.argwhere(exps[:, :e.shape[1]] != e)[:8]
    bad = np.argwhere(act[:, :wl.I] != codes)
    assert bad.size == 0, [(int(r), int(c), int(act[r, c]), int(codes[r, c]), float(a[r, c])) for r, c in bad[:8]]
    assert (act[:, wl.I:] == 0).all()
