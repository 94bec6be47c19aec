"""Pins for the oracle's experts forward (CPU only).

* A brute-force dense evaluation written independently here (bit-level
  decoding, a scan over all e4m3 codes for rounding, an exponent search by
  counting, a dense token x expert loop with no sorting or gathering) must
  agree with the oracle to 1e-12.
* Closed forms: identity-like weights reduce the layer to a textbook
  SwiGLU of the input; the clamp; all-skipped batches; NaN weights in
  skipped slots; padding tokens (the shared-batch slicing example of the
  Mega MoE EP page).
* Planted mistakes: each plausible bug, planted in a copy of the oracle,
  must make the brute-force comparison fail.
"""
import math
import struct

import numpy as np
import pytest
import torch

import oracle.moe as M
from oracle import formats as F
from block_scaled_moe_expert_gb300 import workloads as W


# ---------------------------------------------------------------- brute force
def _bf16(bits):
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def _e4m3(c):
    s = -1.0 if c & 0x80 else 1.0
    e, m = (c >> 3) & 15, c & 7
    if e == 15 and m == 7:
        return math.nan
    return s * (m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))


_E4M3 = np.array([_e4m3(c) for c in range(256)])
_FIN = np.array([c for c in range(256) if not math.isnan(_E4M3[c])])


def _round_e4m3(v):
    """Nearest finite code (same sign), ties to the even code, saturating."""
    sign = 0x80 if math.copysign(1.0, v) < 0 else 0
    cands = _FIN[(_FIN & 0x80) == sign]
    d = np.abs(np.abs(_E4M3[cands]) - min(abs(v), 448.0))
    best = cands[d == d.min()]
    even = best[(best & 1) == 0]
    return int(even[0] if even.size else best[0])


def _exp_rule(amax):
    if amax == 0:
        return 0
    for n in range(-127, 128):
        if amax <= 448.0 * 2.0 ** n:
            return n
    return 127


def _quant_dequant(row):
    out = np.empty(len(row))
    for b0 in range(0, len(row), 128):
        blk = row[b0:b0 + 128]
        n = _exp_rule(max(abs(v) for v in blk))
        for j, v in enumerate(blk):
            out[b0 + j] = _E4M3[_round_e4m3(v / 2.0 ** n)] * 2.0 ** n
    return out


_E2M1_MAG = [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def _round_e2m1(v):
    """Nearest e2m1 value (same sign), ties to the even code, saturating at 6."""
    m = min(abs(v), 6.0)
    d = [abs(m - c) for c in _E2M1_MAG]
    best = [c for c in range(8) if d[c] == min(d)]
    even = [c for c in best if c % 2 == 0]
    return math.copysign(_E2M1_MAG[(even or best)[0]], v)


def _exp_rule_fp4(amax):
    if amax == 0:
        return 0
    for n in range(-127, 128):
        if amax <= 6.0 * 2.0 ** n:
            return n
    return 127


def _quant_dequant_fp4(row):
    out = np.empty(len(row))
    for b0 in range(0, len(row), 32):
        blk = row[b0:b0 + 32]
        n = _exp_rule_fp4(max(abs(v) for v in blk))
        for j, v in enumerate(blk):
            out[b0 + j] = _round_e2m1(v / 2.0 ** n) * 2.0 ** n
    return out


def _weight(fmt, w, s, e, r, c):
    if fmt == "fp8":
        return _E4M3[int(w[e, r, c])] * float(s[e, r // 128, c // 128])
    byte = int(w[e, r, c // 2])
    code = (byte >> 4) if c % 2 else (byte & 15)
    mag = [0, 0.5, 1, 1.5, 2, 3, 4, 6][code & 7]
    return (-mag if code & 8 else mag) * 2.0 ** (int(s[e, r, c // 32]) - 127)


def brute_force(bits, idx, topk_w, wt, limit, act="fp8"):
    fmt, E, H, I = wt["fmt"], wt["E"], wt["H"], wt["I"]
    qd = _quant_dequant_fp4 if act == "fp4" else _quant_dequant
    T, K = idx.shape
    W13 = np.array([[[_weight(fmt, wt["w13"], wt["w13_scale"], e, r, c) for c in range(H)]
                     for r in range(2 * I)] for e in range(E)])
    W2 = np.array([[[_weight(fmt, wt["w2"], wt["w2_scale"], e, r, c) for c in range(I)]
                    for r in range(H)] for e in range(E)])
    out = np.zeros((T, H))
    for t in range(T):
        x = qd([_bf16(b) for b in bits[t]])
        for e in range(E):
            r = sum(float(np.float32(topk_w[t, k])) for k in range(K) if idx[t, k] == e)
            if not any(idx[t, k] == e for k in range(K)):
                continue
            h = W13[e] @ x
            g, u = h[:I], h[I:]
            if limit is not None:
                g = np.minimum(g, limit)
                u = np.clip(u, -limit, limit)
            a = qd(list(g / (1 + np.exp(-g)) * u))
            out[t] += r * (W2[e] @ a)
    return out


def _case(T, H, I, E, K, fmt, skip=0.0, limit=None, seed=3, act="fp8"):
    wl = W.Workload("pin", T, H, I, E, K, fmt, "softmax", skip_frac=skip, swiglu_limit=limit, seed=seed)
    hid, idx, w, wt = W.make_all(wl)
    bits = hid.view(torch.int16).numpy().view(np.uint16)
    wt = {k: (v.numpy() if torch.is_tensor(v) else v) for k, v in wt.items()}
    return bits, idx.numpy(), w.numpy(), wt, limit, act


def _rel(a, b):
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


CASES = [dict(T=3, H=128, I=128, E=3, K=2, fmt="fp8", skip=0.2),
         dict(T=2, H=256, I=128, E=2, K=2, fmt="fp8", limit=0.05),
         dict(T=3, H=128, I=64, E=3, K=2, fmt="fp4", skip=0.2),
         dict(T=2, H=192, I=96, E=2, K=1, fmt="fp4", limit=0.02),
         dict(T=3, H=128, I=64, E=3, K=2, fmt="fp4", skip=0.2, act="fp4"),
         dict(T=2, H=192, I=96, E=2, K=2, fmt="fp4", limit=0.02, act="fp4")]


@pytest.mark.parametrize("case", CASES)
def test_oracle_matches_brute_force(case):
    bits, idx, w, wt, limit, act = _case(**case)
    ref = brute_force(bits, idx, w, wt, limit, act)
    got = M.experts_forward(bits, idx, w, wt, limit, act_fmt=act)
    assert np.abs(ref).max() > 0
    assert _rel(got, ref) < 1e-12


def test_fp4_activations_need_fp4_weights():
    bits, idx, w, wt, limit, _ = _case(**CASES[0])
    with pytest.raises(ValueError):
        M.experts_forward(bits, idx, w, wt, limit, act_fmt="fp4")


# ----------------------------------------------------------------- closed forms
def _identity_weights(fmt, H, I, gate_code, up_code, w2_code, sg, su, s2):
    """FP8 weights: w13 = [sg*c_g*Id ; su*c_u*Id], w2 = s2*c_2*Id (H == I)."""
    assert fmt == "fp8" and H == I
    w13 = np.zeros((1, 2 * I, H), np.uint8)
    w2 = np.zeros((1, H, I), np.uint8)
    for j in range(I):
        w13[0, j, j] = gate_code
        w13[0, I + j, j] = up_code
        w2[0, j, j] = w2_code
    w13s = np.ones((1, 2 * I // 128, H // 128), np.float32)
    w13s[0, : I // 128] = sg
    w13s[0, I // 128:] = su
    w2s = np.full((1, H // 128, I // 128), s2, np.float32)
    return dict(fmt="fp8", E=1, H=H, I=I, w13=w13, w13_scale=w13s, w2=w2, w2_scale=w2s)


def _exact_inputs(rng, T, H):
    """bf16 rows that are exact e4m3 values with amax 448 in every block."""
    codes = rng.integers(0, 0x7F, (T, H)) | (rng.integers(0, 2, (T, H)) << 7)
    x = F.E4M3_TABLE[codes]
    x[:, ::128] = 448.0
    bits = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert (F.bf16_bits_to_f64(bits) == x).all()
    return x, bits


def test_identity_weights_reduce_to_textbook_swiglu():
    rng = np.random.default_rng(21)
    H = I = 256
    x, bits = _exact_inputs(rng, 4, H)
    wt = _identity_weights("fp8", H, I, 0x38, 0x40, 0x38, 0.75, 0.5, 3.0)  # 1.0, 2.0, 1.0
    idx = np.zeros((4, 1), np.int32)
    w = np.ones((4, 1), np.float32)
    got = M.experts_forward(bits, idx, w, wt)
    g = 0.75 * x
    u = 0.5 * 2.0 * x
    a = g * u / (1 + np.exp(-g))
    want = 3.0 * np.array([_quant_dequant(list(r)) for r in a])
    assert np.array_equal(got, want)


def test_clamp_closed_form():
    rng = np.random.default_rng(22)
    H = I = 128
    x, bits = _exact_inputs(rng, 3, H)
    wt = _identity_weights("fp8", H, I, 0x38, 0x38, 0x38, 1 / 16, 1 / 32, 1.0)
    L = 7.0
    got = M.experts_forward(bits, np.zeros((3, 1), np.int32), np.ones((3, 1), np.float32), wt, L)
    g = np.minimum(x / 16, L)
    u = np.clip(x / 32, -L, L)
    want = np.array([_quant_dequant(list(r)) for r in g * u / (1 + np.exp(-g))])
    assert np.array_equal(got, want)
    assert (np.abs(x / 16) > L).any() and (np.abs(x / 32) > L).any()


def test_all_skipped_is_exact_zero():
    bits, idx, w, wt, _, _ = _case(4, 128, 128, 3, 2, "fp8")
    out = M.experts_forward(bits, np.full_like(idx, -1), w, wt)
    assert np.array_equal(out, np.zeros_like(out)) and not np.signbit(out).any()


def test_nan_weight_in_skipped_slot_has_no_effect():
    bits, idx, w, wt, _, _ = _case(4, 128, 128, 3, 2, "fp8")
    idx[1, 0] = -1
    w2 = w.copy()
    w2[1, 0] = np.nan
    a = M.experts_forward(bits, idx, w, wt)
    b = M.experts_forward(bits, idx, w2, wt)
    assert np.array_equal(a, b)


def test_padding_tokens_leave_outputs_unchanged():
    bits, idx, w, wt, _, _ = _case(4, 128, 128, 3, 2, "fp8")
    pad_bits = np.concatenate([bits, bits[:2]])
    pad_idx = np.concatenate([idx, np.full((2, 2), -1, idx.dtype)])
    pad_w = np.concatenate([w, w[:2]])
    a = M.experts_forward(bits, idx, w, wt)
    b = M.experts_forward(pad_bits, pad_idx, pad_w, wt)
    assert np.array_equal(a, b[:4]) and np.array_equal(b[4:], np.zeros((2, 128)))


def test_token_subset_equals_full_rows():
    bits, idx, w, wt, _, _ = _case(6, 128, 128, 3, 2, "fp4")
    full = M.experts_forward(bits, idx, w, wt)
    sub = M.experts_forward(bits, idx, w, wt, tokens=[4, 1])
    assert np.array_equal(sub, full[[4, 1]])


# ------------------------------------------------------------- planted mistakes
def _swap_halves(h, inter, limit):
    return _orig_swiglu(np.concatenate([h[:, inter:], h[:, :inter]], axis=1), inter, limit)


_orig_swiglu = M.swiglu
_orig_dequant = M.dequant_weight
_orig_quant = F.quantize_rows_1x128


def _no_clamp(h, inter, limit):
    return _orig_swiglu(h, inter, None)


def _first_kblock_scale(fmt, w, scale, expert, rows, cols):
    if fmt == "fp8":
        s = np.array(scale, copy=True)
        s[expert] = s[expert][:, :1]
        return _orig_dequant(fmt, w, s, expert, rows, cols)
    return _orig_dequant(fmt, w, scale, expert, rows, cols)


def _nibbles_swapped(fmt, w, scale, expert, rows, cols):
    if fmt == "fp4":
        b = np.asarray(w[expert])
        w = {expert: ((b & 15) << 4) | (b >> 4)}
    return _orig_dequant(fmt, w, scale, expert, rows, cols)


def _exp_off_by_one(x):
    codes, exps = _orig_quant(x)
    return codes, exps + 1  # exponent stored one step too large


_orig_quant_fp4 = F.quantize_rows_1x32_e2m1


def _fp4_exp_off_by_one(x):
    codes, exps = _orig_quant_fp4(x)
    return codes, exps - 1  # exponent stored one step too small


def _fp4_ties_away(v):
    """e2m1 rounding with ties away from zero instead of to the even code."""
    v = np.asarray(v, dtype=np.float64)
    mags = F.E2M1_TABLE[:8]
    m = np.minimum(np.abs(v), 6.0)[..., None]
    d = np.abs(m - mags)
    pick = (d == d.min(axis=-1, keepdims=True)) * np.arange(8)
    return (pick.max(axis=-1) | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def _fp4_block_64(x):
    monkey = F.ACT_BLOCK_FP4
    try:
        F.ACT_BLOCK_FP4 = 64
        codes, exps = _orig_quant_fp4(x)
    finally:
        F.ACT_BLOCK_FP4 = monkey
    return codes, np.repeat(exps, 2, axis=1)[:, :(x.shape[1] + 31) // 32]


@pytest.mark.parametrize("name,target,attr,bad,case", [
    ("gate/up swapped", M, "swiglu", _swap_halves, CASES[0]),
    ("clamp dropped", M, "swiglu", _no_clamp, CASES[1]),
    ("one scale per row block", M, "dequant_weight", _first_kblock_scale, CASES[1]),
    ("fp4 nibbles swapped", M, "dequant_weight", _nibbles_swapped, CASES[2]),
    ("scale exponent off by one", F, "quantize_rows_1x128", _exp_off_by_one, CASES[0]),
    ("fp4 activation exponent off by one", F, "quantize_rows_1x32_e2m1", _fp4_exp_off_by_one, CASES[4]),
    ("fp4 activation blocks of 64", F, "quantize_rows_1x32_e2m1", _fp4_block_64, CASES[5]),
    ("fp4 activation ties away from zero", F, "e2m1_rne_satfinite", _fp4_ties_away, CASES[4]),
])
def test_planted_mistake_is_caught(monkeypatch, name, target, attr, bad, case):
    bits, idx, w, wt, limit, act = _case(**case)
    ref = brute_force(bits, idx, w, wt, limit, act)
    monkeypatch.setattr(target, attr, bad)
    got = M.experts_forward(bits, idx, w, wt, limit, act_fmt=act)
    assert _rel(got, ref) > 1e-6, name


def test_planted_weight_drop_is_caught():
    bits, idx, w, wt, limit, act = _case(**CASES[0])
    ref = brute_force(bits, idx, w, wt, limit, act)
    got = M.experts_forward(bits, idx, np.ones_like(w), wt, limit)
    assert _rel(got, ref) > 1e-3


def test_expert_group_split_used_by_the_full_size_tests():
    """The full-size GPU tests evaluate the oracle per group of experts in
    threads and add the groups' outputs; that equals one oracle call up to the
    order of fp64 additions, and the token sample covers every touched expert."""
    from tests import parity as P
    wl = W.Workload("split", 40, 256, 128, 16, 4, "fp4", "zipf_sigmoid", seed=77, skip_frac=0.1)
    hidden = W.make_hidden(wl)
    idx, w = W.make_routing(wl)
    weights = W.make_weights(wl)
    toks = P.sample_tokens(idx, wl.E, 12, wl.seed)
    assert len(toks) >= 12 and toks[0] == 0 and toks[-1] == wl.T - 1
    ids = idx.numpy()
    assert set(np.unique(ids[toks]).tolist()) - {-1} == set(np.unique(ids).tolist()) - {-1}
    one = P.oracle_out(hidden, idx, w, weights, None, tokens=toks)
    split = P.oracle_out_parallel(hidden, idx, w, weights, None, toks, threads=3)
    assert np.abs(split - one).max() <= 1e-12 * np.abs(one).max()
