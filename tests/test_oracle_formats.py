"""Pins for the oracle's number formats and activation quantizer (CPU only).

The oracle's tables are checked against the OCP specifications' printed
values (tests/golden), against torch's own float8 decode/encode (a library
routine), and the quantizer against a brute-force nearest-value search over
all 256 codes written independently here.
"""
import math

import numpy as np
import pytest
import torch

from oracle import formats as F
from tests.golden_io import read_pairs


def _val(s):
    return float(s)


@pytest.mark.parametrize("name,table", [("e4m3_values.txt", F.E4M3_TABLE),
                                        ("e2m1_values.txt", F.E2M1_TABLE),
                                        ("ue8m0_values.txt", F.UE8M0_TABLE)])
def test_decode_tables_match_spec_landmarks(name, table):
    for code, value in read_pairs(name):
        got = table[int(code, 16)]
        want = _val(value)
        if math.isnan(want):
            assert math.isnan(got), code
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), code


def test_e4m3_table_matches_torch_decode_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double().numpy()
    ours = F.E4M3_TABLE
    nan = np.isnan(ref)
    assert (np.isnan(ours) == nan).all()
    assert (ours[~nan] == ref[~nan]).all()
    assert (np.signbit(ours[~nan]) == np.signbit(ref[~nan])).all()
    assert nan.sum() == 2  # only 0x7F / 0xFF


def test_e2m1_and_ue8m0_closed_forms():
    for c in range(16):
        mag = [0, 0.5, 1, 1.5, 2, 3, 4, 6][c & 7]
        assert F.E2M1_TABLE[c] == (-mag if c & 8 else mag)
    for b in range(255):
        assert F.UE8M0_TABLE[b] == math.ldexp(1.0, b - 127)
    assert math.isnan(F.UE8M0_TABLE[255])


def test_fp4_nibble_order():
    # One byte 0x71: low nibble 0x1 (0.5) is element 0, high nibble 0x7 (6.0) element 1.
    vals = F.decode_e2m1_packed(np.array([[0x71, 0x0A]], dtype=np.uint8), 4)
    assert vals.tolist() == [[0.5, 6.0, -1.0, 0.0]]


def _brute_e4m3(v):
    """Nearest finite e4m3 by scanning all codes; ties -> even mantissa; sat."""
    best, best_d = None, None
    for c in range(256):
        val = F.E4M3_TABLE[c]
        if math.isnan(val):
            continue
        if (c & 0x80) != (0x80 if math.copysign(1, v) < 0 else 0):
            continue
        d = abs(min(abs(v), 448.0) - abs(val))
        if best is None or d < best_d or (d == best_d and (c & 1) == 0 and (best & 1) == 1):
            best, best_d = c, d
    return best


def test_e4m3_quantizer_brute_force_including_ties():
    pos = F.E4M3_TABLE[:0x7F]
    mids = (pos[1:] + pos[:-1]) / 2  # every exact tie
    rng = np.random.default_rng(5)
    rand = rng.standard_normal(3000) * np.exp2(rng.integers(-12, 9, 3000))
    vals = np.concatenate([mids, -mids, pos, -pos, rand, [0.0, -0.0, 447.9, 460.0, 1e6, -1e6, 1e-30, -1e-30]])
    got = F.e4m3_rne_satfinite(vals)
    want = np.array([_brute_e4m3(float(v)) for v in vals], dtype=np.uint8)
    assert (got == want).all(), np.flatnonzero(got != want)[:10]


def test_e4m3_quantizer_matches_torch_cast_in_range():
    # torch's fp32 -> float8_e4m3fn cast rounds to nearest even; inside
    # [-448, 448] it must agree with the oracle code for code.
    rng = np.random.default_rng(6)
    v = np.clip(rng.standard_normal(200000) * np.exp2(rng.integers(-14, 9, 200000)), -448, 448)
    v = v.astype(np.float32).astype(np.float64)
    ref = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (F.e4m3_rne_satfinite(v) == ref).all()


def test_scale_exponent_is_minimal():
    rng = np.random.default_rng(7)
    amax = np.concatenate([
        np.abs(rng.standard_normal(20000)) * np.exp2(rng.integers(-60, 60, 20000)),
        448.0 * np.exp2(np.arange(-40, 40)),              # exact boundaries
        np.nextafter(448.0 * np.exp2(np.arange(-40, 40)), np.inf),
        [1.0, 448.0, 449.0, 224.0, 224.0001]])
    e = F.act_scale_exponent(amax).astype(np.float64)
    assert (amax <= 448.0 * np.exp2(e)).all()
    assert (amax > 448.0 * np.exp2(e - 1)).all()
    assert F.act_scale_exponent(0.0) == 0
    assert F.act_scale_exponent(448.0) == 0 and F.act_scale_exponent(449.0) == 1
    assert F.act_scale_exponent(1e-45) == -127 and F.act_scale_exponent(3e38) == 120


def test_exponent_rule_matches_log2_formula():
    # 2^ceil(log2(amax/448)) from the workload definition, in exact arithmetic,
    # on values where float log2 is safe (away from the boundaries).
    rng = np.random.default_rng(8)
    amax = np.abs(rng.standard_normal(50000)) * np.exp2(rng.integers(-30, 30, 50000)) + 1e-30
    ratio = amax / 448.0
    frac = np.log2(ratio) - np.floor(np.log2(ratio))
    safe = (frac > 1e-9) & (frac < 1 - 1e-9)
    assert (F.act_scale_exponent(amax[safe]) == np.ceil(np.log2(ratio[safe]))).all()


def test_all_bf16_values_quantize_like_brute_force():
    # Every finite bf16 value v, quantized in a block whose amax is fixed to
    # A = 448 * 2^n, must land on the nearest e4m3 code of v / 2^n.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = F.bf16_bits_to_f64(bits)
    v = v[np.isfinite(v)]
    for n in (-3, 0, 5):
        A = 448.0 * 2.0 ** n
        keep = np.abs(v) <= A
        blk = np.zeros((keep.sum(), 128))
        blk[:, 0] = v[keep]
        blk[:, 1] = A
        codes, exps = F.quantize_rows_1x128(blk)
        assert (exps[:, 0] == n).all()
        ref = torch.tensor(v[keep] / 2.0 ** n, dtype=torch.float64).float().to(
            torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert (codes[:, 0] == ref).all()


def test_partial_block_and_roundtrip():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((5, 2880))
    codes, exps = F.quantize_rows_1x128(x)
    assert exps.shape == (5, 23)
    last = np.max(np.abs(x[:, 2816:]), axis=1)
    assert (exps[:, 22] == F.act_scale_exponent(last)).all()
    back = F.dequantize_rows_1x128(codes, exps)
    # e4m3 keeps 4 significant bits: relative error <= 2^-4 for normal codes.
    big = np.abs(x) > 448 * 2.0 ** exps.repeat(128, axis=1)[:, :2880] * 2 ** -6
    assert (np.abs(back - x)[big] <= np.abs(x)[big] * 2 ** -4 + 1e-300).all()


def test_bf16_rounding_helper():
    rng = np.random.default_rng(10)
    v = rng.standard_normal(100000) * np.exp2(rng.integers(-30, 30, 100000))
    v32 = v.astype(np.float32).astype(np.float64)  # fp32 inputs: torch cast is exact RNE
    ref = torch.tensor(v32, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    assert (F.f64_to_bf16_rne(v32) == ref).all()


# ------------------------------------------------------- e2m1 (FP4) activations
def _brute_e2m1(v):
    """Nearest e2m1 code by scanning all 16 codes: same sign, magnitude
    capped at 6, an exact tie going to the code whose mantissa bit is 0."""
    sign = 0x8 if math.copysign(1.0, v) < 0 else 0
    best, best_d = None, None
    for c in range(16):
        if (c & 0x8) != sign:
            continue
        d = abs(min(abs(v), 6.0) - abs(F.E2M1_TABLE[c]))
        if best is None or d < best_d or (d == best_d and (c & 1) == 0 and (best & 1) == 1):
            best, best_d = c, d
    return best


def test_e2m1_rounding_landmarks():
    # ties between neighbouring magnitudes go to the even code; above 6 saturates
    cases = [(0.25, 0x0), (0.26, 0x1), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6),
             (5.0, 0x6), (5.01, 0x7), (6.0, 0x7), (6.5, 0x7), (1e9, 0x7), (0.0, 0x0), (-0.0, 0x8),
             (-0.25, 0x8), (-1.75, 0xC), (-6.0, 0xF)]
    got = F.e2m1_rne_satfinite(np.array([v for v, _ in cases]))
    assert got.tolist() == [c for _, c in cases]


def test_e2m1_quantizer_brute_force_including_ties():
    pos = F.E2M1_TABLE[:8]
    mids = (pos[1:] + pos[:-1]) / 2
    rng = np.random.default_rng(15)
    rand = rng.standard_normal(4000) * np.exp2(rng.integers(-4, 4, 4000))
    vals = np.concatenate([mids, -mids, pos, -pos, rand, [0.0, -0.0, 5.999, 6.001, 100.0, -100.0, 1e-30, -1e-30]])
    got = F.e2m1_rne_satfinite(vals)
    want = np.array([_brute_e2m1(float(v)) for v in vals], dtype=np.uint8)
    assert (got == want).all(), np.flatnonzero(got != want)[:10]


def test_e2m1_scale_exponent_is_minimal():
    rng = np.random.default_rng(16)
    amax = np.concatenate([
        np.abs(rng.standard_normal(20000)) * np.exp2(rng.integers(-60, 60, 20000)),
        6.0 * np.exp2(np.arange(-40, 40)),                 # exact boundaries
        np.nextafter(6.0 * np.exp2(np.arange(-40, 40)), np.inf),
        [1.0, 3.0, 3.0001, 6.0, 6.0001, 12.0]])
    n = F.act_scale_exponent_e2m1(amax).astype(np.float64)
    assert (amax <= 6.0 * np.exp2(n)).all()
    assert (amax > 6.0 * np.exp2(n - 1)).all()
    assert F.act_scale_exponent_e2m1(0.0) == 0
    assert F.act_scale_exponent_e2m1(6.0) == 0 and F.act_scale_exponent_e2m1(6.0001) == 1
    assert F.act_scale_exponent_e2m1(3.0) == -1 and F.act_scale_exponent_e2m1(1.0) == -2
    assert F.act_scale_exponent_e2m1(1e-45) == -127 and F.act_scale_exponent_e2m1(3e38) == 126


def test_e2m1_exponent_rule_matches_log2_formula():
    rng = np.random.default_rng(17)
    amax = np.abs(rng.standard_normal(50000)) * np.exp2(rng.integers(-30, 30, 50000)) + 1e-30
    ratio = amax / 6.0
    frac = np.log2(ratio) - np.floor(np.log2(ratio))
    safe = (frac > 1e-9) & (frac < 1 - 1e-9)
    assert (F.act_scale_exponent_e2m1(amax[safe]) == np.ceil(np.log2(ratio[safe]))).all()


def test_all_bf16_values_quantize_to_e2m1_like_brute_force():
    # Every finite bf16 value v, quantized in a 32-block whose amax is fixed to
    # A = 6 * 2^n, must land on the brute-force code of v / 2^n.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = F.bf16_bits_to_f64(bits)
    v = v[np.isfinite(v)]
    mags = F.E2M1_TABLE[:8]
    for n in (-2, 0, 3):
        A = 6.0 * 2.0 ** n
        keep = np.abs(v) <= A
        blk = np.zeros((keep.sum(), 32))
        blk[:, 0] = v[keep]
        blk[:, 1] = A
        codes, exps = F.quantize_rows_1x32_e2m1(blk)
        assert (exps[:, 0] == n).all()
        # vectorised brute force: distance to every magnitude, ties to the even code
        r = np.abs(v[keep] / 2.0 ** n)[:, None]
        d = np.abs(r - mags[None, :])
        dmin = d.min(axis=1, keepdims=True)
        cand = d == dmin
        even = cand & ((np.arange(8) & 1) == 0)[None, :]
        pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
        want = pick | np.where(np.signbit(v[keep]), 0x8, 0)
        assert (codes[:, 0] == want).all()


def test_e2m1_partial_block_roundtrip_and_packing():
    rng = np.random.default_rng(18)
    x = rng.standard_normal((5, 2880))
    codes, exps = F.quantize_rows_1x32_e2m1(x)
    assert exps.shape == (5, 90) and codes.max() <= 0xF
    back = F.dequantize_rows_1x32_e2m1(codes, exps)
    unit = np.exp2(exps.astype(np.float64)).repeat(32, axis=1)[:, :2880]
    # two significant bits: |error| <= |x| / 4 at and above the block unit,
    # <= unit / 4 below it (the 0.5-spaced codes)
    assert (np.abs(back - x) <= np.maximum(np.abs(x), unit) / 4 + 1e-300).all()
    packed = F.pack_e2m1(codes)
    assert packed.shape == (5, 1440)
    assert np.array_equal(F.decode_e2m1_packed(packed, 2880), F.E2M1_TABLE[codes])
