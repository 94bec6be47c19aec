"""The MoE experts forward, written out pair by pair in fp64 (oracle side).

Test infrastructure only (see the package docstring).

Steps, in the order the pages give them:
1. Flatten the top-k pairs and route them (``oracle.routing``), following
   fp8_grouped_mm_experts_forward (source excerpt on the error page
   "grouped_mm experts dispatch does not support activation_scheme='static'").
2. Quantize each hidden row dynamically in 1x128 blocks to e4m3 with a
   power-of-two scale ("quantizes activations dynamically per-block", same
   page). A token is quantized once; every pair of the token uses the same
   bytes, which is what gathering already-quantized rows gives.
3. GEMM1 through the expert's gate_up weights, dequantized exactly
   (the grouped FP8 x FP8/FP4 matmul named in the deepgemm excerpt).
4. SwiGLU over the [gate | up] halves, with the optional clamp
   (``swiglu_limit``: "absent -> unclamped", Mega MoE docstring):
   gate = min(gate, L), up = clamp(up, -L, L), act = silu(gate) * up.
5. Requantize the activation with the same 1x128 rule (the input of the
   second block-scaled grouped GEMM is again e4m3 with block scales).
6. GEMM2 through down_proj, dequantized exactly.
7. Weight each pair's row by its routing weight, drop skipped pairs (the
   "sentinel rows zeroed" step) and sum the top-k rows of each token in
   ascending k (the deterministic reshape+sum of the same page).

Weights are decoded exactly (value = code * scale in fp64):
* FP8: e4m3 codes with one fp32 scale per 128x128 block; w13 [E, 2I, H],
  w13_scale [E, 2I/128, H/128]; w2 [E, H, I], w2_scale [E, H/128, I/128];
* FP4: e2m1 codes packed two per byte along K (low nibble = even index) with
  one UE8M0 byte per 1x32 block; w13 [E, 2I, H/2], w13_scale [E, 2I, H/32];
  w2 [E, H, I/2], w2_scale [E, H, I/32].
Rows [0, I) of w13 are the gate half and rows [I, 2I) the up half.

``act_fmt`` selects the activation format of steps 2 and 5: "fp8" (e4m3,
1x128 blocks, the pages' dynamic rule) or "fp4" (e2m1, 1x32 blocks with
UE8M0 exponents, for the variant in which both GEMM operands are FP4; the
rule is in ``oracle.formats``). Everything else is the same.
"""
import numpy as np

from . import formats as F
from .routing import route

FP8 = "fp8"
FP4 = "fp4"
ACT_FMTS = (FP8, FP4)


def quantize_act(x, act_fmt):
    """Steps 2 and 5: (codes, exps) of fp64 rows in the activation format."""
    if act_fmt == FP8:
        return F.quantize_rows_1x128(x)
    if act_fmt == FP4:
        return F.quantize_rows_1x32_e2m1(x)
    raise ValueError(act_fmt)


def dequantize_act(codes, exps, act_fmt):
    if act_fmt == FP8:
        return F.dequantize_rows_1x128(codes, exps)
    if act_fmt == FP4:
        return F.dequantize_rows_1x32_e2m1(codes, exps)
    raise ValueError(act_fmt)


def dequant_weight(fmt, w, scale, expert, rows, cols):
    """Exact fp64 copy of one expert's [rows, cols] weight matrix."""
    if fmt == FP8:
        q = F.decode_e4m3(w[expert])
        s = np.asarray(scale[expert], dtype=np.float64)
        s = np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)[:rows, :cols]
        return q * s
    if fmt == FP4:
        q = F.decode_e2m1_packed(w[expert], cols)
        s = F.decode_ue8m0(scale[expert])
        s = np.repeat(s, 32, axis=1)[:, :cols]
        return q * s
    raise ValueError(fmt)


def swiglu(h, inter, limit):
    g = h[:, :inter]
    u = h[:, inter:]
    if limit is not None:
        g = np.minimum(g, limit)
        u = np.clip(u, -limit, limit)
    return g / (1.0 + np.exp(-g)) * u


def expert_mlp(xd, w13d, w2d, inter, limit, act_fmt=FP8):
    """One expert on the dequantized activation rows xd [n, H] (fp64).

    Returns (y [n, H], act codes, act exps) where act = requantized SwiGLU.
    """
    h = xd @ w13d.T
    a = swiglu(h, inter, limit)
    aq, ae = quantize_act(a, act_fmt)
    y = dequantize_act(aq, ae, act_fmt) @ w2d.T
    return y, aq, ae


def experts_forward(hidden_bits, topk_idx, topk_w, weights, swiglu_limit=None,
                    tokens=None, return_taps=False, act_fmt=FP8):
    """fp64 experts forward for the tokens listed in ``tokens`` (default all).

    hidden_bits: uint16 bf16 bit patterns [T, H]; topk_idx: int [T, K];
    topk_w: float32 [T, K]; weights: dict(fmt, E, H, I, w13, w13_scale, w2,
    w2_scale); act_fmt: "fp8" or "fp4" (FP4 weights only). Returns out
    [len(tokens), H] in fp64 (and taps if asked).
    """
    if act_fmt == FP4 and weights["fmt"] != FP4:
        raise ValueError("FP4 activations are defined with FP4 weights")
    fmt, E, H, I = weights["fmt"], weights["E"], weights["H"], weights["I"]
    topk_idx = np.asarray(topk_idx, dtype=np.int64)
    topk_w = np.asarray(topk_w, dtype=np.float32).astype(np.float64)
    T, K = topk_idx.shape
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    x = F.bf16_bits_to_f64(np.asarray(hidden_bits)[tokens])
    xq, xe = quantize_act(x, act_fmt)
    xd = dequantize_act(xq, xe, act_fmt)

    # Per-pair outputs y[(i, k)] for the selected tokens; skipped slots never
    # produce a row, so they contribute exactly zero below.
    ids = topk_idx[tokens]
    y = {}
    act = {}
    for e in np.unique(ids):
        if e < 0 or e >= E:
            continue
        pairs = np.argwhere(ids == e)  # (i, k), row-major = ascending slot
        w13d = dequant_weight(fmt, weights["w13"], weights["w13_scale"], e, 2 * I, H)
        w2d = dequant_weight(fmt, weights["w2"], weights["w2_scale"], e, H, I)
        ye, aq, ae = expert_mlp(xd[pairs[:, 0]], w13d, w2d, I, swiglu_limit, act_fmt)
        for j, (i, k) in enumerate(pairs):
            y[(i, k)] = ye[j]
            act[(i, k)] = (aq[j], ae[j])
        del w13d, w2d

    out = np.zeros((len(tokens), H), dtype=np.float64)
    for i in range(len(tokens)):
        for k in range(K):
            if (i, k) in y:
                out[i] += topk_w[tokens[i], k] * y[(i, k)]
    if return_taps:
        return out, dict(xq=xq, xe=xe, act=act)
    return out


def quantize_hidden(hidden_bits, act_fmt=FP8):
    """Step 2 alone on every token: (codes [T, H], exps [T, blocks])."""
    return quantize_act(F.bf16_bits_to_f64(hidden_bits), act_fmt)


__all__ = ["FP8", "FP4", "ACT_FMTS", "route", "experts_forward", "quantize_hidden", "quantize_act",
           "dequantize_act", "dequant_weight", "swiglu", "expert_mlp"]
