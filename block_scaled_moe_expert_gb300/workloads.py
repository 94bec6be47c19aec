"""Seeded synthetic workloads for the experts forward (inputs only).

This module draws inputs; it holds none of the forward's arithmetic. Both the
CUDA path and the CPU oracle consume the bytes it produces, so it must stay
free of anything either side computes.

Shapes stand in for the model families the transformers pages test the
experts path on (Mixtral, DeepSeek-V3, GPT-OSS); no checkpoint or dataset is
used, every tensor is drawn from a seeded generator:

* hidden states: bf16 ~ N(0, 1), [T, H];
* routing: either softmax top-K over N(0, std) logits (weights renormalised
  over the kept K), or a Zipf(s) expert choice over a seeded permutation of
  the experts, K distinct per token (Gumbel top-K, i.e. sampling without
  replacement with probability proportional to rank^-s), with
  sigmoid-normalised weights w = sigmoid(z) / sum(sigmoid(z)), z ~ N(0, 1);
  a fraction of slots may then be set to -1 (skipped), keeping their weight;
* weights from N(0, 0.02) masters, stored in the format the forward takes:
  FP8 -- e4m3 codes with one fp32 scale per 128x128 block, scale = amax/448;
  FP4 -- e2m1 codes packed two per byte (low nibble = even K index) with one
  UE8M0 byte per 1x32 block, exponent n = min{n : amax <= 6 * 2^n}.

``act_fmt`` names the activation format the forward is asked to use ("fp8":
e4m3 1x128, the pages' rule; "fp4": the FP4 x FP4 variant). It selects the
computation, not the inputs: the drawn bytes are the same.
"""
import math
from dataclasses import dataclass, field

import torch

FP8 = "fp8"
FP4 = "fp4"


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    K: int
    fmt: str
    router: str            # "softmax" | "zipf_sigmoid"
    logit_std: float = 1.0
    zipf_s: float = 1.1
    skip_frac: float = 0.0
    swiglu_limit: float | None = None
    seed: int = 1000
    act_fmt: str = "fp8"   # "fp8" | "fp4" (FP4 weights only)

    @property
    def S(self):
        return self.T * self.K


def _w(name, T, H, I, E, K, fmt, router, seed, **kw):
    return Workload(name=name, T=T, H=H, I=I, E=E, K=K, fmt=fmt, router=router, seed=seed, **kw)


WORKLOADS = {
    "tiny_fp8": _w("tiny_fp8", 16, 256, 128, 8, 2, FP8, "softmax", 1000),
    "mixtral_prefill_fp8": _w("mixtral_prefill_fp8", 4096, 4096, 14336, 8, 2, FP8, "softmax", 1001),
    "dsv3_decode_fp8": _w("dsv3_decode_fp8", 128, 7168, 2048, 256, 8, FP8, "zipf_sigmoid", 1002,
                          skip_frac=0.05),
    "dsv3_prefill_fp8": _w("dsv3_prefill_fp8", 8192, 7168, 2048, 256, 8, FP8, "zipf_sigmoid", 1002,
                           skip_frac=0.05),
    "gptoss_fp8xfp4": _w("gptoss_fp8xfp4", 8192, 2880, 2880, 128, 4, FP4, "softmax", 1003,
                         logit_std=1.5, swiglu_limit=7.0),
}
for _t in (1, 8, 32, 128, 512, 2048):
    WORKLOADS[f"dsv3_decode_fp4_T{_t}"] = _w(f"dsv3_decode_fp4_T{_t}", _t, 7168, 2048, 256, 8, FP4,
                                             "zipf_sigmoid", 1004)
# The FP4 x FP4 variant (e2m1 activations) on the GPT-OSS and DeepSeek-V3
# decode shapes: same inputs as their FP8-activation counterparts.
WORKLOADS["gptoss_fp4xfp4"] = _w("gptoss_fp4xfp4", 8192, 2880, 2880, 128, 4, FP4, "softmax", 1003,
                                 logit_std=1.5, swiglu_limit=7.0, act_fmt=FP4)
for _t in (1, 128):
    WORKLOADS[f"dsv3_decode_fp4xfp4_T{_t}"] = _w(f"dsv3_decode_fp4xfp4_T{_t}", _t, 7168, 2048, 256, 8, FP4,
                                                 "zipf_sigmoid", 1004, act_fmt=FP4)


def scaled(wl: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (e.g. fewer tokens)."""
    d = dict(wl.__dict__)
    d.update(changes)
    return Workload(**d)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_hidden(wl: Workload, device="cpu"):
    g = _gen(device, wl.seed * 7 + 1)
    return torch.randn(wl.T, wl.H, generator=g, device=device).to(torch.bfloat16)


def make_routing(wl: Workload, device="cpu"):
    """(topk_idx int32 [T, K], topk_w float32 [T, K])."""
    g = _gen(device, wl.seed * 7 + 2)
    T, E, K = wl.T, wl.E, wl.K
    if wl.router == "softmax":
        logits = torch.randn(T, E, generator=g, device=device) * wl.logit_std
        top, idx = torch.topk(logits, K, dim=1)
        w = torch.softmax(top, dim=1)
    elif wl.router == "zipf_sigmoid":
        perm = torch.randperm(E, generator=g, device=device)
        rank = torch.empty(E, device=device)
        rank[perm] = torch.arange(1, E + 1, device=device, dtype=torch.float32)
        u = torch.rand(T, E, generator=g, device=device).clamp_(1e-12, 1 - 1e-7)
        gumbel = -torch.log(-torch.log(u))
        _, idx = torch.topk(-wl.zipf_s * torch.log(rank)[None, :] + gumbel, K, dim=1)
        z = torch.randn(T, K, generator=g, device=device)
        sz = torch.sigmoid(z)
        w = sz / sz.sum(dim=1, keepdim=True)
    else:
        raise ValueError(wl.router)
    idx = idx.to(torch.int32)
    if wl.skip_frac > 0:
        drop = torch.rand(T, K, generator=g, device=device) < wl.skip_frac
        idx = torch.where(drop, torch.full_like(idx, -1), idx)
    return idx.contiguous(), w.to(torch.float32).contiguous()


def _fp8_blocks(master):
    """e4m3 codes + fp32 scales per 128x128 block (scale = amax / 448)."""
    R, C = master.shape
    rb, cb = math.ceil(R / 128), math.ceil(C / 128)
    pad = torch.zeros(rb * 128, cb * 128, device=master.device, dtype=torch.float32)
    pad[:R, :C] = master
    blk = pad.view(rb, 128, cb, 128)
    amax = blk.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (blk / scale[:, None, :, None]).to(torch.float8_e4m3fn)
    q = q.view(rb * 128, cb * 128)[:R, :C].contiguous().view(torch.uint8)
    return q, scale.contiguous()


_E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _fp4_blocks(master):
    """e2m1 codes packed two per byte + UE8M0 bytes per 1x32 block."""
    R, C = master.shape
    assert C % 32 == 0
    blk = master.view(R, C // 32, 32)
    amax = blk.abs().amax(dim=2)
    m, ex = torch.frexp(amax)
    n = torch.where(m <= 0.75, ex - 3, ex - 2)
    n = torch.where(amax == 0, torch.zeros_like(n), n).clamp(-127, 127)
    v = blk * torch.pow(2.0, -n.to(torch.float32))[:, :, None]
    mags = torch.tensor(_E2M1_MAG, device=master.device)
    a = v.abs().clamp(max=6.0)
    hi = torch.searchsorted(mags, a.contiguous(), right=False).clamp(max=7)
    lo = (hi - 1).clamp(min=0)
    d_hi = mags[hi] - a
    d_lo = a - mags[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = torch.where(pick_hi, hi, lo)
    code = code | (torch.signbit(v).to(code.dtype) << 3)
    code = code.view(R, C).to(torch.uint8)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).contiguous()
    return packed, (n + 127).to(torch.uint8).contiguous()


def make_weights(wl: Workload, device="cpu"):
    """dict(fmt, E, H, I, w13, w13_scale, w2, w2_scale) as torch tensors."""
    E, H, I = wl.E, wl.H, wl.I
    if wl.fmt == FP8:
        w13 = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=device)
        w13s = torch.empty(E, math.ceil(2 * I / 128), math.ceil(H / 128), device=device)
        w2 = torch.empty(E, H, I, dtype=torch.uint8, device=device)
        w2s = torch.empty(E, math.ceil(H / 128), math.ceil(I / 128), device=device)
        enc = _fp8_blocks
    else:
        w13 = torch.empty(E, 2 * I, H // 2, dtype=torch.uint8, device=device)
        w13s = torch.empty(E, 2 * I, H // 32, dtype=torch.uint8, device=device)
        w2 = torch.empty(E, H, I // 2, dtype=torch.uint8, device=device)
        w2s = torch.empty(E, H, I // 32, dtype=torch.uint8, device=device)
        enc = _fp4_blocks
    for e in range(E):
        g = _gen(device, wl.seed * 1009 + e)
        m13 = torch.randn(2 * I, H, generator=g, device=device) * 0.02
        m2 = torch.randn(H, I, generator=g, device=device) * 0.02
        w13[e], w13s[e] = enc(m13)
        w2[e], w2s[e] = enc(m2)
        del m13, m2
    return dict(fmt=wl.fmt, E=E, H=H, I=I, w13=w13, w13_scale=w13s, w2=w2, w2_scale=w2s)


def make_all(wl: Workload, device="cpu"):
    hidden = make_hidden(wl, device)
    idx, w = make_routing(wl, device)
    weights = make_weights(wl, device)
    return hidden, idx, w, weights
