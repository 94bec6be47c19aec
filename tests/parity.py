"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle
on the same bytes, compare with the tolerances of the method's statement.

Tolerances (bf16 output vs the fp64 oracle):
* relative Frobenius error <= 2e-3;
* elementwise: max(0, |gpu - ref| - ulp_bf16(ref) / 2) <= 1e-2 * RMS(ref).
  The half-ulp allowance is the reading taken for the max-error bound: the
  bf16 output alone cannot meet 1e-2 * RMS for |ref| > 2.56 * RMS, so the
  bound applies to the error beyond the unavoidable final rounding.
"""
import numpy as np
import torch

import oracle.moe as OM
from oracle import formats as OF
from block_scaled_moe_expert_gb300 import binding as B
from block_scaled_moe_expert_gb300 import workloads as W

REL_FRO = 2e-3
MAX_REL_RMS = 1e-2


class LazyExperts:
    """Indexable by expert: copies one expert's weights to host on demand."""

    def __init__(self, t):
        self.t = t
        self.cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache = {e: self.t[e].cpu().numpy()}
        return self.cache[e]


def oracle_weights(weights):
    return dict(fmt=weights["fmt"], E=weights["E"], H=weights["H"], I=weights["I"],
                w13=LazyExperts(weights["w13"]), w13_scale=LazyExperts(weights["w13_scale"]),
                w2=LazyExperts(weights["w2"]), w2_scale=LazyExperts(weights["w2_scale"]))


def bits_of(hidden):
    return hidden.view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_out(hidden, idx, w, weights, limit, tokens=None, act_fmt="fp8"):
    return OM.experts_forward(bits_of(hidden), idx.cpu().numpy(), w.cpu().numpy(), oracle_weights(weights),
                              limit, tokens=tokens, act_fmt=act_fmt)


def oracle_out_parallel(hidden, idx, w, weights, limit, tokens, threads=None, act_fmt="fp8"):
    """oracle_out for many tokens of a large workload, expert groups in threads.

    The pairs of the selected tokens are split by expert into groups; each
    group runs the oracle on its own (the other slots masked to -1, i.e.
    skipped) and the groups' fp64 outputs are added. Only the order of the
    fp64 additions across groups changes (relative effect ~1e-16, far below
    the bf16 tolerances); every expert is dequantized once. numpy releases
    the GIL in the heavy steps, so threads overlap the per-expert work.
    """
    import os
    from concurrent.futures import ThreadPoolExecutor
    ids = idx.cpu().numpy()
    sel = ids[np.asarray(tokens)]
    experts = np.unique(sel[(sel >= 0) & (sel < weights["E"])])
    threads = threads or max(1, min(8, os.cpu_count() or 1))
    groups = [experts[i::2 * threads] for i in range(min(len(experts), 2 * threads))]
    bits = bits_of(hidden)
    wv = w.cpu().numpy()

    def run(group):
        masked = np.where(np.isin(ids, group), ids, -1).astype(ids.dtype)
        return OM.experts_forward(bits, masked, wv, oracle_weights(weights), limit, tokens=tokens, act_fmt=act_fmt)

    out = np.zeros((len(tokens), bits.shape[1]), dtype=np.float64)
    if not groups:
        return out
    with ThreadPoolExecutor(threads) as ex:
        for part in ex.map(run, groups):
            out += part
    return out


def sample_tokens(idx, E, n, seed):
    """At least n tokens (fewer if T < n): the first and last token, one token
    for every expert the batch touches (rarest expert first, each time the
    earliest holder in a seeded order), then seeded random tokens."""
    ids = idx.cpu().numpy()
    T = ids.shape[0]
    rng = np.random.default_rng(seed)
    order = rng.permutation(T)
    pos = np.empty(T, dtype=np.int64)
    pos[order] = np.arange(T)
    chosen = {0, T - 1}
    covered = set(int(e) for t in chosen for e in ids[t])
    valid = (ids >= 0) & (ids < E)
    counts = np.bincount(ids[valid], minlength=E)
    for e in np.argsort(counts, kind="stable"):
        if counts[e] == 0 or int(e) in covered:
            continue
        holders = np.flatnonzero((ids == e).any(axis=1))
        t = int(holders[np.argmin(pos[holders])])
        chosen.add(t)
        covered.update(int(x) for x in ids[t])
    for t in order:
        if len(chosen) >= n:
            break
        chosen.add(int(t))
    return sorted(chosen)


def compare(gpu_bf16, ref):
    g = gpu_bf16.float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    nrm = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(g - ref) / nrm) if nrm > 0 else float(np.abs(g).max())
    _, E = np.frexp(ref)
    half_ulp = np.ldexp(1.0, np.maximum(E - 8, -133)) / 2
    excess = np.maximum(np.abs(g - ref) - half_ulp, 0.0)
    raw = float(np.abs(g - ref).max()) if g.size else 0.0
    return dict(rel_fro=rel, max_excess_over_rms=float(excess.max() / rms) if rms > 0 else float(excess.max()),
                max_raw_over_rms=raw / rms if rms > 0 else raw, rms=rms, finite=bool(np.isfinite(g).all()))


def assert_close(gpu_bf16, ref, what=""):
    m = compare(gpu_bf16, ref)
    assert m["finite"], (what, m)
    assert m["rel_fro"] <= REL_FRO, (what, m)
    assert m["max_excess_over_rms"] <= MAX_REL_RMS, (what, m)
    return m


def lib_fmt(wl):
    """The library's format name for a workload (weights + activations)."""
    return "fp4_act_fp4" if wl.act_fmt == "fp4" else wl.fmt


def run_cuda(wl, device="cuda", hidden=None, idx=None, w=None, weights=None, prepared=None):
    hidden = W.make_hidden(wl, device) if hidden is None else hidden
    if idx is None:
        idx, w = W.make_routing(wl, device)
    weights = W.make_weights(wl, device) if weights is None else weights
    prepared = B.prepare_weights(weights, activations=wl.act_fmt) if prepared is None else prepared
    ws = torch.empty(B.workspace_bytes(prepared.fmt, wl.T, wl.H, wl.I, wl.E, wl.K), dtype=torch.uint8,
                     device=device)
    out = B.experts_forward(hidden, idx, w, prepared, wl.swiglu_limit, workspace=ws)
    torch.cuda.synchronize()
    return dict(hidden=hidden, idx=idx, w=w, weights=weights, prepared=prepared, ws=ws, out=out)


def ws_region(ws, layout, name, dtype, count):
    off = getattr(layout, name)
    nbytes = count * torch.empty(0, dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype)


def sf_exponents(words_u32, rows, nblk):
    """Read the per-(row, block) exponents out of the scale-word layout."""
    w = words_u32.cpu().numpy().astype(np.int64)
    r = np.arange(rows)[:, None]
    b = np.arange(nblk)[None, :]
    idx = ((r // 128) * nblk + b) * 128 + 4 * (r % 32) + (r % 128) // 32
    return (w[idx] & 0xFF) - 127


def sf_exponents_1x32(words_u32, rows, nblk):
    """FP4 activations: the exponent of every 1x32 block, [rows, 4 * nblk]
    (byte j of the (row, 128-column block) word is sub-block j)."""
    w = words_u32.cpu().numpy().astype(np.int64)
    r = np.arange(rows)[:, None]
    b = np.arange(nblk)[None, :]
    idx = ((r // 128) * nblk + b) * 128 + 4 * (r % 32) + (r % 128) // 32
    words = w[idx]
    return np.stack([((words >> (8 * j)) & 0xFF) - 127 for j in range(4)], axis=2).reshape(rows, 4 * nblk)


def unpack_e2m1(packed_u8, cols):
    """Packed e2m1 bytes [R, cols / 2] -> 4-bit codes [R, cols] (even column in the low nibble)."""
    b = np.asarray(packed_u8, dtype=np.uint8)
    c = np.empty((b.shape[0], 2 * b.shape[1]), dtype=np.uint8)
    c[:, 0::2] = b & 0xF
    c[:, 1::2] = b >> 4
    return c[:, :cols]


__all__ = ["oracle_out", "oracle_out_parallel", "sample_tokens", "compare", "assert_close", "run_cuda", "ws_region",
           "sf_exponents", "sf_exponents_1x32", "unpack_e2m1", "lib_fmt", "bits_of", "OF", "OM", "W", "B"]
