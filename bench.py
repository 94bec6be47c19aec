#!/usr/bin/env python
"""Benchmark of the block-scaled MoE experts forward on GB300.

One step = one moe_experts_forward (routing, input quantization, GEMM1 with
the SwiGLU epilogue, GEMM2, combine) over the workload's synthetic batch with
every input resident in HBM. Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
  python bench.py --calibrate-fp8      # dense FP8 GEMM peak of this GPU (one JSON line)

Metric: algorithmic TFLOP/s (6 * H * I * pairs per step; padding rows are not
counted) and tokens/s of the experts forward on one GB300. The default
workload is the largest one that fits one GPU: the DeepSeek-V3-shaped FP8
prefill layer (T=8192, H=7168, I=2048, E=256, K=8, Zipf-skewed routing with
5 % skipped slots). Multi-GPU runs are independent replicas (weak scaling):
the forward has no exchange step on one GPU; `--gpus N` without a torchrun
environment re-launches itself under torchrun with N local ranks.

Legs in the line: `value` (device time, inputs already in HBM), `e2e` (the
same metric through the C ABI with pinned host buffers, copies inside the
timed region), `roofline` (the dominant kernel timed with CUDA events on the
launching stream against the measured peak), `cpu_baseline` (the fp64 oracle
on the host cores over a bounded sample), `clocks` (nvidia-smi sampled during
the timed region). `--impl reference` times the oracle alone on the host
cores, on the same workload and metric.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE experts fwd TFLOPS + tokens/s; % of FP8/FP4 TC peak or HBM BW (1 GB300)"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
DEFAULT_WORKLOAD = "dsv3_prefill_fp8"
FP8_PEAK_RECORD = os.path.join(ROOT, "profiles", "fp8_peak.json")
STAGES = ["route", "quant", "gemm1", "gemm2", "combine"]
L2_FLUSH_BYTES = 256 << 20
# nominal dense tensor rates of a GB300: fp4 13.5 PF against fp8 4.5 PF
FP4_OVER_FP8 = 3.0
ACT_NAME = {"fp8": "e4m3 1x128", "fp4": "e2m1 1x32"}
CPU_SAMPLE_TOKENS = {"mixtral_prefill_fp8": 24, "dsv3_prefill_fp8": 12, "dsv3_decode_fp8": 6, "gptoss_fp8xfp4": 24}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_fp8_peak():
    """The committed dense FP8 GEMM calibration (bench.py --calibrate-fp8 on
    a GB300), or None."""
    try:
        with open(FP8_PEAK_RECORD) as f:
            d = json.load(f)
        return d if d.get("tflops_burst") else None
    except (OSError, ValueError):
        return None


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return ws, int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


def launch_plan(gpus, env, argv, port=None):
    """How to honour --gpus N: ("run", N) inside a matching torchrun world
    (or N == 1 without one), ("spawn", cmd) to re-launch under torchrun with N
    local ranks, ("error", why) when --gpus disagrees with WORLD_SIZE."""
    if gpus < 1:
        return ("error", f"--gpus must be >= 1, got {gpus}")
    if "WORLD_SIZE" in env:
        world = int(env["WORLD_SIZE"])
        if world != gpus:
            return ("error", f"--gpus {gpus} but WORLD_SIZE={world}: launch one rank per GPU")
        return ("run", world)
    if gpus == 1:
        return ("run", 1)
    if port is None:
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={gpus}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"), *argv]
    return ("spawn", cmd)


def kernel_source_digest(sources):
    """sha256 over the GEMM kernel sources with comments and whitespace
    removed (edits to comments do not change what was measured); None if a
    file is missing."""
    import hashlib
    import re
    h = hashlib.sha256()
    for src in sources:
        try:
            with open(os.path.join(ROOT, src), encoding="utf-8") as f:
                text = f.read()
        except OSError:
            return None
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update("".join(text.split()).encode())
    return h.hexdigest()


def measured_traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    GEMM kernel sources changed since the counters were taken."""
    import glob
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic_full_size.json")) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    digest = kernel_source_digest(d.get("sources", []))
    cur = sorted(glob.glob(os.path.join(ROOT, "block_scaled_moe_expert_gb300", "csrc", "*.cuh")))
    if digest is None or len(cur) + 1 != len(d.get("sources", [])) or digest != d.get("kernel_source_sha256"):
        return None
    return d.get("bytes_per_launch", {}).get(workload, {}).get(kernel)


def max_over_ranks(x, device="cpu"):
    """Max of a float over all ranks (identity on one rank). Each rank is an
    independent replica, so the job's time is the slowest rank's time."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank, world, seconds):
    """Whole-job throughput: every rank processes the same per-rank work."""
    return world * units_per_rank / seconds


def weight_bytes_per_expert(wl, which):
    """Algorithmic bytes of one expert's weight (codes + scales)."""
    rows, k = (2 * wl.I, wl.H) if which == 13 else (wl.H, wl.I)
    if wl.fmt == "fp8":
        return rows * k + 4 * ((rows + 127) // 128) * ((k + 127) // 128)
    return rows * k // 2 + rows * (k // 32)


def launches_per_forward(wl):
    """Kernels one forward launches: one for FP4 weights with at most 8 pairs
    per expert and at most 32 slots (the single-launch forward); otherwise the
    routing (one kernel up to 8192 slots, else histogram + scan + scatter),
    the quantization kernel, GEMM1, GEMM2 and the combine (inside GEMM2 for
    FP4 weights with at most 8 pairs per expert and at most 256 slots, 64
    with FP4 activations)."""
    S = wl.T * wl.K
    decode = wl.fmt == "fp4" and S <= 8 * wl.E
    if decode and S <= 32:
        return 1  # the single-launch decode forward
    combine = 0 if (decode and S <= (64 if wl.act_fmt == "fp4" else 256)) else 1
    return (2 if S <= 8192 else 4) + 2 + combine


def routing_stats(idx_cpu, E):
    ids = idx_cpu.reshape(-1)
    valid = ids[(ids >= 0) & (ids < E)]
    return int(valid.size), int(np.unique(valid).size)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while it runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.dev = device_index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "20"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.p = None
        return self

    def __exit__(self, *a):
        if self.p is not None:
            time.sleep(0.1)
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()

    def summary(self, t0, t1):
        self.f.flush()
        rows = []
        with open(self.f.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) == 8:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        # under load: samples at the top of the observed power range
        pw = [num(r[2]) or 0.0 for r in rows]
        thr = max(pw) * 0.5 if pw else 0
        loaded = [num(r[0]) for r, p in zip(rows, pw) if p >= thr and num(r[0]) is not None] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": num(rows[0][1]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


def cpu_baseline(wl, hidden, idx, w, weights, n_tok):
    """Time the oracle (as it stands) on the first n_tok tokens."""
    import torch
    from oracle import moe as OM

    class Lazy:
        def __init__(self, t):
            self.t, self.k, self.v = t, None, None

        def __getitem__(self, e):
            if self.k != int(e):
                self.k, self.v = int(e), self.t[int(e)].cpu().numpy()
            return self.v

    wts = dict(fmt=wl.fmt, E=wl.E, H=wl.H, I=wl.I, **{k: Lazy(weights[k]) for k in
                                                        ("w13", "w13_scale", "w2", "w2_scale")})
    toks = np.arange(min(n_tok, wl.T))
    bits = hidden[:len(toks)].view(torch.int16).cpu().numpy().view(np.uint16)
    ids = idx[:len(toks)].cpu().numpy()
    ws = w[:len(toks)].cpu().numpy()
    bits_full = np.zeros((len(toks), wl.H), np.uint16)
    bits_full[:] = bits
    t0 = time.perf_counter()
    OM.experts_forward(bits_full, ids, ws, wts, wl.swiglu_limit, act_fmt=wl.act_fmt)
    dt = time.perf_counter() - t0
    pairs, _ = routing_stats(ids, wl.E)
    cores = len(os.sched_getaffinity(0))
    return {"value": 6.0 * wl.H * wl.I * pairs / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"first {len(toks)} tokens ({pairs} pairs) of {wl.name}, fp64 numpy, {dt:.1f} s",
            "tokens_per_s": len(toks) / dt}


def run_reference(args, wl):
    """Reference arm: the fp64 oracle on the host cores, per step one token."""
    ws, rank, _ = dist_env()
    if ws > 1:
        # host-only arm: the ranks meet over gloo, rank 0 alone does the work
        import torch.distributed as dist
        dist.init_process_group("gloo")
        try:
            if rank == 0:
                _reference_line(args, wl, ws)
            dist.barrier()
        finally:
            dist.destroy_process_group()
        return
    _reference_line(args, wl, ws)


def _reference_line(args, wl, ws):
    import torch
    from block_scaled_moe_expert_gb300 import workloads as W
    from oracle import moe as OM
    small = W.scaled(wl, T=min(wl.T, 64))
    hidden = W.make_hidden(small)
    idx, w = W.make_routing(small)
    # One expert's worth of synthetic weights (same shapes and distribution)
    # stands in for every expert: the oracle's cost does not depend on the
    # values, and drawing all E experts on the host would dominate the run.
    touched = sorted({int(e) for e in idx.reshape(-1).tolist() if 0 <= e < wl.E})
    one = W.make_weights(W.scaled(wl, E=1), "cpu")
    one = {k: one[k][0].numpy() for k in ("w13", "w13_scale", "w2", "w2_scale")}

    class Gen:
        def __init__(self, key):
            self.key = key

        def __getitem__(self, e):
            return one[self.key]

    wts = dict(fmt=wl.fmt, E=wl.E, H=wl.H, I=wl.I, **{k: Gen(k) for k in ("w13", "w13_scale", "w2", "w2_scale")})
    bits = hidden.view(torch.int16).numpy().view(np.uint16)
    ids = idx.numpy()
    wv = w.numpy()
    times, pairs = [], []
    for step in range(args.warmup + args.steps):
        t = step % small.T
        t0 = time.perf_counter()
        OM.experts_forward(bits, ids, wv, wts, wl.swiglu_limit, tokens=[t], act_fmt=wl.act_fmt)
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            pairs.append(routing_stats(ids[t:t + 1], wl.E)[0])
    total = sum(times)
    flops = 6.0 * wl.H * wl.I * sum(pairs)
    # the same config keys as the GPU arm: its routing is drawn on the device
    # (the device generator's stream differs from the host's), so the full
    # batch's routing is drawn there when a device exists (not timed)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    full_pairs, full_touched = routing_stats(W.make_routing(wl, dev)[0].cpu().numpy(), wl.E)
    value = flops / total / 1e12
    cores = len(os.sched_getaffinity(0))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "K": wl.K,
                       "weights": wl.fmt, "activations": ACT_NAME[wl.act_fmt], "swiglu_limit": wl.swiglu_limit,
                       "pairs": full_pairs, "touched_experts": full_touched, "parallelism": f"replicas{ws}",
                       "l2": "not applicable: the oracle runs on the host"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"one token of {wl.name} per step (synthetic expert weights), fp64 numpy"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "tokens_per_s": args.steps / total, "touched_experts_sample": len(touched)}
    print(json.dumps(line), flush=True)


def rooflines(wl, stage_ms, pairs, touched, ms_step, peaks, peak_src, fp8):
    """(roofline of the dominant kernel, roofline of the whole forward).

    Dominant kernel: the single launch where one kernel runs the forward,
    else the slower GEMM; its bound is the slower of its tensor-core time
    (algorithmic flops / dense peak of the operand types) and its HBM time
    (algorithmic bytes: touched-expert weights + activation rows in and out,
    / the copy bandwidth). The whole forward takes max(flops / tensor peak,
    bytes / HBM peak) with bytes = touched-expert weights (w13 + w2, codes
    and scales) + hidden in + output out (bf16) + ids and routing weights.
    """
    flops = 6.0 * wl.H * wl.I * pairs
    fbytes = (weight_bytes_per_expert(wl, 13) + weight_bytes_per_expert(wl, 2)) * touched \
        + 2 * wl.T * wl.H * 2 + 8 * wl.T * wl.K
    single = "single_launch" in stage_ms
    if single:
        # the single launch does the forward's work and moves its bytes
        dom = "single_launch"
        frac_1 = 1.0
        kflops = flops
        kbytes = fbytes
    else:
        dom = max(("gemm1", "gemm2"), key=lambda k: stage_ms[k])
        frac_1 = 2.0 / 3.0 if dom == "gemm1" else 1.0 / 3.0
        kflops = flops * frac_1
        wb = weight_bytes_per_expert(wl, 13 if dom == "gemm1" else 2) * touched
        # activation rows: e4m3 codes (e2m1, two per byte, with FP4
        # activations) plus one 4-byte scale word per 128 columns
        per = 2 if wl.act_fmt == "fp4" else 1
        if dom == "gemm1":
            act = pairs * (wl.H // per + 4 * ((wl.H + 127) // 128)) + pairs * (wl.I // per + 4 * ((wl.I + 127) // 128))
        else:
            act = pairs * (wl.I // per + 4 * ((wl.I + 127) // 128)) + pairs * wl.H * 4
        kbytes = wb + act
    peak_tc_2x = 2.0 * peaks["bf16_tflops"]  # fp8 dense = 2 x bf16 dense (nominal 4.5 / 2.25 PF)
    if fp8 is not None:
        peak_tc = fp8["tflops_burst"]
        tc_src = (f"measured fp8: cuBLASLt e4m3 {fp8['n']}^3 GEMM, best of {fp8['reps']} "
                  f"(profiles/fp8_peak.json); sustained {fp8['tflops_sustained']:.0f}")
    else:
        peak_tc = peak_tc_2x
        tc_src = f"{peak_src}: 2 x bf16 burst (fp8/bf16 nominal ratio 2)"
    if wl.act_fmt == "fp4":
        # e2m1 x e2m1 runs at the FP4 tensor rate: the FP8 figure above times
        # the nominal FP4 / FP8 dense ratio (13.5 / 4.5 PF)
        peak_tc *= FP4_OVER_FP8
        peak_tc_2x *= FP4_OVER_FP8
        tc_src = f"fp4 = {FP4_OVER_FP8:g} x ({tc_src}), the nominal dense fp4/fp8 ratio"
    peak_hbm = peaks["hbm_gbs"]
    t_tc = kflops / (peak_tc * 1e12)
    t_hbm = kbytes / (peak_hbm * 1e9)
    secs = stage_ms[dom] * 1e-3
    if t_tc >= t_hbm:
        achieved = kflops / secs / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak_tc, "unit": "TFLOP/s",
                "frac": achieved / peak_tc, "peak_source": tc_src,
                "frac_vs_2x_bf16": achieved / peak_tc_2x, "frac_vs_spec_5pf": achieved / 5000.0}
    else:
        achieved = kbytes / secs / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak_hbm, "unit": "GB/s", "frac": achieved / peak_hbm,
                "peak_source": f"{peak_src}: copy bandwidth", "frac_vs_spec_8tbs": achieved / 8000.0}
    alg_units = (f"{frac_1:.3f} x 6*H*I*pairs flops = {kflops / 1e9:.1f} GFLOP; touched-expert weight + "
                 f"{'hidden, output, ids and weights' if single else 'activation'} bytes = {kbytes / 1e9:.3f} GB; "
                 f"roofline times tensor {t_tc * 1e3:.3f} ms, hbm {t_hbm * 1e3:.3f} ms")
    traffic = measured_traffic(wl.name, dom)
    roof.update({"kernel": dom, "traffic": traffic, "traffic_unit": "bytes per launch" if traffic else None,
                 "kernel_ms": stage_ms[dom], "algorithmic": alg_units})
    f_tc, f_hbm = flops / (peak_tc * 1e12), fbytes / (peak_hbm * 1e9)
    fwd_roof = {"bound": "tensor" if f_tc >= f_hbm else "hbm", "roofline_ms": max(f_tc, f_hbm) * 1e3,
                "tensor_ms": f_tc * 1e3, "hbm_ms": f_hbm * 1e3, "bytes": fbytes,
                "frac": max(f_tc, f_hbm) * 1e3 / ms_step, "peaks": {"tensor_tflops": peak_tc, "hbm_gbs": peak_hbm}}
    roof["forward_frac"] = fwd_roof["frac"]
    return roof, fwd_roof


def run_ours(args, wl):
    import torch
    from block_scaled_moe_expert_gb300 import binding as B
    from block_scaled_moe_expert_gb300 import build as BLD
    from block_scaled_moe_expert_gb300 import workloads as W

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    BLD.build()
    dev = torch.device("cuda", local)
    hidden, idx, w, weights = W.make_all(wl, dev)
    # The one-shot weight transform, timed on its own (not part of a step).
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record()
    prepared = B.prepare_weights(weights, activations=wl.act_fmt)
    p1.record()
    torch.cuda.synchronize()
    prepare_ms = p0.elapsed_time(p1)
    ws = torch.empty(B.workspace_bytes(prepared.fmt, wl.T, wl.H, wl.I, wl.E, wl.K), dtype=torch.uint8, device=dev)
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    pairs, touched = routing_stats(idx.cpu().numpy(), wl.E)
    flops = 6.0 * wl.H * wl.I * pairs

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    def new_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record()
        return evs

    for _ in range(args.warmup):
        B.experts_forward(hidden, idx, w, prepared, wl.swiglu_limit, workspace=ws, out=out)
    torch.cuda.synchronize()
    if B.device_status(ws) != 0:
        raise RuntimeError("device status flags set during warm-up")

    step_ev = [new_events(2) for _ in range(args.steps)]
    stage_ev = [new_events(6) for _ in range(args.steps)]
    start, stop = new_events(2)
    # L2 flush between timed steps: a write larger than L2 (129 MB) evicts
    # the previous step's weights and activations, so every step starts cold;
    # a read of another buffer larger than L2 then replaces the dirty lines
    # with clean ones, so their write-back is not charged to the next step.
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def flush_l2(s):
        flush.fill_(s & 0xFF)
        flush_r.sum()
    torch.cuda.synchronize()
    peaks, peak_src = load_peaks()
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        t_wall0 = time.time()
        start.record()
        for s in range(args.steps):
            flush_l2(s)
            step_ev[s][0].record()
            B.experts_forward(hidden, idx, w, prepared, wl.swiglu_limit, workspace=ws, out=out)
            step_ev[s][1].record()
        stop.record()
        torch.cuda.synchronize()
        barrier()
        t_wall1 = time.time()
        # Per-kernel times: the same steps again through the entry point that
        # records an event at every stage boundary (the events sit between
        # the kernels, so this pass is kept out of the headline number).
        for s in range(args.steps):
            flush_l2(s)
            B.experts_forward_timed(hidden, idx, w, prepared, stage_ev[s], wl.swiglu_limit, workspace=ws, out=out)
        torch.cuda.synchronize()
    clocks = clk.summary(t_wall0, t_wall1)
    # Device time of the forwards alone (the flushes between steps are
    # outside the per-step events), max over ranks.
    fwd_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    total_ms = max_over_ranks(fwd_ms, dev)
    ms_step = total_ms / args.steps
    region_ms = start.elapsed_time(stop)
    del flush, flush_r
    stage_ms = {name: statistics.fmean(ev[i].elapsed_time(ev[i + 1]) for ev in stage_ev)
                for i, name in enumerate(STAGES)}
    status = B.device_status(ws)

    # e2e: every step copies its inputs from pinned host memory and reads its
    # result back, inside the timed region. The copies run on two copy
    # streams (host->device, device->host) with two buffer sets, so step i+1's
    # inputs land and step i-1's result leaves while step i computes, as a
    # serving loop would do.
    e2e = None
    if not args.no_e2e:
        nb = 2
        h_hidden = hidden.cpu().pin_memory()
        h_idx = idx.cpu().pin_memory()
        h_w = w.cpu().pin_memory()
        h_out = [torch.empty(wl.T, wl.H, dtype=torch.bfloat16).pin_memory() for _ in range(nb)]
        d_in = [(torch.empty_like(hidden), torch.empty_like(idx), torch.empty_like(w)) for _ in range(nb)]
        d_out = [torch.empty_like(out) for _ in range(nb)]
        sc = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(args.steps)]
        ev_done = [torch.cuda.Event() for _ in range(args.steps)]
        ev_back = [torch.cuda.Event() for _ in range(args.steps)]
        e0, e1 = new_events(2)
        torch.cuda.synchronize()
        barrier()
        e0.record(sc)
        s_in.wait_stream(sc)
        s_out.wait_stream(sc)
        for i in range(args.steps):
            b = i % nb
            with torch.cuda.stream(s_in):
                if i >= nb:
                    s_in.wait_event(ev_done[i - nb])  # step i-2 no longer reads this input set
                d_in[b][0].copy_(h_hidden, non_blocking=True)
                d_in[b][1].copy_(h_idx, non_blocking=True)
                d_in[b][2].copy_(h_w, non_blocking=True)
                ev_in[i].record(s_in)
            sc.wait_event(ev_in[i])
            if i >= nb:
                sc.wait_event(ev_back[i - nb])  # step i-2's result has left this output buffer
            B.experts_forward(d_in[b][0], d_in[b][1], d_in[b][2], prepared, wl.swiglu_limit, workspace=ws,
                              out=d_out[b])
            ev_done[i].record(sc)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[i])
                h_out[b].copy_(d_out[b], non_blocking=True)
                ev_back[i].record(s_out)
        sc.wait_stream(s_out)
        e1.record(sc)
        torch.cuda.synchronize()
        if not torch.equal(h_out[(args.steps - 1) % nb], out.cpu()):
            raise RuntimeError("end-to-end result differs from the device-resident run")
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dev) / args.steps
        e2e = {"value": replica_throughput(flops, world, e2e_ms * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": hidden.numel() * 2 + idx.numel() * 4 + w.numel() * 4,
               "d2h_bytes_per_step": out.numel() * 2, "ms_per_step": e2e_ms,
               "pipeline": "pinned host buffers; H2D and D2H on two copy streams overlapped with the "
                           "neighbouring steps' compute (2 buffer sets)"}

    # Rooflines of the dominant kernel and of the whole forward
    if launches_per_forward(wl) == 1:
        # one kernel runs the whole forward (its time lands in the first
        # stage; the later events are recorded back to back)
        stage_ms["single_launch"] = stage_ms["route"]
    roof, fwd_roof = rooflines(wl, stage_ms, pairs, touched, ms_step, peaks, peak_src, load_fp8_peak())

    line = {"metric": METRIC, "value": replica_throughput(flops, world, ms_step * 1e-3) / 1e12, "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e2m1" if wl.act_fmt == "fp4" else ("e4m3" if wl.fmt == "fp8" else "e4m3xe2m1"),
            "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "K": wl.K,
                       "weights": wl.fmt, "activations": ACT_NAME[wl.act_fmt], "swiglu_limit": wl.swiglu_limit,
                       "pairs": pairs,
                       "touched_experts": touched, "parallelism": f"replicas{world}",
                       "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write, then a "
                             f"{L2_FLUSH_BYTES >> 20} MiB read); expert weights also exceed L2"},
            "tokens_per_s": replica_throughput(wl.T, world, ms_step * 1e-3),
            "stage_ms": stage_ms, "prepare_ms_once": prepare_ms, "region_ms_incl_flush": region_ms, "roofline": roof,
            "forward_roofline": fwd_roof, "gpu_launches": launches_per_forward(wl) * args.steps, "clocks": clocks,
            "device_status": status}
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, hidden, idx, w, weights,
                                            args.cpu_tokens or CPU_SAMPLE_TOKENS.get(wl.name, 4))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def calibrate_fp8(args):
    """Dense FP8 tensor-core peak of this GPU: torch._scaled_mm (cuBLASLt) on
    e4m3 n x n x n with per-tensor scales and a bf16 output, best of `reps`
    back-to-back launches timed with CUDA events (burst), then launches back
    to back for about 4 s (sustained, under the power cap), with the clocks
    sampled meanwhile. Prints one JSON line."""
    import torch
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    n, reps = 8192, 10
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn).t()  # column-major operand
    one = torch.ones((), device=dev)

    def mm():
        return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    for _ in range(5):
        mm()
    torch.cuda.synchronize()
    flop = 2.0 * n ** 3
    best = float("inf")
    with ClockSampler(0) as clk:
        t_wall0 = time.time()
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            mm()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        # sustained: batches of 50 launches until about 4 s have passed
        iters, ms = 0, 0.0
        while ms < 4000.0:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(50):
                mm()
            e1.record()
            torch.cuda.synchronize()
            ms += e0.elapsed_time(e1)
            iters += 50
        t_wall1 = time.time()
    clocks = clk.summary(t_wall0, t_wall1)
    line = {"what": "dense FP8 (e4m3) GEMM peak", "how": "torch._scaled_mm (cuBLASLt), per-tensor scales, "
            "bf16 out, CUDA events", "n": n, "reps": reps, "tflops_burst": flop / (best * 1e-3) / 1e12,
            "tflops_sustained": flop * iters / (ms * 1e-3) / 1e12, "sustained_s": ms / 1e3,
            "gpu": torch.cuda.get_device_name(0), "torch": torch.__version__, "clocks": clocks}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--calibrate-fp8", action="store_true", help="measure the dense FP8 GEMM peak and exit")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=0)
    ap.add_argument("--tokens", type=int, default=0, help="override T (smaller profiling cases)")
    ap.add_argument("--experts", type=int, default=0, help="override E (smaller profiling cases)")
    args = ap.parse_args()
    if args.calibrate_fp8:
        calibrate_fp8(args)
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    plan = launch_plan(args.gpus, os.environ, sys.argv[1:])
    if plan[0] == "error":
        raise SystemExit(plan[1])
    if plan[0] == "spawn":
        raise SystemExit(subprocess.call(plan[1]))
    from block_scaled_moe_expert_gb300 import workloads as W
    wl = W.WORKLOADS[args.workload]
    # a changed shape is another workload: its name says so, and the per-launch
    # DRAM record of the named workload does not apply to it
    if args.tokens:
        wl = W.scaled(wl, T=args.tokens, name=f"{wl.name}@T{args.tokens}")
    if args.experts:
        wl = W.scaled(wl, E=args.experts, name=f"{wl.name}@E{args.experts}")
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
