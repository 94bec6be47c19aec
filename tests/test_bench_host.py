"""CPU: host logic of bench.py.

* the number of kernel launches a forward makes (bench.py reports it as
  gpu_launches) follows the thresholds compiled into the library;
* the digest that keys the committed DRAM-traffic record ignores comments
  and whitespace but not code, and is None when a source is missing;
* the algorithmic weight bytes per expert, against sizes worked out by hand
  from the two weight formats;
* the reference arm (`--impl reference`, the oracle on the host) prints one
  JSON line with the contract's keys and the GPU arm's config keys.
"""
import json
import os
import re
import subprocess
import sys

import bench
from block_scaled_moe_expert_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_scaled_moe_expert_gb300", "csrc")


def _const(name, fname):
    m = re.search(rf"constexpr int {name} = (\d+);", open(os.path.join(CSRC, fname)).read())
    assert m, name
    return int(m.group(1))


def test_launch_count_follows_the_library_thresholds():
    fused = _const("kFusedCombineSlots", "moe_internal.cuh")
    per_expert = _const("kDecodePairsPerExpert", "moe_internal.cuh")
    single = _const("kSingleCtaSlots", "route.cu")

    def wl(T, K, E, fmt):
        return W.Workload("case", T, 256, 128, E, K, fmt, "softmax", seed=1)

    # routing (one kernel, or histogram + scan + scatter) + quantization
    assert bench.launches_per_forward(wl(fused, 1, 8, "fp8")) == 2 + 2 + 1
    assert bench.launches_per_forward(wl(single, 1, 8, "fp8")) == 2 + 2 + 1
    assert bench.launches_per_forward(wl(single + 1, 1, 8, "fp8")) == 4 + 2 + 1
    # FP4 decode mode (at most per_expert pairs per expert) with at most
    # `fused` slots: the combine runs inside GEMM2; with at most `one` slots
    # the whole forward is one launch
    one = _const("kSingleLaunchSlots", "moe_internal.cuh")
    E = fused // per_expert
    assert bench.launches_per_forward(wl(fused, 1, E, "fp4")) == 2 + 2
    assert bench.launches_per_forward(wl(one, 1, E, "fp4")) == 1
    assert bench.launches_per_forward(wl(one + 1, 1, E, "fp4")) == 2 + 2
    assert bench.launches_per_forward(wl(fused, 1, E, "fp8")) == 2 + 2 + 1
    assert bench.launches_per_forward(wl(fused, 1, E - 1, "fp4")) == 2 + 2 + 1  # not decode mode
    assert bench.launches_per_forward(wl(fused + 1, 1, 4 * E, "fp4")) == 2 + 2 + 1  # decode, separate combine
    # FP4 activations: the single launch up to `one` slots, the decode mode's
    # fused combine up to `fused4` slots
    fused4 = _const("kFusedCombineSlotsFp4Act", "moe_internal.cuh")
    assert bench.launches_per_forward(W.scaled(wl(one, 1, E, "fp4"), act_fmt="fp4")) == 1
    assert bench.launches_per_forward(W.scaled(wl(fused4, 1, E, "fp4"), act_fmt="fp4")) == 2 + 2
    assert bench.launches_per_forward(W.scaled(wl(fused4 + 1, 1, E, "fp4"), act_fmt="fp4")) == 2 + 2 + 1
    assert bench.launches_per_forward(W.scaled(wl(single + 1, 1, E, "fp4"), act_fmt="fp4")) == 4 + 2 + 1
    # every named workload is one of these cases
    for name, w in W.WORKLOADS.items():
        S = w.T * w.K
        decode = w.fmt == "fp4" and S <= per_expert * w.E
        if decode and S <= one:
            assert bench.launches_per_forward(w) == 1, name
        else:
            front = 2 if S <= single else 4
            lim = fused4 if w.act_fmt == "fp4" else fused
            assert bench.launches_per_forward(w) == front + 2 + (0 if decode and S <= lim else 1), name


def test_traffic_digest_ignores_comments_but_not_code(tmp_path, monkeypatch):
    src = "block_scaled_moe_expert_gb300/csrc/gemm.cu"
    text = open(os.path.join(ROOT, src)).read()
    d = tmp_path / "block_scaled_moe_expert_gb300" / "csrc"
    d.mkdir(parents=True)
    f = d / "gemm.cu"
    f.write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_source_digest([src])
    assert base is not None
    f.write_text(text.replace("// Grouped block-scaled GEMMs", "//   Grouped   GEMMs, reworded") +
                 "\n/* a trailing\n   block comment */\n\n")
    assert bench.kernel_source_digest([src]) == base
    needle = "kThreads = 384;"
    assert needle in text
    f.write_text(text.replace(needle, "kThreads = 256;"))
    assert bench.kernel_source_digest([src]) != base
    f.unlink()
    assert bench.kernel_source_digest([src]) is None


def test_weight_bytes_per_expert_by_hand():
    mix = W.WORKLOADS["mixtral_prefill_fp8"]  # H 4096, I 14336, FP8 + fp32 per 128x128
    assert bench.weight_bytes_per_expert(mix, 13) == 28672 * 4096 + 4 * 224 * 32
    assert bench.weight_bytes_per_expert(mix, 2) == 4096 * 14336 + 4 * 32 * 112
    oss = W.WORKLOADS["gptoss_fp8xfp4"]  # H = I = 2880, FP4 + one byte per 1x32
    assert bench.weight_bytes_per_expert(oss, 13) == 5760 * 1440 + 5760 * 90
    assert bench.weight_bytes_per_expert(oss, 2) == 2880 * 1440 + 2880 * 90


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_fp8", "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert (d["n_gpus"], d["steps"], d["warmup"], d["vs_baseline"]) == (1, 3, 3, None)
    assert d["dtype"] == "f64" and d["data"] == "synthetic" and d["scaling"] == "weak"
    assert set(d["config"]) == {"workload", "T", "H", "I", "E", "K", "weights", "swiglu_limit", "pairs",
                                "touched_experts", "parallelism", "l2", "activations"}
    assert d["config"]["workload"] == "tiny_fp8" and d["config"]["pairs"] == 32
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_gpus_flag_plan():
    """--gpus N: runs in place inside a matching torchrun world (or alone for
    N = 1), re-launches under torchrun with N local ranks otherwise, and
    refuses a world size that disagrees."""
    assert bench.launch_plan(1, {}, []) == ("run", 1)
    assert bench.launch_plan(4, {"WORLD_SIZE": "4"}, []) == ("run", 4)
    kind, why = bench.launch_plan(8, {"WORLD_SIZE": "2"}, [])
    assert kind == "error" and "WORLD_SIZE=2" in why
    assert bench.launch_plan(0, {}, [])[0] == "error"
    kind, cmd = bench.launch_plan(2, {}, ["--gpus", "2", "--steps", "3"], port=29555)
    assert kind == "spawn"
    assert cmd[1:3] == ["-m", "torch.distributed.run"] and "--nproc-per-node=2" in cmd
    assert "--master-addr=127.0.0.1" in cmd and cmd[-4:] == ["--gpus", "2", "--steps", "3"]


def test_gpus_flag_mismatch_exits_nonzero():
    env = dict(os.environ, WORLD_SIZE="2", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "4",
                        "--workload", "tiny_fp8", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode != 0 and "WORLD_SIZE=2" in r.stderr


def test_gpus_flag_spawns_gloo_ranks():
    """bench.py --gpus 2 without torchrun re-launches itself with 2 local
    ranks; on the host-only reference arm they meet over gloo and rank 0
    prints the one JSON line, with n_gpus = 2."""
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR",
                                                            "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "tiny_fp8", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["config"]["parallelism"] == "replicas2"


def test_shape_overrides_rename_the_workload(monkeypatch):
    """--tokens / --experts give another workload: its name changes, so the
    DRAM record of the named full-size workload is not reported for it."""
    seen = {}

    def fake_run(args, wl):
        seen["wl"] = wl

    monkeypatch.setattr(bench, "run_ours", fake_run)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", "dsv3_decode_fp4_T1", "--experts", "64",
                                      "--tokens", "2"])
    bench.main()
    wl = seen["wl"]
    assert (wl.T, wl.E) == (2, 64) and wl.name == "dsv3_decode_fp4_T1@T2@E64"
    assert bench.measured_traffic(wl.name, "single_launch") is None
    assert bench.measured_traffic("dsv3_decode_fp4_T1", "single_launch") is not None


PEAKS = {"bf16_tflops": 2000.0, "hbm_gbs": 7000.0}
FP8 = {"tflops_burst": 3500.0, "tflops_sustained": 3300.0, "n": 8192, "reps": 10}


def test_roofline_tensor_bound_prefill_by_hand():
    wl = W.WORKLOADS["mixtral_prefill_fp8"]  # H 4096, I 14336, 8 experts
    sm = {"route": 0.02, "quant": 0.02, "gemm1": 0.75, "gemm2": 0.41, "combine": 0.03}
    roof, fwd = bench.rooflines(wl, sm, 8192, 8, 1.25, PEAKS, "test", FP8)
    flops1 = 4 * 4096 * 14336 * 8192  # GEMM1: 2 * pairs * H * 2I
    assert roof["kernel"] == "gemm1" and roof["bound"] == "tensor" and roof["peak"] == 3500.0
    assert abs(roof["achieved"] - flops1 / 0.75e-3 / 1e12) < 1e-9
    assert abs(roof["frac_vs_2x_bf16"] - roof["achieved"] / 4000.0) < 1e-12
    # forward: 6 H I pairs at 3500 TFLOP/s against 1.25 ms
    assert fwd["bound"] == "tensor"
    assert abs(fwd["frac"] - (6 * 4096 * 14336 * 8192 / 3500e12) / 1.25e-3) < 1e-12


def test_roofline_hbm_bound_decode_by_hand():
    wl = W.WORKLOADS["dsv3_decode_fp4_T128"]  # H 7168, I 2048, FP4 weights
    sm = {"route": 0.015, "quant": 0.01, "gemm1": 0.52, "gemm2": 0.27, "combine": 0.012}
    roof, _ = bench.rooflines(wl, sm, 1024, 190, 0.81, PEAKS, "test", FP8)
    w13 = 4096 * 7168 // 2 + 4096 * (7168 // 32)  # e2m1 codes + one UE8M0 byte per 32
    act = 1024 * (7168 + 4 * 56) + 1024 * (2048 + 4 * 16)  # e4m3 rows + scale words, in and out
    assert roof["kernel"] == "gemm1" and roof["bound"] == "hbm" and roof["peak"] == 7000.0
    assert abs(roof["achieved"] - (190 * w13 + act) / 0.52e-3 / 1e9) < 1e-6


def test_roofline_fp4_activations_and_single_launch_by_hand():
    wl = W.WORKLOADS["gptoss_fp4xfp4"]  # H = I = 2880, e2m1 activations
    sm = {"route": 0.02, "quant": 0.04, "gemm1": 0.36, "gemm2": 0.21, "combine": 0.07}
    roof, fwd = bench.rooflines(wl, sm, 32768, 128, 0.70, PEAKS, "test", FP8)
    assert fwd["peaks"]["tensor_tflops"] == 3 * 3500.0  # FP4 rate: 3 x the FP8 figure
    w13 = 5760 * 1440 + 5760 * 90
    act = 32768 * (1440 + 4 * 23) + 32768 * (1440 + 4 * 23)  # e2m1 rows: half a byte per element
    assert roof["bound"] == "hbm" and abs(roof["achieved"] - (128 * w13 + act) / 0.36e-3 / 1e9) < 1e-6
    # one launch: the forward's flops and bytes against the launch's time
    one = W.WORKLOADS["dsv3_decode_fp4_T1"]
    sm1 = {"route": 0.066, "quant": 0.002, "gemm1": 0.002, "gemm2": 0.002, "combine": 0.002,
           "single_launch": 0.066}
    roof1, fwd1 = bench.rooflines(one, sm1, 8, 8, 0.066, PEAKS, "test", FP8)
    per_expert = 3 * 7168 * 2048 // 2 + (4096 * 224 + 7168 * 64)
    fbytes = 8 * per_expert + 2 * 7168 * 2 + 8 * 8
    assert roof1["kernel"] == "single_launch" and fwd1["bytes"] == fbytes
    assert abs(roof1["achieved"] - fbytes / 0.066e-3 / 1e9) < 1e-6


def test_header_states_the_library_thresholds():
    """The C header documents the batch sizes at which the forward changes
    shape; they must be the library's constants."""
    hdr = open(os.path.join(ROOT, "include", "moe_experts.h")).read()
    hdr = re.sub(r"\s*\n\s*\*\s*", " ", hdr)  # join the comment lines
    fused = _const("kFusedCombineSlots", "moe_internal.cuh")
    fused4 = _const("kFusedCombineSlotsFp4Act", "moe_internal.cuh")
    one = _const("kSingleLaunchSlots", "moe_internal.cuh")
    per_expert = _const("kDecodePairsPerExpert", "moe_internal.cuh")
    assert f"T*K <= {fused} and T*K <= {per_expert}E" in hdr or f"T*K <= {per_expert}E and T*K <= {fused}" in hdr
    assert f"T*K <= {fused4} for MOE_W_FP4_ACT_FP4" in hdr
    assert f"T*K <= {one} and T*K <= {per_expert}E" in hdr
