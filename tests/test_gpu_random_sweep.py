"""GPU: a seeded sweep of random configurations against the fp64 oracle.

Each configuration draws the weight format, the hidden and intermediate
widths (ragged against the 256-wide GEMM tiles, within the library's
alignment rules: multiples of 128 for FP8, of 64 for FP4), the number of
experts, top-k, tokens (from one token, the single-launch forward, through
FP4 decode batches, to several m-tiles per expert), the routing (softmax or
Zipf with sigmoid weights), skipped slots and the SwiGLU clamp. The draws are
fixed by the seed, so the sweep is the same on every run; every forward must
meet the bf16 output tolerances and leave the device status clear.
"""
import numpy as np
import pytest

from tests import parity as P

pytestmark = pytest.mark.gpu

W = P.W


def _configs(n=16, seed=20240):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        fmt = "fp8" if i % 2 == 0 else "fp4"
        step = 128 if fmt == "fp8" else 64
        lo = 128 // step  # the library takes H, I >= 128
        H = int(rng.integers(lo, 9)) * step
        I = int(rng.integers(lo, 9)) * step
        E = int(rng.choice([4, 8, 16, 33, 64]))
        K = int(min(E, rng.choice([1, 2, 4, 8])))
        T = int(rng.choice([1, 3, 17, 64, 150, 300]))
        router = str(rng.choice(["softmax", "zipf_sigmoid"]))
        skip = float(rng.choice([0.0, 0.1]))
        limit = None if rng.random() < 0.5 else float(np.round(rng.uniform(0.1, 5.0), 3))
        out.append(W.Workload(f"sweep{i}_{fmt}_T{T}_H{H}_I{I}_E{E}_K{K}", T, H, I, E, K, fmt, router,
                              seed=3000 + i, skip_frac=skip, swiglu_limit=limit))
    return out


@pytest.mark.parametrize("wl", _configs(), ids=lambda w: w.name)
def test_random_configuration_matches_oracle(wl):
    r = P.run_cuda(wl)
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], wl.swiglu_limit)
    P.assert_close(r["out"], ref, wl.name)
    assert P.B.device_status(r["ws"]) == 0
