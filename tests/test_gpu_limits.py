"""GPU: the largest shapes the library accepts, on few tokens: E = 512 experts,
K = 32 slots per token, H = 32768 or I = 32768 (the longest K loops and the
widest N grids of both GEMMs). Routing and quantization bit-exact, outputs
within the tolerances, against the oracle.
"""
import pytest

from tests import parity as P
from tests.test_gpu_route_quant import _check_route_quant

pytestmark = pytest.mark.gpu

W = P.W

CASES = [
    # 512 experts, 32 slots per token: 2048 slots on the single-CTA routing path
    W.Workload("e512_k32", 64, 256, 128, 512, 32, "fp8", "softmax", seed=61),
    # 32 slots per token over 9600 slots: the multi-CTA routing path, FP4
    W.Workload("k32_multicta_fp4", 300, 256, 128, 40, 32, "fp4", "zipf_sigmoid", seed=62, skip_frac=0.05),
    # 32 slots per token in an FP4 decode batch of 256 slots: the combine fused
    # into GEMM2 sums 32 rows per token
    W.Workload("k32_fused_combine_fp4", 8, 256, 128, 40, 32, "fp4", "softmax", seed=65),
    # H = 32768: GEMM1 runs 256 K blocks, GEMM2 128 N tiles
    W.Workload("h32768_fp8", 40, 32768, 128, 2, 1, "fp8", "softmax", seed=63),
    # I = 32768: GEMM1 runs 256 N tiles, GEMM2 256 K blocks
    W.Workload("i32768_fp4", 24, 128, 32768, 2, 2, "fp4", "softmax", seed=64, swiglu_limit=7.0),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_largest_shapes(wl):
    r = P.run_cuda(wl)
    _check_route_quant(wl, r)
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], wl.swiglu_limit)
    P.assert_close(r["out"], ref, wl.name)
    assert P.B.device_status(r["ws"]) == 0


def test_shapes_beyond_the_limits_are_refused():
    for fmt, E, H, I in [("fp8", 513, 256, 128), ("fp8", 8, 32896, 128), ("fp4", 8, 128, 32832)]:
        assert P.B.lib().moe_workspace_bytes(P.B.FMT[fmt], 4, H, I, E, 2) == 0
    assert P.B.lib().moe_workspace_bytes(P.B.FMT["fp8"], 4, 256, 128, 8, 33) == 0
