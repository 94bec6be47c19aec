"""GPU: every workload at full size, in the launch configuration bench.py times.

The oracle computes sampled tokens one by one (first, last and seeded random
tokens); properties that hold at any size are checked on the whole output:
routing bit-exact against the oracle's stable sort, every output finite, no
device flag raised, and the all-skipped rows exactly zero.
"""
import numpy as np
import pytest
import torch

from oracle.routing import route
from tests import parity as P

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

W = P.W
SAMPLE = {"mixtral_prefill_fp8": 4, "dsv3_decode_fp8": 6, "dsv3_prefill_fp8": 3, "gptoss_fp8xfp4": 12,
          "dsv3_decode_fp4_T1": 1, "dsv3_decode_fp4_T8": 4, "dsv3_decode_fp4_T32": 4, "dsv3_decode_fp4_T128": 4,
          "dsv3_decode_fp4_T512": 3, "dsv3_decode_fp4_T2048": 3}


@pytest.mark.parametrize("name", list(SAMPLE), ids=str)
def test_full_size_workload(name):
    wl = W.WORKLOADS[name]
    r = P.run_cuda(wl)
    out = r["out"]
    assert torch.isfinite(out.float()).all()
    assert P.B.device_status(r["ws"]) == 0

    # routing of the whole batch against the oracle
    L = P.B.workspace_layout(wl.fmt, wl.T, wl.H, wl.I, wl.E, wl.K)
    ref_route = route(r["idx"].cpu().numpy(), wl.E, L.row_align)
    inv = P.ws_region(r["ws"], L, "inv", torch.int32, wl.S).cpu().numpy()
    assert (inv == ref_route["inv"]).all()

    # all-skipped tokens are exact +0
    skipped = (r["idx"] < 0).all(dim=1)
    if skipped.any():
        assert (out[skipped].view(torch.int16) == 0).all()

    # sampled tokens against the fp64 oracle
    rng = np.random.default_rng(wl.seed)
    n = SAMPLE[name]
    toks = sorted({0, wl.T - 1, *rng.choice(wl.T, size=min(n, wl.T), replace=False).tolist()})[:max(n, 1)]
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], wl.swiglu_limit, tokens=toks)
    m = P.assert_close(out[toks], ref, name)
    print(name, toks, m)
