"""GPU: every workload at full size, in the launch configuration bench.py times.

The oracle computes a sample of at least 64 tokens per workload: the first and
last token, one token for every expert the batch touches (so every touched
expert's weights pass through the comparison), then seeded random tokens.
Properties that hold at any size are checked on the whole output:
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
NAMES = ["mixtral_prefill_fp8", "dsv3_decode_fp8", "dsv3_prefill_fp8", "gptoss_fp8xfp4", "dsv3_decode_fp4_T1",
         "dsv3_decode_fp4_T8", "dsv3_decode_fp4_T32", "dsv3_decode_fp4_T128", "dsv3_decode_fp4_T512",
         "dsv3_decode_fp4_T2048", "gptoss_fp4xfp4", "dsv3_decode_fp4xfp4_T1", "dsv3_decode_fp4xfp4_T128"]
MIN_SAMPLE = 64


@pytest.mark.parametrize("name", NAMES, ids=str)
def test_full_size_workload(name):
    wl = W.WORKLOADS[name]
    r = P.run_cuda(wl)
    out = r["out"]
    assert torch.isfinite(out.float()).all()
    assert P.B.device_status(r["ws"]) == 0

    # routing of the whole batch against the oracle
    L = P.B.workspace_layout(P.lib_fmt(wl), wl.T, wl.H, wl.I, wl.E, wl.K)
    ref_route = route(r["idx"].cpu().numpy(), wl.E, L.row_align)
    inv = P.ws_region(r["ws"], L, "inv", torch.int32, wl.S).cpu().numpy()
    assert (inv == ref_route["inv"]).all()

    # all-skipped tokens are exact +0
    skipped = (r["idx"] < 0).all(dim=1)
    if skipped.any():
        assert (out[skipped].view(torch.int16) == 0).all()

    # sampled tokens against the fp64 oracle
    toks = P.sample_tokens(r["idx"], wl.E, MIN_SAMPLE, wl.seed)
    sel = r["idx"].cpu().numpy()[toks]
    touched = set(np.unique(r["idx"].cpu().numpy()).tolist()) - {-1}
    assert set(np.unique(sel).tolist()) - {-1} == touched
    assert len(toks) >= min(MIN_SAMPLE, wl.T)
    ref = P.oracle_out_parallel(r["hidden"], r["idx"], r["w"], r["weights"], wl.swiglu_limit, toks,
                                act_fmt=wl.act_fmt)
    m = P.assert_close(out[toks], ref, name)
    print(name, len(toks), "tokens,", len(touched), "experts", m)
