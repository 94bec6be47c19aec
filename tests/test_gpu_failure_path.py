"""GPU: the failure path of the pipeline waits, without a GPU fault.

The library's self-test launches one CTA whose thread waits, through the
bounded mbarrier wait the GEMM pipeline uses, on a phase that nothing
completes. The wait must give up after its bound (about one second of SM
clock), the kernel must report MOE_DEV_TIMEOUT in the workspace status word
and return, and the context must stay usable: a forward afterwards matches
the oracle and raises no flag.
"""
import time

import pytest
import torch

from tests import parity as P

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports_timeout():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    flags = P.B.selftest_wait_timeout(ws)
    dt = time.perf_counter() - t0
    assert flags == P.B.MOE_DEV_TIMEOUT
    assert 0.1 < dt < 30.0, dt
    assert P.B.device_status(ws) == 0  # reading the status clears it

    wl = P.W.WORKLOADS["tiny_fp8"]
    r = P.run_cuda(wl)
    P.assert_close(r["out"], P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], wl.swiglu_limit),
                   "forward after a timed-out wait")
    assert P.B.device_status(r["ws"]) == 0


def test_selftest_refuses_host_memory():
    host = torch.zeros(256, dtype=torch.uint8).pin_memory()
    assert P.B.lib().moe_selftest_wait_timeout(host.data_ptr(), 256, None) == 4  # MOE_ERR_DEVICE_MISMATCH
