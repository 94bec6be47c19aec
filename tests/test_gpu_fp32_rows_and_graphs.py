"""GPU: the weighted fp32 per-pair rows and the final rounding; the forward
inside a CUDA graph.

The method keeps the per-pair outputs in fp32 and rounds once to bf16 after
the top-k sum. The rows are read back from the workspace and summed here in
fp32 in the same ascending-k order as the combine kernel: that fp32 output
must meet the elementwise bound 1e-2 * RMS literally (no half-ulp allowance,
which only exists because of the final bf16 rounding), and its bf16
round-to-nearest-even must be the library's output bit for bit.
"""
import numpy as np
import pytest
import torch

from tests import parity as P

pytestmark = pytest.mark.gpu

W = P.W

CASES = [
    W.Workload("fp8_ragged", 300, 512, 384, 4, 2, "fp8", "softmax", seed=11),
    W.Workload("fp8_zipf_skips", 200, 256, 256, 32, 8, "fp8", "zipf_sigmoid", seed=13, skip_frac=0.05),
    W.Workload("fp4_gptoss_like", 300, 2880, 2880, 8, 4, "fp4", "softmax", seed=15, logit_std=1.5,
               swiglu_limit=7.0),
]


def fp32_topk_sum(r, wl):
    L = P.B.workspace_layout(wl.fmt, wl.T, wl.H, wl.I, wl.E, wl.K)
    S = wl.T * wl.K
    inv = P.ws_region(r["ws"], L, "inv", torch.int32, S).view(wl.T, wl.K).cpu().numpy()
    y = P.ws_region(r["ws"], L, "y", torch.float32, L.row_capacity * wl.H).view(L.row_capacity, wl.H)
    y = y.cpu().numpy()
    out = np.zeros((wl.T, wl.H), dtype=np.float32)
    for k in range(wl.K):  # ascending k, fp32 adds, skipped slots never read
        rows = inv[:, k]
        v = rows >= 0
        out[v] = out[v] + y[rows[v]]
    return out


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_fp32_rows_meet_the_literal_bound_and_round_to_the_output(wl):
    r = P.run_cuda(wl)
    out32 = fp32_topk_sum(r, wl)
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], wl.swiglu_limit)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = np.abs(out32.astype(np.float64) - ref)
    assert float(err.max()) <= P.MAX_REL_RMS * rms, (float(err.max()) / rms)
    assert float(np.linalg.norm(out32 - ref) / np.linalg.norm(ref)) <= P.REL_FRO
    rounded = torch.from_numpy(out32).to(torch.bfloat16)
    assert torch.equal(rounded.view(torch.int16), r["out"].cpu().view(torch.int16))


@pytest.mark.parametrize("wl", [CASES[0], W.scaled(W.WORKLOADS["dsv3_decode_fp4_T8"], H=512, I=256)],
                         ids=lambda w: w.name)
def test_forward_replays_from_a_cuda_graph(wl):
    """All launches are stream-ordered and allocation-free: one forward is
    captured into a CUDA graph; replays on new inputs copied into the captured
    buffers give the eager forward's bits."""
    r = P.run_cuda(wl)
    hidden, idx, w = r["hidden"].clone(), r["idx"].clone(), r["w"].clone()
    ws = torch.empty_like(r["ws"])
    out = torch.empty_like(r["out"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        P.B.experts_forward(hidden, idx, w, r["prepared"], wl.swiglu_limit, workspace=ws, out=out)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        P.B.experts_forward(hidden, idx, w, r["prepared"], wl.swiglu_limit, workspace=ws, out=out)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), r["out"].view(torch.int16))
    # new inputs in the same buffers
    hidden2 = W.make_hidden(W.scaled(wl, seed=wl.seed + 7), "cuda")
    idx2, w2 = W.make_routing(W.scaled(wl, seed=wl.seed + 7), "cuda")
    hidden.copy_(hidden2)
    idx.copy_(idx2)
    w.copy_(w2)
    g.replay()
    eager = P.B.experts_forward(hidden2, idx2, w2, r["prepared"], wl.swiglu_limit)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert P.B.device_status(ws) == 0
