"""GPU: the experts forward through the C ABI against the fp64 oracle.

Sizes the oracle finishes in seconds that still span several m and n tiles
with ragged tails, in both weight formats, plus the degenerate cases.
"""
import numpy as np
import pytest
import torch

from tests import parity as P

pytestmark = pytest.mark.gpu

W = P.W

CASES = [
    W.WORKLOADS["tiny_fp8"],
    W.Workload("fp8_ragged", 300, 512, 384, 4, 2, "fp8", "softmax", seed=11),
    W.Workload("fp8_ragged_clamp", 300, 512, 384, 4, 2, "fp8", "softmax", seed=12, swiglu_limit=0.3),
    W.Workload("fp8_zipf_skips", 200, 256, 256, 32, 8, "fp8", "zipf_sigmoid", seed=13, skip_frac=0.05),
    W.Workload("fp4_small", 64, 256, 128, 8, 2, "fp4", "softmax", seed=14),
    W.Workload("fp4_gptoss_like", 300, 2880, 2880, 8, 4, "fp4", "softmax", seed=15, logit_std=1.5,
               swiglu_limit=7.0),
    W.Workload("fp4_ragged_h", 130, 320, 192, 5, 3, "fp4", "softmax", seed=16, swiglu_limit=0.2),
    # FP4 with few pairs per expert (mostly one partly filled m-tile each)
    W.Workload("fp4_small_ragged", 40, 320, 192, 8, 3, "fp4", "softmax", seed=17, swiglu_limit=0.25),
    W.Workload("fp4_small_zipf", 64, 512, 256, 32, 8, "fp4", "zipf_sigmoid", seed=18, skip_frac=0.05),
    W.Workload("fp4_small_T1", 1, 512, 384, 16, 4, "fp4", "softmax", seed=19),
    # FP4 with at most 8 pairs per expert on average: the decode mode of the
    # grouped GEMMs (32-row token chunks). Zipf routing gives some experts
    # 2-4 chunks, i.e. chunks in every 32-row quarter of a 128-row block.
    W.Workload("fp4_decode_chunks", 40, 320, 192, 64, 8, "fp4", "zipf_sigmoid", seed=24, swiglu_limit=0.25),
    W.Workload("fp4_decode_dsv3_like", 48, 1024, 512, 64, 8, "fp4", "zipf_sigmoid", seed=25, skip_frac=0.05),
]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_forward_matches_oracle(wl):
    r = P.run_cuda(wl)
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], wl.swiglu_limit)
    m = P.assert_close(r["out"], ref, wl.name)
    assert P.B.device_status(r["ws"]) == 0
    print(wl.name, m)


def test_deterministic_and_batch_invariant():
    wl = CASES[1]
    r = P.run_cuda(wl)
    again = P.B.experts_forward(r["hidden"], r["idx"], r["w"], r["prepared"], wl.swiglu_limit)
    assert torch.equal(again.view(torch.int16), r["out"].view(torch.int16))
    # Appending all-skipped tokens (the padded last slice of the shared-batch
    # example) changes no bit of the real tokens and gives +0 rows.
    pad = 37
    hid = torch.cat([r["hidden"], r["hidden"][:pad]])
    idx = torch.cat([r["idx"], torch.full((pad, wl.K), -1, dtype=torch.int32, device="cuda")])
    w = torch.cat([r["w"], r["w"][:pad]])
    out = P.B.experts_forward(hid, idx, w, r["prepared"], wl.swiglu_limit)
    assert torch.equal(out[:wl.T].view(torch.int16), r["out"].view(torch.int16))
    assert (out[wl.T:].view(torch.int16) == 0).all()


def test_small_batch_matches_the_same_tokens_in_a_larger_batch():
    """240 slots and the same tokens inside a batch of 280: the same bits
    (the routing's padded layout moves, the rows' results do not). For FP4
    decode batches, where the small batch also combines in GEMM2's epilogue,
    see test_fp4_fused_combine_matches_the_combine_kernel."""
    wl = W.Workload("fused_vs_split", 120, 256, 256, 8, 2, "fp8", "zipf_sigmoid", seed=41, skip_frac=0.1)
    r = P.run_cuda(wl)
    extra = 20
    hid = torch.cat([r["hidden"], r["hidden"][:extra]])
    idx = torch.cat([r["idx"], r["idx"][:extra]])
    w = torch.cat([r["w"], r["w"][:extra]])
    out = P.B.experts_forward(hid, idx, w, r["prepared"])
    assert torch.equal(out[:wl.T].view(torch.int16), r["out"].view(torch.int16))
    P.assert_close(r["out"], P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], None), "fused")


def test_all_skipped_gives_positive_zero():
    wl = W.scaled(CASES[1], T=50)
    idx = torch.full((wl.T, wl.K), -1, dtype=torch.int32, device="cuda")
    w = torch.rand(wl.T, wl.K, device="cuda")
    r = P.run_cuda(wl, idx=idx, w=w)
    assert (r["out"].view(torch.int16) == 0).all()


def test_nan_weight_in_skipped_slot_is_never_read():
    wl = CASES[1]
    r = P.run_cuda(wl)
    idx = r["idx"].clone()
    w = r["w"].clone()
    idx[5, 0] = -1
    idx[17, 1] = -1
    a = P.B.experts_forward(r["hidden"], idx, w, r["prepared"])
    w[5, 0] = float("nan")
    w[17, 1] = float("inf")
    b = P.B.experts_forward(r["hidden"], idx, w, r["prepared"])
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    ref = P.oracle_out(r["hidden"], idx, w, r["weights"], None)
    P.assert_close(b, ref, "nan weights")


@pytest.mark.parametrize("T", [1, 2, 127, 129])
def test_small_token_counts(T):
    wl = W.Workload("fp8_small_T", T, 256, 256, 6, 2, "fp8", "softmax", seed=20 + T)
    r = P.run_cuda(wl)
    P.assert_close(r["out"], P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], None), f"T={T}")


def test_single_expert_top1():
    wl = W.Workload("e1k1", 200, 256, 128, 1, 1, "fp8", "softmax", seed=31)
    r = P.run_cuda(wl)
    P.assert_close(r["out"], P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], None), "E=1,K=1")


def test_zero_tokens_enqueues_nothing():
    wl = CASES[0]
    weights = W.make_weights(wl, "cuda")
    prepared = P.B.prepare_weights(weights)
    hid = torch.empty(0, wl.H, dtype=torch.bfloat16, device="cuda")
    idx = torch.empty(0, wl.K, dtype=torch.int32, device="cuda")
    w = torch.empty(0, wl.K, dtype=torch.float32, device="cuda")
    out = P.B.experts_forward(hid, idx, w, prepared)
    assert out.shape == (0, wl.H)


def test_refusals():
    wl = CASES[0]
    r = P.run_cuda(wl)
    with pytest.raises(ValueError):
        P.B.experts_forward(r["hidden"].float(), r["idx"], r["w"], r["prepared"])
    with pytest.raises(NotImplementedError):
        P.B.experts_forward(r["hidden"], r["idx"], r["w"], r["prepared"], activation_scheme="static")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(P.B.MoeError):
        P.B.experts_forward(r["hidden"], r["idx"], r["w"], r["prepared"], workspace=small)
    host = r["hidden"].cpu()
    L = P.B.lib()
    st = L.moe_experts_forward(host.data_ptr(), r["idx"].data_ptr(), r["w"].data_ptr(), wl.T, wl.H, wl.I, wl.E,
                               wl.K, 0, r["prepared"].w13_prep.data_ptr(), r["prepared"].w2_prep.data_ptr(),
                               float("nan"), r["ws"].data_ptr(), r["ws"].numel(), r["out"].data_ptr(), None)
    assert st == 4  # MOE_ERR_DEVICE_MISMATCH: a host pointer


def test_fp4_token_outputs_do_not_depend_on_the_batch():
    """8 tokens alone and inside a 68-token batch (other experts' m-tiles, more
    rows in the same tiles): the same bits, and both match the oracle."""
    wl = W.Workload("fp4_batch", 8, 512, 256, 8, 4, "fp4", "softmax", seed=23)
    r = P.run_cuda(wl)
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], None)
    P.assert_close(r["out"], ref, "8 tokens")
    extra = 60
    g = torch.Generator(device="cuda").manual_seed(5)
    hid = torch.cat([r["hidden"], (torch.randn(extra, wl.H, generator=g, device="cuda")).to(torch.bfloat16)])
    idx = torch.cat([r["idx"], torch.randint(0, wl.E, (extra, wl.K), generator=g, device="cuda", dtype=torch.int32)])
    w = torch.cat([r["w"], torch.rand(extra, wl.K, generator=g, device="cuda")])
    out = P.B.experts_forward(hid, idx, w, r["prepared"])
    assert torch.equal(out[:wl.T].view(torch.int16), r["out"].view(torch.int16))


def test_fp4_decode_mode_expert_with_four_chunks():
    """One expert takes 100 tokens in a batch with at most 8 pairs per expert
    on average: its rows span four 32-row chunks, one in each quarter of its
    128-row block (each chunk's scale words sit in a different column)."""
    wl = W.Workload("fp4_four_chunks", 100, 512, 256, 64, 2, "fp4", "softmax", seed=26, swiglu_limit=3.0)
    idx, w = W.make_routing(wl, "cuda")
    idx[:, 0] = 5
    idx[:, 1] = torch.where(idx[:, 1] == 5, torch.full_like(idx[:, 1], 6), idx[:, 1])
    r = P.run_cuda(wl, idx=idx, w=w)
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], wl.swiglu_limit)
    P.assert_close(r["out"], ref, "four chunks")


def test_fp4_fused_combine_matches_the_combine_kernel():
    """FP4 decode batches of at most 256 slots sum each token's rows in GEMM2's
    epilogue; the same tokens in a larger decode batch go through the separate
    combine kernel. Same bits either way, +0 rows for tokens whose slots are
    all skipped, and H = 320 ends halfway through a 128-column half."""
    wl = W.Workload("fp4_fused_combine", 30, 320, 192, 64, 4, "fp4", "zipf_sigmoid", seed=28, skip_frac=0.3)
    idx, w = W.make_routing(wl, "cuda")
    idx[3] = -1
    idx[17] = -1
    r = P.run_cuda(wl, idx=idx, w=w)
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], None)
    P.assert_close(r["out"], ref, "fused combine")
    assert (r["out"][3].view(torch.int16) == 0).all() and (r["out"][17].view(torch.int16) == 0).all()
    extra = 40  # 70 tokens x 4 = 280 slots: still decode mode, separate combine
    g = torch.Generator(device="cuda").manual_seed(6)
    hid = torch.cat([r["hidden"], torch.randn(extra, wl.H, generator=g, device="cuda").to(torch.bfloat16)])
    idx2 = torch.cat([idx, torch.randint(0, wl.E, (extra, wl.K), generator=g, device="cuda", dtype=torch.int32)])
    w2 = torch.cat([w, torch.rand(extra, wl.K, generator=g, device="cuda")])
    out = P.B.experts_forward(hid, idx2, w2, r["prepared"])
    assert torch.equal(out[:wl.T].view(torch.int16), r["out"].view(torch.int16))


@pytest.mark.parametrize("T,K,E", [(1, 8, 64), (3, 8, 40), (8, 4, 16)])
def test_fp4_small_decode_batches_match_larger_batches(T, K, E):
    """FP4 decode batches of at most 32 slots (GEMM2 starts its first weight
    copies before waiting for GEMM1): duplicate ids, skipped slots and an
    all-skipped token give the same bits as the same tokens inside a larger
    batch, and match the oracle."""
    wl = W.Workload(f"fp4_first_units_T{T}", T, 512, 256, E, K, "fp4", "zipf_sigmoid", seed=30 + T)
    idx, w = W.make_routing(wl, "cuda")
    idx[0, 1] = idx[0, 0]  # duplicate id in one token
    idx[0, 2] = -1
    if T > 2:
        idx[1] = -1  # all slots skipped
        idx[2, 0] = E - 1
    r = P.run_cuda(wl, idx=idx, w=w)
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], r["weights"], None)
    P.assert_close(r["out"], ref, wl.name)
    assert P.B.device_status(r["ws"]) == 0
    extra = 40 // K + 1  # pushes the batch past 32 slots
    g = torch.Generator(device="cuda").manual_seed(7)
    hid = torch.cat([r["hidden"], torch.randn(extra, wl.H, generator=g, device="cuda").to(torch.bfloat16)])
    idx2 = torch.cat([idx, torch.randint(0, E, (extra, K), generator=g, device="cuda", dtype=torch.int32)])
    w2 = torch.cat([w, torch.rand(extra, K, generator=g, device="cuda")])
    out = P.B.experts_forward(hid, idx2, w2, r["prepared"])
    assert torch.equal(out[:T].view(torch.int16), r["out"].view(torch.int16))


@pytest.mark.parametrize("T,H,I,E,K,skip", [(1, 7168, 2048, 256, 8, 0.0), (4, 1024, 512, 64, 8, 0.05),
                                            (2, 512, 384, 256, 8, 0.0), (8, 320, 192, 32, 4, 0.3),
                                            (16, 256, 128, 64, 2, 0.0), (32, 256, 128, 8, 1, 0.0)])
def test_single_launch_forward_matches_the_kernel_sequence(T, H, I, E, K, skip):
    """Small FP4 decode batches (at most 8 pairs per expert, at most 32
    slots) run the whole forward as one cooperative launch: routing and
    quantization, then one work list of GEMM1 and GEMM2 units in which every
    GEMM2 unit waits on device counters for its chunk's GEMM1 units, the
    combine in GEMM2's epilogue. The same inputs through the multi-kernel
    sequence (the debug entry point runs it) give the same bits, twice in a
    row, and both match the oracle."""
    wl = W.Workload(f"single_T{T}", T, H, I, E, K, "fp4", "zipf_sigmoid", seed=60 + T, skip_frac=skip,
                    swiglu_limit=7.0 if T == 8 else None)
    assert wl.S <= 32 and wl.S <= 8 * wl.E
    r = P.run_cuda(wl)
    assert P.B.device_status(r["ws"]) == 0
    for _ in range(2):
        out = P.B.experts_forward(r["hidden"], r["idx"], r["w"], r["prepared"], wl.swiglu_limit, workspace=r["ws"])
        seq, _, ws2 = P.B.debug_forward_act_f32(r["hidden"], r["idx"], r["w"], r["prepared"], wl.swiglu_limit)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), r["out"].view(torch.int16))
        assert torch.equal(seq.view(torch.int16), r["out"].view(torch.int16))
        assert P.B.device_status(r["ws"]) == 0 and P.B.device_status(ws2) == 0
    toks = list(range(min(T, 24)))
    ref = P.oracle_out_parallel(r["hidden"], r["idx"], r["w"], r["weights"], wl.swiglu_limit, toks)
    P.assert_close(r["out"][toks], ref, wl.name)
