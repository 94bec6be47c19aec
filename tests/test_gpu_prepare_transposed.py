"""GPU: the one-shot transform of transposed expert weights (N contiguous, the
storage the experts dispatch serves with the `_nn` grouped GEMM) writes the
same prepared bytes as the transform of the K-major storage, so the forward
gives the same bits.
"""
import pytest
import torch

from tests import parity as P

pytestmark = pytest.mark.gpu

W = P.W


def _unpack_k(c):
    """[E, N, K/2] bytes, low nibble = even k -> [E, N, K] codes."""
    return torch.stack([c & 0xF, c >> 4], dim=-1).flatten(-2)


def _pack_n(c):
    """[E, K, N] codes -> [E, K, N/2] bytes, low nibble = even n."""
    return (c[..., 0::2] | (c[..., 1::2] << 4)).contiguous()


def transposed(weights):
    """The same weights in the N-major storage."""
    t = dict(weights)
    if weights["fmt"] == "fp8":
        for k in ("w13", "w13_scale", "w2", "w2_scale"):
            t[k] = weights[k].transpose(1, 2).contiguous()
    else:
        t["w13"] = _pack_n(_unpack_k(weights["w13"]).transpose(1, 2))
        t["w2"] = _pack_n(_unpack_k(weights["w2"]).transpose(1, 2))
        t["w13_scale"] = weights["w13_scale"].transpose(1, 2).contiguous()
        t["w2_scale"] = weights["w2_scale"].transpose(1, 2).contiguous()
    return t


CASES = [
    W.Workload("fp8_ragged", 96, 512, 384, 4, 2, "fp8", "softmax", seed=11),
    W.Workload("fp4_ragged", 96, 320, 192, 5, 3, "fp4", "softmax", seed=16, swiglu_limit=0.2),
    W.Workload("fp4_gptoss_like", 64, 2880, 2880, 3, 2, "fp4", "softmax", seed=15, swiglu_limit=7.0),
]


def test_pack_helpers_round_trip():
    c = torch.randint(0, 256, (2, 6, 8), dtype=torch.uint8, device="cuda")
    codes = _unpack_k(c)
    assert codes.shape == (2, 6, 16) and int(codes.max()) <= 15
    assert torch.equal(codes[..., 0], c[..., 0] & 0xF) and torch.equal(codes[..., 1], c[..., 0] >> 4)
    assert torch.equal(_pack_n(codes), c)


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_transposed_storage_prepares_the_same_bytes(wl):
    weights = W.make_weights(wl, "cuda")
    a = P.B.prepare_weights(weights)
    b = P.B.prepare_weights(transposed(weights), transposed=True)
    torch.cuda.synchronize()
    assert torch.equal(a.w13_prep, b.w13_prep)
    assert torch.equal(a.w2_prep, b.w2_prep)
    r = P.run_cuda(wl, weights=weights, prepared=b)
    ref = P.oracle_out(r["hidden"], r["idx"], r["w"], weights, wl.swiglu_limit)
    P.assert_close(r["out"], ref, wl.name)
