"""The router (logits -> top-k ids and weights) vs the CPU oracle's
topk_route: ids bit-exact (the selection is taken on the same float32 values
on both sides), weights within 1e-6 relative; then its output fed to the layer."""
import numpy as np
import pytest
import torch

from mxfp4_mixture_experts_gb300 import synth
from helpers import gate
from oracle import mxfp4_moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_mixture_experts_gb300 import moe
    return moe


def check(moe, logits, k, scoring, bias=None):
    ids, w = moe.router(logits.cuda(), k, scoring, None if bias is None else bias.cuda())
    torch.cuda.synchronize()
    rid, rw = O.topk_route(logits.numpy(), k, scoring, None if bias is None else bias.numpy())
    got_ids = ids.cpu().numpy()
    assert np.array_equal(got_ids, rid), np.argwhere(got_ids != rid)[:5]
    got_w = w.cpu().numpy().astype(np.float64)
    ok = np.isfinite(rw)
    assert np.all(np.abs(got_w[ok] - rw[ok]) <= 1e-6 * np.abs(rw[ok]) + 1e-12)
    return got_ids, got_w


@pytest.mark.parametrize("T,E,k,scoring,bias_sigma", [
    (1, 128, 4, "softmax_topk", 0.0),        # the gpt-oss shapes
    (32, 128, 4, "softmax_topk", 0.0),
    (32, 256, 8, "sigmoid_renorm", 0.0),     # the GLM shapes
    (32, 256, 8, "sigmoid_renorm", 0.5),     # the wide-K shape (skewing bias)
    (8192, 256, 8, "sigmoid_renorm", 0.0),   # a prefill chunk
    (300, 100, 7, "softmax_topk", 0.3),      # E not a multiple of 32
    (17, 9, 9, "sigmoid_renorm", 0.0),       # k = E
    (40, 1024, 32, "softmax_topk", 0.0),     # the largest E and k
])
def test_router_matches_oracle(moe, T, E, k, scoring, bias_sigma):
    g = torch.Generator().manual_seed(T * 131 + E + k)
    logits = torch.randn(T, E, generator=g)
    bias = bias_sigma * torch.randn(E, generator=g) if bias_sigma > 0 else None
    check(moe, logits, k, scoring, bias)


def test_router_ties_to_the_lower_index(moe):
    """Logits on a coarse grid (many exact ties) and rows of equal logits."""
    g = torch.Generator().manual_seed(5)
    logits = torch.round(torch.randn(64, 256, generator=g) * 2) / 2
    logits[0] = 0.25
    logits[1, ::3] = 3.0
    for scoring in ("softmax_topk", "sigmoid_renorm"):
        ids, _ = check(moe, logits, 8, scoring)
        assert list(ids[0]) == list(range(8))
        assert list(ids[1]) == [0, 3, 6, 9, 12, 15, 18, 21]


def test_router_float32_sum_decides(moe):
    """1 + 2^-25 rounds to 1 in float32: expert 1 ties expert 0 and loses."""
    logits = torch.tensor([[1.0, 1.0, 0.0, -1.0]], dtype=torch.float32)
    bias = torch.tensor([0.0, 2.0 ** -25, 0.0, 0.0], dtype=torch.float32)
    ids, _ = check(moe, logits, 2, "sigmoid_renorm", bias)
    assert list(ids[0]) == [0, 1]
    bias[1] = 2.0 ** -23
    ids, _ = check(moe, logits, 2, "sigmoid_renorm", bias)
    assert list(ids[0]) == [1, 0]


def test_router_nan_ranks_last(moe):
    logits = torch.randn(4, 64, generator=torch.Generator().manual_seed(6))
    logits[:, 5] = float("nan")
    logits[2, :] = float("nan")
    logits[2, 40] = 1.0
    ids, _ = check(moe, logits, 4, "softmax_topk")
    assert not (ids[[0, 1, 3]] == 5).any()
    assert ids[2, 0] == 40


def test_router_feeds_the_layer(moe):
    """Router output -> mxfp4_moe_forward equals the oracle layer on the
    oracle router's ids and weights (the gate)."""
    shape = synth.custom_shape(K=320, I=128, E=16, topk=4)
    case = synth.make_case(shape, 12, seed=40)
    g = torch.Generator().manual_seed(41)
    logits = torch.randn(12, 16, generator=g)
    ids, w = moe.router(logits.cuda(), 4, "softmax_topk")
    y = moe.forward(case.hidden.cuda(), ids, w, case.w13.cuda(), case.s13.cuda(),
                    case.w2.cuda(), case.s2.cuda())
    torch.cuda.synchronize()
    rid, rw = O.topk_route(logits.numpy(), 4, "softmax_topk")
    case.topk_ids = torch.from_numpy(rid)
    case.topk_weights = torch.from_numpy(rw.astype(np.float32))
    gate(y, case)
