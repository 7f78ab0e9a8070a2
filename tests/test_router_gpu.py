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


def check_grouped(moe, logits, k, scoring, bias, n_group, topk_group, bias_in_weights):
    ids, w = moe.router_grouped(logits.cuda(), k, scoring, None if bias is None else bias.cuda(),
                                n_group, topk_group, bias_in_weights)
    torch.cuda.synchronize()
    rid, rw = O.topk_route(logits.numpy(), k, scoring, None if bias is None else bias.numpy(),
                           n_group, topk_group, bias_in_weights)
    got_ids = ids.cpu().numpy()
    assert np.array_equal(got_ids, rid), np.argwhere(got_ids != rid)[:5]
    got_w = w.cpu().numpy().astype(np.float64)
    ok = np.isfinite(rw)
    assert np.all(np.abs(got_w[ok] - rw[ok]) <= 1e-6 * np.abs(rw[ok]) + 1e-12)
    return got_ids, got_w


@pytest.mark.parametrize("T,E,k,scoring,n_group,topk_group,bias_sigma,in_w", [
    (32, 256, 8, "sigmoid_renorm", 8, 4, 0.5, False),      # 8 groups of 32, bias steers only
    (8192, 256, 8, "sigmoid_renorm", 8, 4, 0.5, False),    # a prefill chunk
    (64, 128, 4, "softmax_topk", 4, 2, 0.0, True),
    (100, 160, 6, "softmax_topk", 32, 3, 0.3, True),       # groups of 5
    (40, 1024, 32, "sigmoid_renorm", 32, 8, 0.2, False),   # the largest E, k and n_group
    (17, 96, 12, "sigmoid_renorm", 3, 1, 0.0, True),       # one group kept
    (5, 8, 8, "softmax_topk", 2, 2, 0.0, True),            # k = E
    (33, 256, 8, "softmax_topk", 1, 1, 0.7, False),        # no groups, bias steers only
])
def test_grouped_router_matches_oracle(moe, T, E, k, scoring, n_group, topk_group, bias_sigma,
                                       in_w):
    g = torch.Generator().manual_seed(T * 17 + E + n_group)
    logits = torch.randn(T, E, generator=g)
    bias = bias_sigma * torch.randn(E, generator=g) if bias_sigma > 0 else None
    check_grouped(moe, logits, k, scoring, bias, n_group, topk_group, in_w)


def test_grouped_router_ties_and_nan(moe):
    """Coarse logits (tied experts and tied group scores), a group of NaN
    logits (its score is -inf) and a row of equal logits (the lowest groups
    and ids win)."""
    g = torch.Generator().manual_seed(9)
    logits = torch.round(torch.randn(48, 64, generator=g) * 2) / 2
    logits[0] = 0.5
    logits[1, 8:16] = float("nan")
    logits[2, :] = float("nan")
    logits[2, 50] = 0.0
    for scoring in ("softmax_topk", "sigmoid_renorm"):
        for in_w in (True, False):
            ids, _ = check_grouped(moe, logits, 6, scoring, None, 8, 3, in_w)
            assert list(ids[0]) == [0, 1, 2, 3, 4, 5]
            assert not ((ids[1] >= 8) & (ids[1] < 16)).any()
            assert ids[2, 0] == 50


def test_plain_router_is_grouped_router_with_one_group(moe):
    g = torch.Generator().manual_seed(10)
    logits = torch.randn(200, 256, generator=g).cuda()
    bias = (0.5 * torch.randn(256, generator=g)).cuda()
    a = moe.router(logits, 8, "sigmoid_renorm", bias)
    b = moe.router_grouped(logits, 8, "sigmoid_renorm", bias, 1, 1, True)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))
