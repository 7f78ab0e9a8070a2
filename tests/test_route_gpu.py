"""Routing / permute kernel vs the oracle: bit-exact counts, offsets, lists
and invalid-id count."""
import numpy as np
import pytest
import torch

from oracle import mxfp4_moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_mixture_experts_gb300 import moe
    return moe


def check(moe, ids_np, E, many_ctas=False):
    ids = torch.as_tensor(ids_np, dtype=torch.int32, device="cuda")
    cnt, off, lst, status = moe.route(ids, E, many_ctas=many_ctas)
    torch.cuda.synchronize()
    rt = O.route(ids_np, E)
    assert np.array_equal(cnt.cpu().numpy(), rt["count"])
    assert np.array_equal(off.cpu().numpy(), rt["offset"])
    n = int(rt["offset"][-1])
    got = lst.cpu().numpy()
    assert np.array_equal(got[:n], rt["list"])
    assert np.all(got[n:] == -1)
    assert int(status[0]) == rt["invalid"]
    assert int(status[1]) == len(rt["touched"])


@pytest.mark.parametrize("T,k,E", [(1, 4, 128), (7, 3, 8), (32, 8, 256), (33, 4, 32),
                                   (1000, 8, 256), (8192, 8, 256), (5, 2, 1024)])
def test_route_random(moe, T, k, E):
    rng = np.random.default_rng(T * 1000 + k)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    check(moe, ids, E)


def test_route_padding_and_invalid(moe):
    rng = np.random.default_rng(1)
    ids = rng.integers(-1, 12, size=(97, 5)).astype(np.int32)   # -1 padding, >= 10 invalid
    check(moe, ids, 10)


def test_route_all_to_one_expert(moe):
    check(moe, np.full((300, 4), 5, dtype=np.int32), 16)


def test_route_nothing_routed(moe):
    check(moe, np.full((6, 2), -1, dtype=np.int32), 8)


def test_route_skewed_prefill(moe):
    rng = np.random.default_rng(2)
    p = rng.dirichlet(np.full(256, 0.3))
    ids = rng.choice(256, size=(8192, 8), p=p).astype(np.int32)
    check(moe, ids, 256)


# the prefill path's sort over many CTAs (mxfp4_moe_route_ws): from 8192
# routes on, chunks of routes per CTA; below, the one-CTA sort
@pytest.mark.parametrize("T,k,E", [(1000, 8, 256), (1024, 8, 256), (8192, 8, 256), (8191, 3, 1024),
                                   (16384, 4, 128), (65536, 8, 32), (3000, 3, 7)])
def test_route_many_ctas_random(moe, T, k, E):
    rng = np.random.default_rng(T * 7 + k)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int32)
    check(moe, ids, E, many_ctas=True)


def test_route_many_ctas_padding_invalid_skew(moe):
    rng = np.random.default_rng(5)
    p = rng.dirichlet(np.full(256, 0.2))
    ids = rng.choice(256, size=(8192, 8), p=p).astype(np.int32)
    ids[rng.random(ids.shape) < 0.05] = -1      # padding
    ids[rng.random(ids.shape) < 0.02] = 300     # invalid
    check(moe, ids, 256, many_ctas=True)


def test_route_many_ctas_all_to_one_expert(moe):
    check(moe, np.full((4096, 4), 3, dtype=np.int32), 16, many_ctas=True)
    check(moe, np.full((4096, 4), -1, dtype=np.int32), 16, many_ctas=True)
