"""Pins of the oracle's expert-window and per-route forms (``forward_window``)
to identities with the pinned layer (no GPU needed): the windows of any
partition of the experts sum to the whole layer; per-route outputs weighted
and summed over the slots give the layer; a window holding all experts is
the layer; routes outside the window contribute nothing. Planted mistakes
must make a check fail."""
import types

import numpy as np

from oracle import mxfp4_moe_oracle as O
from test_oracle_pins import small_case


def case(seed, T=5, K=64, I=32, E=6, k=3):
    rng = np.random.default_rng(seed)
    return small_case(rng, T, K, I, E, k)


def check_window_partition(O, seed=71):
    hb, ids, w, w13, s13, w2, s2 = case(seed)
    full = O.forward(hb, ids, w, w13, s13, w2, s2)
    bad = []
    for cut in (1, 2, 4):
        lo = O.forward_window(hb, ids, w, w13[:cut], s13[:cut], w2[:cut], s2[:cut], 0)
        hi = O.forward_window(hb, ids, w, w13[cut:], s13[cut:], w2[cut:], s2[cut:], cut)
        if not np.allclose(lo + hi, full, rtol=1e-12, atol=1e-12 * np.abs(full).max()):
            bad.append(f"windows [0,{cut}) + [{cut},6) differ from the layer")
    whole = O.forward_window(hb, ids, w, w13, s13, w2, s2, 0)
    if not np.array_equal(whole, full):
        bad.append("the window of all experts is not the layer")
    none = O.forward_window(hb, ids, w, w13[:2], s13[:2], w2[:2], s2[:2], 100)
    if not np.all(none == 0):
        bad.append("a window no route falls in is not zero")
    return bad


def check_per_route_sum(O, seed=72):
    hb, ids, w, w13, s13, w2, s2 = case(seed)
    ids = ids.copy()
    ids[2, 1] = -1
    full = O.forward(hb, ids, w, w13, s13, w2, s2)
    o = O.forward_window(hb, ids, w, w13, s13, w2, s2, 0, per_route=True)
    T, k = ids.shape
    y = np.zeros_like(full)
    for j in range(k):
        y += w[:, j:j + 1].astype(np.float64) * o[np.arange(T) * k + j]
    bad = []
    if not np.allclose(y, full, rtol=1e-12, atol=1e-12 * np.abs(full).max()):
        bad.append("weighted per-route outputs do not sum to the layer")
    if not np.all(o[2 * k + 1] == 0):
        bad.append("a padding route's row is not zero")
    # a route's row does not depend on its weight
    o2 = O.forward_window(hb, ids, (3 * w).astype(np.float32), w13, s13, w2, s2, 0, per_route=True)
    if not np.array_equal(o2, o):
        bad.append("per-route rows depend on the routing weights")
    return bad


def test_window_partition():
    assert check_window_partition(O) == []


def test_per_route_sum():
    assert check_per_route_sum(O) == []


def test_window_pins_catch_planted_mistakes():
    def window_off_by_one(hb, ids, w, w13, s13, w2, s2, expert_base=0, per_route=False,
                          intermediate="bf16"):
        return O.forward_window(hb, ids, w, w13, s13, w2, s2, expert_base + 1, per_route,
                                intermediate)

    def weighted_routes(hb, ids, w, w13, s13, w2, s2, expert_base=0, per_route=False,
                        intermediate="bf16"):
        o = O.forward_window(hb, ids, w, w13, s13, w2, s2, expert_base, per_route, intermediate)
        if per_route:
            o = o * np.asarray(w, dtype=np.float64).reshape(-1, 1)
        return o

    for fn, check in ((window_off_by_one, check_window_partition),
                      (weighted_routes, check_per_route_sum)):
        ns = types.SimpleNamespace(**{k: getattr(O, k) for k in dir(O) if not k.startswith("__")})
        ns.forward_window = fn
        assert check(ns) != [], fn.__name__
