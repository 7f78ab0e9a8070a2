"""Pins of the oracle's router (``topk_route``) to things other than itself
(no GPU needed): brute force over all k-subsets on tiny expert counts,
closed-form weights, the tie rule, and the float32 selection reading; planted
mistakes must make a check fail."""
import itertools
import math
import types

import numpy as np

from oracle import mxfp4_moe_oracle as O


def brute_ids(x, k):
    """The k-subset, listed in selection order, that is lexicographically best
    under (value descending, index ascending), by enumeration."""
    E = len(x)
    best = None
    for sub in itertools.permutations(range(E), k):
        key = tuple((-float(x[e]), e) for e in sub)
        ok = all(key[i] <= key[i + 1] for i in range(k - 1))
        if ok and (best is None or key < best[0]):
            best = (key, sub)
    return list(best[1])


def check_router_bruteforce(O, seed=31):
    rng = np.random.default_rng(seed)
    bad = []
    for E, k in ((5, 2), (6, 3), (7, 4), (4, 4), (6, 1)):
        lg = rng.standard_normal((6, E)).astype(np.float32)
        lg[0, :] = 0.5                       # all tied
        lg[1, 1] = lg[1, 3] = lg[1].max() + 1  # a tied maximum
        for scoring in ("softmax_topk", "sigmoid_renorm"):
            ids, _ = O.topk_route(lg, k, scoring)
            for t in range(lg.shape[0]):
                want = brute_ids(lg[t], k)
                if list(ids[t]) != want:
                    bad.append(f"E {E} k {k} {scoring} row {t}: {list(ids[t])} != {want}")
    return bad


def check_router_weights(O, seed=32):
    """Weights that the definitions fix: equal chosen logits give 1/k; the
    softmax of two chosen logits a, b is (1 / (1 + e^(b - a)), ...) and equals
    (0.75, 0.25) at b - a = -ln 3; sigmoid renorm of logits 0 and ln 3 is
    (1/2, 3/4) / (5/4) = (0.4, 0.6); weights sum to 1."""
    bad = []
    lg = np.zeros((1, 6), dtype=np.float32)
    for scoring in ("softmax_topk", "sigmoid_renorm"):
        _, w = O.topk_route(lg, 3, scoring)
        if not np.allclose(w, 1.0 / 3.0, rtol=0, atol=1e-15):
            bad.append(f"{scoring}: equal logits do not give 1/k")
    l3 = np.float32(math.log(3.0))
    lg = np.array([[0.0, -2.0, np.float32(-l3), -3.0]], dtype=np.float32)
    ids, w = O.topk_route(lg, 2, "softmax_topk")
    d = float(np.float32(-l3))
    want = np.array([1.0 / (1.0 + math.exp(d)), 1.0 - 1.0 / (1.0 + math.exp(d))])
    if list(ids[0]) != [0, 2] or not np.allclose(w[0], want, rtol=0, atol=1e-15):
        bad.append(f"softmax of (0, -ln 3): {ids[0]} {w[0]}")
    if not abs(want[0] - 0.75) < 1e-7:
        bad.append("softmax closed form")
    lg = np.array([[-5.0, float(l3), 0.0, -3.0]], dtype=np.float32)
    ids, w = O.topk_route(lg, 2, "sigmoid_renorm")
    s3 = 1.0 / (1.0 + math.exp(-float(l3)))
    want = np.array([s3, 0.5]) / (s3 + 0.5)
    if list(ids[0]) != [1, 2] or not np.allclose(w[0], want, rtol=0, atol=1e-15):
        bad.append(f"sigmoid renorm of (ln 3, 0): {ids[0]} {w[0]}")
    if not abs(want[0] - 0.6) < 1e-7:
        bad.append("sigmoid renorm closed form")
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((20, 64)).astype(np.float32)
    for scoring in ("softmax_topk", "sigmoid_renorm"):
        _, w = O.topk_route(lg, 8, scoring)
        if not np.allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14) or (w <= 0).any():
            bad.append(f"{scoring}: weights do not sum to 1 or are not positive")
        if scoring == "softmax_topk" and not (np.diff(w, axis=1) <= 0).all():
            bad.append("softmax weights not in selection order")
    return bad


def check_router_float32_selection(O):
    """The selection runs on float32(logit + bias): 1 + 2^-25 rounds to 1 in
    float32, so expert 1 (logit 1, bias 2^-25) ties expert 0 (logit 1) and the
    lower index wins; in exact arithmetic expert 1 would come first. A bias of
    2^-23 (one float32 ulp at 1) does move expert 1 ahead."""
    bad = []
    lg = np.array([[1.0, 1.0, 0.0]], dtype=np.float32)
    for b1, want in ((2.0 ** -25, 0), (2.0 ** -23, 1)):
        bias = np.array([0.0, b1, 0.0], dtype=np.float32)
        for scoring in ("softmax_topk", "sigmoid_renorm"):
            ids, _ = O.topk_route(lg, 1, scoring, bias)
            if int(ids[0, 0]) != want:
                bad.append(f"bias {b1} {scoring}: chose {int(ids[0, 0])}, want {want}")
    return bad


def check_router_bias_moves_selection(O, seed=33):
    """A large bias on one expert puts it first for every token."""
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((10, 16)).astype(np.float32)
    bias = np.zeros(16, dtype=np.float32)
    bias[11] = 100.0
    ids, w = O.topk_route(lg, 4, "sigmoid_renorm", bias)
    bad = []
    if not (ids[:, 0] == 11).all():
        bad.append("a +100 bias did not select the expert first")
    return bad


def test_router_bruteforce():
    assert check_router_bruteforce(O) == []


def test_router_weights_closed_forms():
    assert check_router_weights(O) == []


def test_router_float32_selection():
    assert check_router_float32_selection(O) == []


def test_router_bias_moves_selection():
    assert check_router_bias_moves_selection(O) == []


def _with(fn):
    ns = types.SimpleNamespace(**{k: getattr(O, k) for k in dir(O) if not k.startswith("__")})
    ns.topk_route = fn
    return ns


def test_router_pins_catch_planted_mistakes():
    def ties_high(logits, topk, scoring, bias=None):
        x = np.asarray(logits, dtype=np.float32)
        if bias is not None:
            x = (x + np.asarray(bias, dtype=np.float32)).astype(np.float32)
        ids = np.array([sorted(range(x.shape[1]), key=lambda e: (-float(r[e]), -e))[:topk]
                        for r in x], dtype=np.int32)
        return ids, O.topk_route(logits, topk, scoring, bias)[1]

    def double_sum(logits, topk, scoring, bias=None):
        x = np.asarray(logits, dtype=np.float64)
        if bias is not None:
            x = x + np.asarray(bias, dtype=np.float64)
        ids = np.array([sorted(range(x.shape[1]), key=lambda e: (-float(r[e]), e))[:topk]
                        for r in x], dtype=np.int32)
        return ids, O.topk_route(logits, topk, scoring, bias)[1]

    def softmax_all(logits, topk, scoring, bias=None):
        ids, w = O.topk_route(logits, topk, scoring, bias)
        if scoring == "softmax_topk":   # softmax over all E, then pick
            x = np.asarray(logits, dtype=np.float64)
            z = np.exp(x - x.max(axis=1, keepdims=True))
            z = z / z.sum(axis=1, keepdims=True)
            w = np.take_along_axis(z, ids.astype(np.int64), axis=1)
        return ids, w

    def no_renorm(logits, topk, scoring, bias=None):
        ids, w = O.topk_route(logits, topk, scoring, bias)
        if scoring == "sigmoid_renorm":
            x = np.take_along_axis(np.asarray(logits, dtype=np.float64), ids.astype(np.int64), 1)
            w = 1.0 / (1.0 + np.exp(-x))
        return ids, w

    cases = {
        "ties to the higher index": (ties_high, check_router_bruteforce),
        "selection in double": (double_sum, check_router_float32_selection),
        "softmax over all experts": (softmax_all, check_router_weights),
        "sigmoid without renormalisation": (no_renorm, check_router_weights),
    }
    for name, (fn, check) in cases.items():
        assert check(_with(fn)) != [], f"pin did not catch planted mistake: {name}"


# --- grouped top-k and a selection-only bias ----------------------------------

def check_router_grouped_hand(O):
    """Hand-worked cases of grouped top-k (groups of consecutive ids, a
    group's score its largest logit):
    * E = 8 in 4 groups of 2, keep 2 groups, k = 3, logits
      (10, -1 | 3, 2.9 | 2, 1 | 2.95, 2.8): group scores 10, 3, 2, 2.95 keep
      groups 0 and 1, so the choice is 0, 2, 3; without groups it is 0, 2, 6;
    * E = 6 in 3 groups, keep 1, k = 2, logits (5, -4 | 4, 3.5 | 0, 0): the
      largest logit (5) keeps group 0 (ids 0, 1), although group 1 has the
      larger sum;
    * E = 4 in 2 groups, keep 1, k = 1, logits (1, 0 | 0, 1): the groups
      tie, the lower group wins, expert 0."""
    bad = []
    lg = np.array([[10, -1, 3, 2.9, 2, 1, 2.95, 2.8]], dtype=np.float32)
    for scoring in ("softmax_topk", "sigmoid_renorm"):
        ids, _ = O.topk_route(lg, 3, scoring, None, 4, 2)
        if list(ids[0]) != [0, 2, 3]:
            bad.append(f"grouped {scoring}: {list(ids[0])} != [0, 2, 3]")
        ids, _ = O.topk_route(lg, 3, scoring)
        if list(ids[0]) != [0, 2, 6]:
            bad.append(f"ungrouped {scoring}: {list(ids[0])} != [0, 2, 6]")
    ids, _ = O.topk_route(np.array([[5, -4, 4, 3.5, 0, 0]], dtype=np.float32), 2,
                          "sigmoid_renorm", None, 3, 1)
    if list(ids[0]) != [0, 1]:
        bad.append(f"group score is the largest logit: {list(ids[0])} != [0, 1]")
    ids, _ = O.topk_route(np.array([[1, 0, 0, 1]], dtype=np.float32), 1, "softmax_topk",
                          None, 2, 1)
    if list(ids[0]) != [0]:
        bad.append(f"tied groups: {list(ids[0])} != [0]")
    return bad


def brute_grouped(x, k, n_group, topk_group):
    """Grouped choice by a second formulation: a group is kept when fewer than
    topk_group groups beat it (a larger score, or an equal score and a lower
    index); the experts then by enumeration over the kept ones."""
    E = len(x)
    gs = E // n_group
    score = [max(float(v) for v in x[g * gs:(g + 1) * gs]) for g in range(n_group)]
    kept = [g for g in range(n_group)
            if sum(1 for h in range(n_group)
                   if score[h] > score[g] or (score[h] == score[g] and h < g)) < topk_group]
    elig = [e for e in range(E) if e // gs in kept]
    sub = brute_ids(np.array([x[e] for e in elig]), k)
    return [elig[i] for i in sub]


def check_router_grouped_bruteforce(O, seed=34):
    rng = np.random.default_rng(seed)
    bad = []
    for E, n_group, topk_group, k in ((6, 3, 1, 2), (8, 4, 2, 3), (8, 2, 1, 4), (9, 3, 2, 4),
                                      (8, 4, 4, 3), (6, 1, 1, 3)):
        lg = rng.standard_normal((8, E)).astype(np.float32)
        lg[0, :] = 0.25                                   # everything tied
        lg[1] = np.round(lg[1] * 2) / 2                   # coarse grid: ties
        lg[2, ::2] = lg[2].max() + 1                      # tied group maxima
        for t in range(lg.shape[0]):
            ids, _ = O.topk_route(lg[t:t + 1], k, "softmax_topk", None, n_group, topk_group)
            want = brute_grouped(lg[t], k, n_group, topk_group)
            if list(ids[0]) != want:
                bad.append(f"E {E} groups {n_group}/{topk_group} k {k} row {t}: "
                           f"{list(ids[0])} != {want}")
    return bad


def check_router_grouped_special_cases(O, seed=35):
    """Keeping every group, or a single group holding all experts, is the
    ungrouped router."""
    rng = np.random.default_rng(seed)
    lg = rng.standard_normal((12, 64)).astype(np.float32)
    bias = (0.5 * rng.standard_normal(64)).astype(np.float32)
    ref = O.topk_route(lg, 6, "sigmoid_renorm", bias)
    bad = []
    for n_group, topk_group in ((8, 8), (1, 1)):
        got = O.topk_route(lg, 6, "sigmoid_renorm", bias, n_group, topk_group)
        if not (np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])):
            bad.append(f"{n_group}/{topk_group} groups differ from the plain router")
    return bad


def check_router_selection_bias(O):
    """With the bias steering the choice only, logits (1, 0.5, 0) and bias
    (0, 1, 0) choose experts 1, 0 (x = 1.5, 1) and weigh them by the unbiased
    logits (0.5, 1): softmax (1 / (1 + e^0.5), 1 / (1 + e^-0.5)) and sigmoid
    renorm (s(0.5), s(1)) / (s(0.5) + s(1)); with the bias in the weights,
    (1 / (1 + e^-0.5), 1 / (1 + e^0.5)) and (s(1.5), s(1)) / sum. Without a
    bias the two readings agree."""
    def sg(z):
        return 1.0 / (1.0 + math.exp(-z))
    lg = np.array([[1.0, 0.5, 0.0]], dtype=np.float32)
    bias = np.array([0.0, 1.0, 0.0], dtype=np.float32)
    want = {
        ("softmax_topk", False): [sg(-0.5), sg(0.5)],
        ("softmax_topk", True): [sg(0.5), sg(-0.5)],
        ("sigmoid_renorm", False): [sg(0.5) / (sg(0.5) + sg(1.0)), sg(1.0) / (sg(0.5) + sg(1.0))],
        ("sigmoid_renorm", True): [sg(1.5) / (sg(1.5) + sg(1.0)), sg(1.0) / (sg(1.5) + sg(1.0))],
    }
    bad = []
    for (scoring, in_w), wv in want.items():
        ids, w = O.topk_route(lg, 2, scoring, bias, bias_in_weights=in_w)
        if list(ids[0]) != [1, 0] or not np.allclose(w[0], wv, rtol=0, atol=1e-15):
            bad.append(f"{scoring} bias_in_weights={in_w}: {list(ids[0])} {w[0]} != {wv}")
    rng = np.random.default_rng(36)
    lg = rng.standard_normal((6, 32)).astype(np.float32)
    a = O.topk_route(lg, 4, "softmax_topk", None, bias_in_weights=False)
    b = O.topk_route(lg, 4, "softmax_topk", None)
    if not (np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])):
        bad.append("without a bias the selection-only reading changes the result")
    return bad


def test_router_grouped_hand_cases():
    assert check_router_grouped_hand(O) == []


def test_router_grouped_bruteforce():
    assert check_router_grouped_bruteforce(O) == []


def test_router_grouped_special_cases():
    assert check_router_grouped_special_cases(O) == []


def test_router_selection_only_bias():
    assert check_router_selection_bias(O) == []


def test_grouped_pins_catch_planted_mistakes():
    def grouped(logits, topk, scoring, bias=None, n_group=1, topk_group=1,
                bias_in_weights=True, score="max", strided=False, tie_high=False):
        """The oracle's grouped selection with one step changed."""
        x = np.asarray(logits, dtype=np.float32)
        if bias is not None:
            x = (x + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)
        T, E = x.shape
        gs = E // n_group
        grp = (lambda e: e % n_group) if strided else (lambda e: e // gs)
        ids = np.empty((T, topk), dtype=np.int32)
        for t in range(T):
            members = [[e for e in range(E) if grp(e) == g] for g in range(n_group)]
            agg = max if score == "max" else sum
            gscore = [agg(float(x[t, e]) for e in m) for m in members]
            kept = sorted(range(n_group),
                          key=lambda g: (-gscore[g], -g if tie_high else g))[:topk_group]
            elig = [e for e in range(E) if grp(e) in kept]
            ids[t] = sorted(elig, key=lambda e: (-float(x[t, e]), e))[:topk]
        ref_w = O.topk_route(logits, topk, scoring, bias, n_group, topk_group, bias_in_weights)[1]
        return ids, ref_w

    def weights_always_biased(logits, topk, scoring, bias=None, n_group=1, topk_group=1,
                              bias_in_weights=True):
        return O.topk_route(logits, topk, scoring, bias, n_group, topk_group, True)

    cases = {
        "group score is the sum": (lambda *a, **kw: grouped(*a, **kw, score="sum"),
                                   check_router_grouped_hand),
        "strided groups": (lambda *a, **kw: grouped(*a, **kw, strided=True),
                           check_router_grouped_hand),
        "tied groups to the higher index": (lambda *a, **kw: grouped(*a, **kw, tie_high=True),
                                            check_router_grouped_bruteforce),
        "bias always in the weights": (weights_always_biased, check_router_selection_bias),
    }
    for name, (fn, check) in cases.items():
        assert check(_with(fn)) != [], f"pin did not catch planted mistake: {name}"
