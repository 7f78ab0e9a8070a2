"""Pins of the oracle's gpt-oss form (``forward_oai``, ``swiglu_oai``) to
things other than itself (no GPU needed): exact values of the activation that
follow from its definition ("MXFP4 MoE decode kernels", Design, Fused
epilogues), closed forms of the layer when the weights vanish, and a brute
force over exact rationals on tiny shapes that reads the interleaved rows by its
own indexing ("Read the served layout": gate and up rows interleaved). Each
check returns a list of failures, and planted mistakes in a copy of the oracle
must make at least one of them fail.
"""
import math
import types
from fractions import Fraction

import numpy as np
import pytest

from oracle import mxfp4_moe_oracle as O
from test_oracle_pins import dequant_by_bits, small_case


def oai_case(rng, T, K, I, E, k, bias_scale=1.0):
    hb, ids, w, w13, s13, w2, s2 = small_case(rng, T, K, I, E, k)
    b13 = (bias_scale * rng.standard_normal((E, 2 * I))).astype(np.float32)
    b2 = (bias_scale * rng.standard_normal((E, K))).astype(np.float32)
    return hb, ids, w, w13, s13, b13, w2, s2, b2


# ---------------------------------------------------------------------------
# the activation
# ---------------------------------------------------------------------------
def check_oai_activation(O):
    """Values that the definition fixes exactly:
    * gate 0 or up -1 give 0 whatever the other input;
    * the gate cap: every gate >= 7 gives the value at 7; no lower cap;
    * the up clamp: up >= 7 gives the value at 7, up <= -7 the value at -7;
    * sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4, so at gate = +-ln(3)/1.702
      the value is gate * 3/4 * (up + 1) or gate * 1/4 * (up + 1);
    * g sigmoid(a g) - (-g) sigmoid(-a g) = g (sigmoid(x) + sigmoid(-x) = 1),
      so f(g, u) - f(-g, u) = g (u + 1) wherever |g| <= 7."""
    f = O.swiglu_oai
    bad = []
    us = np.array([-9.0, -7.0, -3.5, -1.0, 0.0, 0.25, 2.0, 6.5, 7.0, 11.0])
    gs = np.array([-12.0, -7.0, -2.0, -0.5, 0.0, 0.75, 3.0, 6.9, 7.0, 7.01, 50.0])
    if not np.all(f(np.zeros_like(us), us) == 0.0):
        bad.append("gate 0 is not 0")
    if not np.all(f(gs, -np.ones_like(gs)) == 0.0):
        bad.append("up -1 is not 0")
    for u in us:
        at7 = f(7.0, u)
        if not (f(7.01, u) == at7 and f(50.0, u) == at7 and f(1e30, u) == at7):
            bad.append(f"gate cap: gate > 7 differs from gate = 7 at up {u}")
        if u != -1.0 and f(-12.0, u) == f(-7.0, u):
            bad.append("gate is capped from below")
    for g in gs:
        if not (f(g, 7.5) == f(g, 7.0) and f(g, 1e30) == f(g, 7.0)):
            bad.append(f"up clamp above at gate {g}")
        if not (f(g, -7.5) == f(g, -7.0) and f(g, -1e30) == f(g, -7.0)):
            bad.append(f"up clamp below at gate {g}")
        if g != 0.0 and f(g, 6.5) == f(g, 7.0):
            bad.append("up clamped below 7")
    g3 = math.log(3.0) / 1.702
    for u in us:
        uc = min(max(u, -7.0), 7.0)
        for g, sig in ((g3, 0.75), (-g3, 0.25)):
            want = g * sig * (uc + 1.0)
            if not abs(f(g, u) - want) <= 1e-15 * max(1.0, abs(want)):
                bad.append(f"sigmoid(1.702 g) at g = {g:.6f}, up {u}: {f(g, u)} != {want}")
    for g in (0.3, 1.0, 2.5, 6.0, 7.0):
        for u in (-3.0, 0.0, 4.0):
            d = f(g, u) - f(-g, u)
            if not abs(d - g * (u + 1.0)) <= 1e-13 * abs(g * (u + 1.0)):
                bad.append(f"f(g,u) - f(-g,u) != g (u+1) at g {g}, u {u}")
    if not np.isnan(f(np.nan, 1.0)) or not np.isnan(f(1.0, np.nan)):
        bad.append("NaN does not propagate")
    return bad


# ---------------------------------------------------------------------------
# closed forms of the layer
# ---------------------------------------------------------------------------
def check_oai_bias_only(O, seed=11):
    """All weight codes 0 (value 0 for every scale): o = b2[e] per route, so
    y_t = sum over valid slots of w_tj * b2[e_tj] exactly (in float64)."""
    rng = np.random.default_rng(seed)
    T, K, I, E, k = 5, 64, 32, 6, 3
    hb, ids, w, w13, s13, b13, w2, s2, b2 = oai_case(rng, T, K, I, E, k)
    w13 = np.zeros_like(w13)
    w2 = np.zeros_like(w2)
    ids = ids.copy()
    ids[1, 2] = -1                                    # a padding slot
    want = np.zeros((T, K))
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            if 0 <= e < E:
                want[t] += float(w[t, j]) * b2[e].astype(np.float64)
    bad = []
    for mode in ("bf16", "fp32"):
        got = O.forward_oai(hb, ids, w, w13, s13, b13, w2, s2, b2, intermediate=mode)
        if not np.allclose(got, want, rtol=1e-15, atol=0.0):
            bad.append(f"bias-only layer, mode {mode}: max err {np.abs(got - want).max()}")
    return bad


def check_oai_gate_bias_closed_form(O, seed=12):
    """w13 codes 0, gate bias ln(3)/1.702 (sigmoid exactly 3/4) on pair i,
    gate bias 0 on the other pairs, up bias c: h = g3 * 3/4 * (c + 1) on pair i
    and 0 elsewhere, so o = W2[:, i] h_i + b2 with W2 from an independent
    dequant (fp32 intermediate)."""
    rng = np.random.default_rng(seed)
    T, K, I, E, k = 2, 64, 32, 1, 1
    hb, _, _, w13, s13, b13, w2, s2, b2 = oai_case(rng, T, K, I, E, k)
    ids = np.zeros((T, 1), dtype=np.int32)
    w = np.array([[0.5], [2.0]], dtype=np.float32)
    w13 = np.zeros_like(w13)
    g3 = math.log(3.0) / 1.702
    i, c = 5, 1.5
    b13 = np.zeros((E, 2 * I), dtype=np.float64)
    b13[0, 2 * i] = g3            # gate of pair i (even row)
    b13[0, 1::2] = c              # every up bias
    h = np.zeros(I)
    h[i] = g3 * 0.75 * (c + 1.0)
    W2 = dequant_by_bits(w2[0], s2[0])
    o = W2 @ h + b2[0].astype(np.float64)
    want = np.stack([0.5 * o, 2.0 * o])
    got = O.forward_oai(hb, ids, w, w13, s13, b13, w2, s2, b2, intermediate="fp32")
    bad = []
    if not np.allclose(got, want, rtol=1e-13, atol=1e-13 * np.abs(want).max()):
        bad.append(f"gate-bias closed form: max err {np.abs(got - want).max()}")
    return bad


def exact_layer_oai(hb, ids, w, w13, s13, b13, w2, s2, b2, mode):
    """Brute force for tiny shapes: dot products in exact rationals with the
    gate of pair n read from row 2n and the up from row 2n + 1, biases added
    exactly, the activation at 50 digits, the w2 bias per route."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    T, k = ids.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    K = w2.shape[1]
    xs = [[Fraction(float(v)) for v in row]
          for row in (hb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)]
    alpha = mpmath.mpf(1702) / 1000

    def act(g, u):
        g = min(g, mpmath.mpf(7))
        u = min(max(u, mpmath.mpf(-7)), mpmath.mpf(7))
        return g / (1 + mpmath.e ** (-alpha * g)) * (u + 1)

    y = np.zeros((T, K))
    for t in range(T):
        acc = [Fraction(0)] * K
        for j in range(k):
            e = int(ids[t, j])
            if e < 0 or e >= E:
                continue
            W13 = dequant_by_bits(w13[e], s13[e])
            W2 = dequant_by_bits(w2[e], s2[e])
            h = []
            for n in range(I):
                g = sum(Fraction(W13[2 * n, c]) * xs[t][c] for c in range(K)) + Fraction(float(b13[e, 2 * n]))
                u = sum(Fraction(W13[2 * n + 1, c]) * xs[t][c] for c in range(K)) + Fraction(float(b13[e, 2 * n + 1]))
                hv = act(mpmath.mpf(g.numerator) / g.denominator, mpmath.mpf(u.numerator) / u.denominator)
                hf = float(hv)
                if mode == "bf16":
                    hf = float(O.round_to_bf16(np.array([hf]))[0])
                    h.append(Fraction(hf))
                else:
                    h.append(hv)
            for m in range(K):
                if mode == "bf16":
                    o = sum(Fraction(W2[m, n]) * h[n] for n in range(I)) + Fraction(float(b2[e, m]))
                else:
                    o = Fraction(float(sum(mpmath.mpf(W2[m, n]) * h[n] for n in range(I)))) + Fraction(float(b2[e, m]))
                acc[m] += Fraction(float(w[t, j])) * o
        y[t] = [float(a) for a in acc]
    return y


def check_oai_bruteforce_tiny(O, seed=13):
    rng = np.random.default_rng(seed)
    hb, ids, w, w13, s13, b13, w2, s2, b2 = oai_case(rng, 3, 32, 32, 3, 2, bias_scale=4.0)
    bad = []
    for mode in ("bf16", "fp32"):
        want = exact_layer_oai(hb, ids, w, w13, s13, b13, w2, s2, b2, mode)
        got = O.forward_oai(hb, ids, w, w13, s13, b13, w2, s2, b2, intermediate=mode)
        rel = np.abs(got - want).max() / np.abs(want).max()
        if not rel <= 1e-12:
            bad.append(f"brute force mode {mode}: max rel {rel}")
    return bad


def check_oai_clamps_active(O, seed=14):
    """On inputs of the workloads' statistics (K = 512), the pre-activations
    reach past the cap and clamp, so the pins above see them at work: some
    gates exceed 7, some ups leave [-7, 7], and reading the rows as [gate; up]
    instead of interleaved moves the output far past the 3e-3 gate."""
    rng = np.random.default_rng(seed)
    T, K, I, E, k = 4, 512, 256, 4, 2
    hb, ids, w, w13, s13, b13, w2, s2, b2 = oai_case(rng, T, K, I, E, k)
    x = O.bf16_bits_to_float(hb)
    W = O.dequant(w13[ids[0, 0]], s13[ids[0, 0]])
    g = x @ W[0::2].T
    u = x @ W[1::2].T
    bad = []
    if not (g > 7).any():
        bad.append("no gate above the cap")
    if not (np.abs(u) > 7).any():
        bad.append("no up outside the clamp")
    base = O.forward_oai(hb, ids, w, w13, s13, b13, w2, s2, b2)
    blocked = np.concatenate([w13[:, 0::2], w13[:, 1::2]], axis=1)
    sblocked = np.concatenate([s13[:, 0::2], s13[:, 1::2]], axis=1)
    other = O.forward_oai(hb, ids, w, blocked, sblocked, b13, w2, s2, b2)
    rel = np.linalg.norm(other - base) / np.linalg.norm(base)
    if not rel > 0.1:
        bad.append(f"[gate; up] reading only moved rel_l2 by {rel}")
    return bad


# ---------------------------------------------------------------------------
# tests
# ---------------------------------------------------------------------------
def test_oai_activation_exact_values():
    assert check_oai_activation(O) == []


def test_oai_bias_only_closed_form():
    assert check_oai_bias_only(O) == []


def test_oai_gate_bias_closed_form():
    assert check_oai_gate_bias_closed_form(O) == []


def test_oai_bruteforce_tiny_exact():
    assert check_oai_bruteforce_tiny(O) == []


def test_oai_clamps_active_and_interleave_matters():
    assert check_oai_clamps_active(O) == []


# ---------------------------------------------------------------------------
# planted mistakes
# ---------------------------------------------------------------------------
def _oracle_with(**repl):
    """A copy of the oracle's namespace with names replaced; forward_oai is
    re-bound to it (unless replaced) so it calls the replaced activation."""
    ns = types.SimpleNamespace(**{k: getattr(O, k) for k in dir(O) if not k.startswith("__")})
    for k, v in repl.items():
        setattr(ns, k, v)
    if "forward_oai" not in repl:
        fn = O.forward_oai
        g = dict(fn.__globals__)
        g.update(vars(ns))
        ns.forward_oai = types.FunctionType(fn.__code__, g, fn.__name__, fn.__defaults__,
                                            fn.__closure__)
    return ns


def _act(alpha=1.702, cap_lo=None, up_lo=-7.0, up_hi=7.0, plus_one=1.0):
    def f(g, u):
        g = np.minimum(np.asarray(g, dtype=np.float64), 7.0)
        if cap_lo is not None:
            g = np.maximum(g, cap_lo)
        u = np.clip(np.asarray(u, dtype=np.float64), up_lo, up_hi)
        return g * (1.0 / (1.0 + np.exp(-alpha * g))) * (u + plus_one)
    return f


def test_oai_pins_catch_planted_mistakes():
    def fwd_swapped_pairs(hb, ids, w, w13, s13, b13, w2, s2, b2, **kw):
        sw = w13.copy(); sw[:, 0::2], sw[:, 1::2] = w13[:, 1::2], w13[:, 0::2]
        ss = s13.copy(); ss[:, 0::2], ss[:, 1::2] = s13[:, 1::2], s13[:, 0::2]
        bb = np.array(b13, dtype=np.float64).copy()
        bb[:, 0::2], bb[:, 1::2] = np.array(b13)[:, 1::2], np.array(b13)[:, 0::2]
        return O.forward_oai(hb, ids, w, sw, ss, bb, w2, s2, b2, **kw)

    def fwd_bias2_per_token(hb, ids, w, w13, s13, b13, w2, s2, b2, **kw):
        # the w2 bias added once per token (unweighted) instead of per route
        y = O.forward_oai(hb, ids, w, w13, s13, b13, w2, s2, np.zeros_like(b2), **kw)
        e0 = np.asarray(ids)[:, 0].clip(0)
        return y + np.asarray(b2, dtype=np.float64)[e0]

    def fwd_no_bias13(hb, ids, w, w13, s13, b13, w2, s2, b2, **kw):
        return O.forward_oai(hb, ids, w, w13, s13, np.zeros_like(b13), w2, s2, b2, **kw)

    mutants = {
        "alpha 1.0": (_oracle_with(swiglu_oai=_act(alpha=1.0)), [check_oai_activation, check_oai_gate_bias_closed_form]),
        "gate capped below": (_oracle_with(swiglu_oai=_act(cap_lo=-7.0)), [check_oai_activation]),
        "up not clamped below": (_oracle_with(swiglu_oai=_act(up_lo=-1e300)), [check_oai_activation]),
        "no +1 on up": (_oracle_with(swiglu_oai=_act(plus_one=0.0)), [check_oai_activation, check_oai_gate_bias_closed_form]),
        "gate/up swapped in pairs": (_oracle_with(forward_oai=fwd_swapped_pairs), [check_oai_bruteforce_tiny, check_oai_gate_bias_closed_form]),
        "w2 bias per token": (_oracle_with(forward_oai=fwd_bias2_per_token), [check_oai_bias_only]),
        "w13 bias dropped": (_oracle_with(forward_oai=fwd_no_bias13), [check_oai_gate_bias_closed_form, check_oai_bruteforce_tiny]),
    }
    for name, (m, checks) in mutants.items():
        for check in checks:
            assert check(m) != [], f"{check.__name__} did not catch planted mistake: {name}"
