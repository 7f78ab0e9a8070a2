"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each check is a function returning a list of failures, so the same check can
be run against the oracle as written (must pass) and against a copy of the
oracle with a planted mistake (must fail): that shows each pin is able to
catch the mistake it is meant to catch.
"""
import math
import os
from fractions import Fraction

import numpy as np
import torch

from oracle import mxfp4_moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# Independent constructions (written from the format definitions, no table)
# ---------------------------------------------------------------------------
def e2m1_by_bits(code: int) -> float:
    """E2M1 value from its bit fields: sign bit 3, exponent bits 2..1 (bias 1),
    mantissa bit 0; exponent 0 is subnormal (m * 0.5)."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = m * 0.5 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


def bf16_bits_by_integers(code: int, sbyte: int) -> int:
    """bf16 bit pattern of E2M1(code) * 2^(sbyte-127) built with integer
    arithmetic only (value = N * 2^P with a small integer N)."""
    if sbyte == 255:
        return -1  # NaN: compared as a class, not by payload
    sign = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        N, P = m, sbyte - 127 - 1           # m * 0.5 * 2^(s-127)
    else:
        N, P = 2 + m, e - 2 + sbyte - 127   # (1 + m/2) * 2^(e-1) = (2+m) * 2^(e-2)
    if N == 0:
        return sign << 15
    # normalise N * 2^P = 1.f * 2^X
    X = P + N.bit_length() - 1
    if X > 127:
        return (sign << 15) | 0x7F80      # overflow -> inf
    if X >= -126:
        frac = (N << 7 >> (N.bit_length() - 1)) & 0x7F   # N has <= 2 significant bits
        return (sign << 15) | ((X + 127) << 7) | frac
    # subnormal: value = F * 2^-133 with integer F < 128
    shift = P + 133
    assert shift >= 0, "E2M1 * 2^-127 never drops below the subnormal grid"
    return (sign << 15) | (N << shift)


# ---------------------------------------------------------------------------
# Checks (return lists of failure strings)
# ---------------------------------------------------------------------------
def check_golden_table(O):
    bad = []
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_codes.txt"))
            if l.strip() and not l.startswith("#")]
    for code_s, val_s in rows:
        code, want = int(code_s), float(val_s)
        packed = np.array([[code | (code << 4)] * 16], dtype=np.uint8)
        got = O.dequant(packed, np.array([[127]], dtype=np.uint8))[0]
        if not all(math.copysign(1, g) == math.copysign(1, want) and g == want for g in got):
            bad.append(f"code {code}: {got[:2]} != {want}")
        if e2m1_by_bits(code) != want or math.copysign(1, e2m1_by_bits(code)) != math.copysign(1, want):
            bad.append(f"bit construction disagrees with golden for code {code}")
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e8m0_examples.txt"))
            if l.strip() and not l.startswith("#")]
    for b_s, v_s in rows:
        b = int(b_s)
        want = float("nan") if v_s == "nan" else float.fromhex(v_s)
        got = float(O.e8m0_value(np.array([b]))[0])
        if not ((math.isnan(want) and math.isnan(got)) or got == want):
            bad.append(f"e8m0 {b}: {got} != {want}")
    return bad


def check_dequant_sweep(O):
    """All 16 codes x all 256 scale bytes: oracle bf16 bits == integer construction."""
    bad = []
    codes = np.arange(16, dtype=np.uint8)
    for s in range(256):
        # one row of 32 values: codes 0..15 twice, packed low nibble first
        vals = np.concatenate([codes, codes])
        packed = (vals[0::2] | (vals[1::2] << 4)).astype(np.uint8)[None, :]
        got = O.float_to_bf16_bits(O.dequant(packed, np.array([[s]], dtype=np.uint8)))[0]
        for i, c in enumerate(vals.tolist()):
            want = bf16_bits_by_integers(c, s)
            g = int(got[i])
            if want == -1:
                if not ((g & 0x7F80) == 0x7F80 and (g & 0x7F) != 0):
                    bad.append(f"s={s} code={c}: expected NaN, got {g:#06x}")
            elif g != want:
                bad.append(f"s={s} code={c}: {g:#06x} != {want:#06x}")
    return bad


def check_low_nibble_first(O):
    packed = np.array([[0x21] + [0] * 15], dtype=np.uint8)  # low nibble 1 (0.5), high 2 (1.0)
    got = O.dequant(packed, np.array([[127]], dtype=np.uint8))[0, :2]
    return [] if got.tolist() == [0.5, 1.0] else [f"nibble order: {got}"]


def brute_route(ids, E):
    flat = np.asarray(ids).reshape(-1)
    R = flat.size
    count, lst = [], []
    for e in range(E):
        rs = [r for r in range(R) if flat[r] == e]
        count.append(len(rs))
        lst += rs
    invalid = int(sum(1 for r in range(R) if flat[r] >= E))
    return np.array(count), np.array(lst, dtype=np.int64), invalid


def check_route(O, seed=0):
    rng = np.random.default_rng(seed)
    bad = []
    cases = [
        rng.integers(-1, 9, size=(7, 3)),                 # padding and invalid ids
        np.full((5, 2), 3),                               # all routes to one expert
        rng.integers(0, 64, size=(2, 2)),                 # E >> R
        np.full((3, 4), -1),                              # nothing routed
        rng.integers(0, 8, size=(33, 4)),                 # more than one warp of routes
    ]
    Es = [8, 8, 64, 8, 8]
    for ids, E in zip(cases, Es):
        rt = O.route(ids, E)
        c, l, inv = brute_route(ids, E)
        if not np.array_equal(rt["count"], c):
            bad.append(f"count {rt['count']} != {c}")
        if not np.array_equal(rt["list"], l):
            bad.append(f"list {rt['list']} != {l}")
        if rt["invalid"] != inv:
            bad.append(f"invalid {rt['invalid']} != {inv}")
        if not np.array_equal(rt["offset"], np.concatenate([[0], np.cumsum(c)])):
            bad.append("offset")
        if not np.array_equal(rt["touched"], np.nonzero(c)[0]):
            bad.append("touched")
    return bad


def small_case(rng, T, K, I, E, k, scales=(118, 124)):
    hidden = torch.from_numpy(rng.standard_normal((T, K), dtype=np.float32)).to(torch.bfloat16)
    hb = hidden.view(torch.int16).numpy().view(np.uint16)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32) + 0.1
    w13 = rng.integers(0, 256, (E, 2 * I, K // 2), dtype=np.uint8)
    s13 = rng.integers(scales[0], scales[1] + 1, (E, 2 * I, K // 32), dtype=np.uint8)
    w2 = rng.integers(0, 256, (E, K, I // 2), dtype=np.uint8)
    s2 = rng.integers(scales[0], scales[1] + 1, (E, K, I // 32), dtype=np.uint8)
    return hb, ids, w, w13, s13, w2, s2


def dequant_by_bits(packed, scale):
    """Independent dequant: per-code bit construction, scale by math.ldexp."""
    table = np.array([e2m1_by_bits(c) for c in range(16)])
    rows, half = packed.shape
    out = np.empty((rows, 2 * half))
    for n in range(rows):
        for c in range(2 * half):
            byte = int(packed[n, c // 2])
            code = (byte >> 4) if (c & 1) else (byte & 0xF)
            out[n, c] = math.ldexp(table[code], int(scale[n, c // 32]) - 127)
    return out


def check_dense_mlp(O, seed=1):
    """One expert, top-1 with weight 1: the layer is a dense MLP
    W2 . (silu(Wg x) * (Wu x)) computed here with independent dequant and a
    numpy float64 matmul."""
    rng = np.random.default_rng(seed)
    T, K, I = 3, 64, 32
    hb, _, _, w13, s13, w2, s2 = small_case(rng, T, K, I, 1, 1)
    ids = np.zeros((T, 1), dtype=np.int32)
    w = np.ones((T, 1), dtype=np.float32)
    x = (hb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    W13 = dequant_by_bits(w13[0], s13[0])
    W2 = dequant_by_bits(w2[0], s2[0])
    g = x @ W13[:I].T
    u = x @ W13[I:].T
    h = g / (1.0 + np.exp(-g)) * u
    want_b = h @ W2.T
    want_a = O.round_to_bf16(h) @ W2.T
    bad = []
    for mode, want in (("fp32", want_b), ("bf16", want_a)):
        got = O.forward(hb, ids, w, w13, s13, w2, s2, intermediate=mode)
        rel = np.linalg.norm(got - want) / np.linalg.norm(want)
        if not rel <= 1e-12:
            bad.append(f"dense MLP mode {mode}: rel {rel}")
    return bad


def exact_layer(hb, ids, w, w13, s13, w2, s2, mode):
    """Brute force for tiny shapes: dot products in exact rationals, SiLU at 50
    digits, combine in slot order (mode bf16 rounds h via the pinned rounder)."""
    import mpmath
    mpmath.mp.dps = 50
    T, k = ids.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    K = w2.shape[1]
    xs = [[Fraction(float(v)) for v in row]
          for row in (hb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)]
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
                g = sum(Fraction(W13[n, c]) * xs[t][c] for c in range(K))
                u = sum(Fraction(W13[I + n, c]) * xs[t][c] for c in range(K))
                gm = mpmath.mpf(g.numerator) / g.denominator
                hv = gm / (1 + mpmath.e ** (-gm)) * (mpmath.mpf(u.numerator) / u.denominator)
                hf = float(hv)
                if mode == "bf16":
                    hf = float(O.round_to_bf16(np.array([hf]))[0])
                h.append(Fraction(hf) if mode == "bf16" else hv)
            for m in range(K):
                if mode == "bf16":
                    o = sum(Fraction(W2[m, n]) * h[n] for n in range(I))
                    acc[m] += Fraction(float(w[t, j])) * o
                else:
                    o = sum(mpmath.mpf(W2[m, n]) * h[n] for n in range(I))
                    acc[m] += Fraction(float(w[t, j])) * Fraction(float(o))
        y[t] = [float(a) for a in acc]
    return y


def check_bruteforce_tiny(O, seed=2):
    rng = np.random.default_rng(seed)
    hb, ids, w, w13, s13, w2, s2 = small_case(rng, 3, 32, 32, 3, 2)
    bad = []
    for mode in ("bf16", "fp32"):
        want = exact_layer(hb, ids, w, w13, s13, w2, s2, mode)
        got = O.forward(hb, ids, w, w13, s13, w2, s2, intermediate=mode)
        rel = np.abs(got - want).max() / np.abs(want).max()
        if not rel <= 1e-12:
            bad.append(f"brute force mode {mode}: max rel {rel}")
    return bad


def check_invariants(O, seed=3):
    rng = np.random.default_rng(seed)
    T, K, I, E, k = 5, 64, 32, 6, 3
    hb, ids, w, w13, s13, w2, s2 = small_case(rng, T, K, I, E, k)
    base = O.forward(hb, ids, w, w13, s13, w2, s2)
    bad = []
    # expert relabelling
    perm = rng.permutation(E)
    inv = np.argsort(perm)
    got = O.forward(hb, perm[ids].astype(np.int32), w, w13[inv], s13[inv], w2[inv], s2[inv])
    if not np.array_equal(got, base):
        bad.append("expert relabelling changed the output")
    # token permutation
    tp = rng.permutation(T)
    got = O.forward(hb[tp], ids[tp], w[tp], w13, s13, w2, s2)
    if not np.array_equal(got, base[tp]):
        bad.append("token permutation is not a row permutation")
    # power-of-two weight scaling
    got = O.forward(hb, ids, (2 * w).astype(np.float32), w13, s13, w2, s2)
    if not np.array_equal(got, 2 * base):
        bad.append("scaling the weights by 2 did not scale y by exactly 2")
    # padding slots contribute nothing
    ids_pad = ids.copy()
    ids_pad[:, -1] = -1
    got = O.forward(hb, ids_pad, w, w13, s13, w2, s2)
    want = O.forward(hb, ids[:, :-1], w[:, :-1], w13, s13, w2, s2)
    if not np.array_equal(got, want):
        bad.append("a -1 slot changed the output")
    return bad


def check_negative_control(O, seed=4):
    """Swapping the [gate; up] halves must move the output far past the 3e-3
    gate on inputs of the workloads' statistics (SiLU driven non-linear)."""
    rng = np.random.default_rng(seed)
    T, K, I, E, k = 4, 512, 256, 4, 2
    hb, ids, w, w13, s13, w2, s2 = small_case(rng, T, K, I, E, k)
    base = O.forward(hb, ids, w, w13, s13, w2, s2)
    swapped = np.concatenate([w13[:, I:], w13[:, :I]], axis=1)
    sswapped = np.concatenate([s13[:, I:], s13[:, :I]], axis=1)
    got = O.forward(hb, ids, w, swapped, sswapped, w2, s2)
    rel = np.linalg.norm(got - base) / np.linalg.norm(base)
    bad = []
    if not rel > 0.1:
        bad.append(f"[up; gate] control only moved rel_l2 by {rel}")
    # the pre-activations are large, so SiLU is far from linear
    x = O.bf16_bits_to_float(hb)
    g = x @ O.dequant(w13[ids[0, 0]], s13[ids[0, 0]])[:I].T
    if not np.sqrt(np.mean(g ** 2)) > 2.0:
        bad.append("gate pre-activation RMS too small to drive SiLU non-linear")
    return bad


# ---------------------------------------------------------------------------
# Tests
# ---------------------------------------------------------------------------
def test_golden_tables():
    assert check_golden_table(O) == []


def test_dequant_sweep_all_codes_all_scales():
    assert check_dequant_sweep(O) == []


def test_low_nibble_first():
    assert check_low_nibble_first(O) == []


def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(5)
    np.seterr(over="ignore")
    f = rng.standard_normal(20000).astype(np.float32) * np.float32(2.0) ** rng.integers(-140, 128, 20000).astype(np.float32)
    ties = (np.float32(1.0) + np.float32(2.0) ** np.float32(-8)) * np.float32(2.0) ** rng.integers(-120, 120, 200).astype(np.float32)
    edge = np.array([3.3895313892515355e38, 3.3961775292304e38, 1e-40, -1e-45, 0.0, -0.0,
                     np.float32(1.0) + np.float32(3.0) * np.float32(2.0) ** np.float32(-8)], dtype=np.float32)
    v = np.concatenate([f, ties, -ties, edge]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = O.round_to_bf16(v.astype(np.float64))
    both_nan = np.isnan(want) & np.isnan(got)
    same = (got == want) & (np.signbit(got) == np.signbit(want))
    assert np.all(same | both_nan), v[~(same | both_nan)][:10]


def test_bf16_bits_roundtrip():
    np.seterr(invalid="ignore")
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_bits_to_float(bits)
    back = O.float_to_bf16_bits(vals)
    nan = np.isnan(vals)
    assert np.array_equal(back[~nan], bits[~nan])


def test_route_against_brute_force():
    assert check_route(O) == []


def test_dense_mlp_special_case():
    assert check_dense_mlp(O) == []


def test_bruteforce_tiny_exact():
    assert check_bruteforce_tiny(O) == []


def test_invariants():
    assert check_invariants(O) == []


def test_negative_control_gate_up_order():
    assert check_negative_control(O) == []


def test_outputs_finite_on_workload_statistics():
    rng = np.random.default_rng(6)
    hb, ids, w, w13, s13, w2, s2 = small_case(rng, 2, 2880, 2880, 2, 1)
    y = O.forward(hb, ids, w, w13, s13, w2, s2)
    assert np.all(np.isfinite(y))
    assert 1.0 < np.sqrt(np.mean(y ** 2)) < 1e5


def test_touched_bytes():
    ids = np.array([[0, 1], [1, 2]])
    assert O.touched_bytes(ids, 4, 64, 32) == 3 * (3 * 32 * 64 * 17 // 32)


# ---------------------------------------------------------------------------
# Planted mistakes: every pin above must catch the mistake it is aimed at.
# ---------------------------------------------------------------------------
class _Mutant:
    """A shallow copy of the oracle module namespace with one function replaced."""

    def __init__(self, **repl):
        self.__dict__.update({k: getattr(O, k) for k in dir(O) if not k.startswith("__")})
        self.__dict__.update(repl)
        # functions in the oracle look names up in their own module globals, so
        # re-bind forward/dequant to this namespace where they are replaced
        if "dequant" in repl or "unpack_codes" in repl or "E2M1_TABLE" in repl or "e8m0_value" in repl:
            self.dequant = repl.get("dequant", _rebind(O.dequant, self))
            self.forward = _rebind(O.forward, self)
        if "route" in repl or "silu" in repl or "round_to_bf16" in repl:
            self.forward = _rebind(O.forward, self)


def _rebind(fn, ns):
    import types
    g = dict(fn.__globals__)
    g.update({k: v for k, v in ns.__dict__.items()})
    return types.FunctionType(fn.__code__, g, fn.__name__, fn.__defaults__, fn.__closure__)


def test_pins_catch_planted_mistakes():
    def high_first(p):
        p = np.asarray(p, dtype=np.uint8)
        c = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
        c[..., 0::2] = p >> 4
        c[..., 1::2] = p & 0x0F
        return c

    bad_table = O.E2M1_TABLE.copy()
    bad_table[8:] = -bad_table[:8] + 0.0   # loses the sign of -0
    bad_table2 = O.E2M1_TABLE.copy()
    bad_table2[5], bad_table2[6] = 4.0, 3.0

    def scale_off_by_one(s):
        s = np.asarray(s).astype(np.int64)
        return np.where(s == 255, np.nan, np.ldexp(1.0, s - 126))

    def swapped_route(ids, E):
        rt = O.route(ids, E)
        rt = dict(rt)
        rt["list"] = rt["list"][::-1].copy()   # wrong order inside/among groups
        return rt

    def silu_wrong(z):
        return z / (1.0 + np.exp(z))

    mutants = {
        "high nibble first": (_Mutant(unpack_codes=high_first), check_low_nibble_first),
        "-0 lost": (_Mutant(E2M1_TABLE=bad_table), check_dequant_sweep),
        "codes 5/6 swapped": (_Mutant(E2M1_TABLE=bad_table2), check_golden_table),
        "scale bias 126": (_Mutant(e8m0_value=scale_off_by_one), check_dequant_sweep),
        "route order": (_Mutant(route=swapped_route), check_route),
        "silu sign": (_Mutant(silu=silu_wrong), check_dense_mlp),
    }
    for name, (m, check) in mutants.items():
        assert check(m) != [], f"pin did not catch planted mistake: {name}"


def test_gate_up_swap_caught_by_dense_mlp():
    """An oracle that reads [up; gate] fails the dense-MLP pin."""
    def fwd_swapped(hb, ids, w, w13, s13, w2, s2, intermediate="bf16", tokens=None):
        I = w13.shape[1] // 2
        return O.forward(hb, ids, w, np.concatenate([w13[:, I:], w13[:, :I]], 1),
                         np.concatenate([s13[:, I:], s13[:, :I]], 1), w2, s2,
                         intermediate=intermediate, tokens=tokens)
    m = _Mutant()
    m.forward = fwd_swapped
    assert check_dense_mlp(m) != []


def test_slot_order_weights_caught_by_brute_force():
    def fwd_rev(hb, ids, w, *a, **kw):
        return O.forward(hb, ids, np.ascontiguousarray(w[:, ::-1]), *a, **kw)
    m = _Mutant()
    m.forward = fwd_rev
    assert check_bruteforce_tiny(m) != []
