"""Pins of the oracle's MXFP4 encoder (``encode``) to things other than itself
(no GPU needed): exact round trips of representable blocks, blocks whose codes
and scale bytes follow from the rules by hand ("GLM-5.2 and GLM-5.3 (744B) in
MXFP4 on Gaudi 2", What was built, "MXFP4 encoder": the OCP shared exponent
floor(log2(amax)) - 2 and the Quark bump when amax / 2^X >= 7), the pages'
statement that the Quark rule is the more accurate one, and planted mistakes."""
import math
import types

import numpy as np
import torch

from oracle import mxfp4_moe_oracle as O


def bits(vals, cols=32):
    """bf16 bit patterns of a [rows, cols] block list (values exact in bf16)."""
    x = torch.tensor(vals, dtype=torch.float32)
    if x.dim() == 1:
        x = torch.nn.functional.pad(x, (0, cols - x.numel())).unsqueeze(0)
    xb = x.to(torch.bfloat16)
    assert np.array_equal(xb.float().numpy(), x.numpy(), equal_nan=True), \
        "test values must be exact in bf16"
    return xb.view(torch.int16).numpy().view(np.uint16)


def codes_of(packed):
    p = np.asarray(packed, dtype=np.uint8)
    c = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    c[..., 0::2] = p & 0xF
    c[..., 1::2] = p >> 4
    return c


def check_encoder_round_trip(O, seed=51):
    """Blocks of representable values (random codes x 2^(s-127)) come back
    unchanged in value under both rules (their amax / 2^X is 4 or 6, so the
    Quark rule never bumps)."""
    rng = np.random.default_rng(seed)
    packed = rng.integers(0, 256, (6, 64), dtype=np.uint8)
    scale = rng.integers(100, 150, (6, 4), dtype=np.uint8)
    v = O.dequant(packed, scale)
    hb = O.float_to_bf16_bits(v)
    bad = []
    if not np.array_equal(O.bf16_bits_to_float(hb), v):
        bad.append("test values not exact in bf16")
    for rule in ("ocp", "quark"):
        p2, s2 = O.encode(hb, rule)
        back = O.dequant(p2, s2)
        same = (back == v) | (np.isnan(back) & np.isnan(v))
        if not same.all():
            bad.append(f"{rule}: round trip changed {int((~same).sum())} values")
        if not np.array_equal(np.signbit(back), np.signbit(v)):
            bad.append(f"{rule}: round trip changed a sign (-0)")
    return bad


def check_encoder_closed_forms(O):
    bad = []

    def enc(vals, rule="ocp"):
        p, s = O.encode(bits(vals), rule)
        return list(codes_of(p)[0][:len(vals)]), int(s[0, 0])

    # amax 6: X = 0 (byte 127); midpoints round to the even mantissa
    c, s = enc([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -6.0, -0.75])
    if s != 127 or c != [7, 0, 2, 2, 4, 4, 6, 6, 15, 10]:
        bad.append(f"midpoints: byte {s}, codes {c}")
    # just above a midpoint rounds up (0.25 + 2^-9, bf16)
    c, s = enc([6.0, 0.251953125, 0.7578125])
    if c != [7, 1, 2]:
        bad.append(f"above midpoints: {c}")
    # amax 7: OCP keeps X = 0 and saturates 7 to 6; Quark bumps to X = 1
    # (byte 128) and 7 / 2 = 3.5 rounds to 4
    if enc([7.0, 1.0], "ocp") != ([7, 2], 127):
        bad.append(f"amax 7 OCP: {enc([7.0, 1.0], 'ocp')}")
    if enc([7.0, 1.0], "quark") != ([6, 1], 128):
        bad.append(f"amax 7 Quark: {enc([7.0, 1.0], 'quark')}")
    # 6.9375 < 7: no bump
    if enc([6.9375], "quark") != ([7], 127):
        bad.append(f"amax 6.9375 Quark: {enc([6.9375], 'quark')}")
    # amax 1: X = -2 (byte 125), values x4: 4 (code 6), 0.5 (1), -1.5 (8 | 3)
    if enc([1.0, 0.125, -0.375]) != ([6, 1, 11], 125):
        bad.append(f"amax 1: {enc([1.0, 0.125, -0.375])}")
    # zeros: byte 0, codes 0; -0 keeps its sign bit
    if enc([0.0, -0.0]) != ([0, 8], 0):
        bad.append(f"zeros: {enc([0.0, -0.0])}")
    # a subnormal amax (2^-133): X clamped to -127 (byte 0); 2^-6 rounds to 0
    if enc([2.0 ** -133]) != ([0], 0):
        bad.append(f"subnormal amax: {enc([2.0 ** -133])}")
    # the largest bf16 (1.9921875 x 2^127): X = 125; OCP saturates, Quark bumps
    big = 1.9921875 * 2.0 ** 127
    if enc([big], "ocp") != ([7], 252) or enc([big], "quark") != ([6], 253):
        bad.append(f"largest bf16: {enc([big], 'ocp')} {enc([big], 'quark')}")
    # non-finite blocks: byte 255 (NaN), codes 0
    for nf in (float("nan"), float("inf"), float("-inf")):
        if enc([1.0, nf]) != ([0, 0], 255):
            bad.append(f"non-finite {nf}: {enc([1.0, nf])}")
    # blocks are independent: a second block in the row has its own scale
    p, s = O.encode(bits([[6.0] + [0.0] * 31 + [0.5] + [0.0] * 31], cols=64))
    if list(s[0]) != [127, 124]:
        bad.append(f"two blocks: {list(s[0])}")
    return bad


def rel_error(O, x_bits, rule):
    p, s = O.encode(x_bits, rule)
    x = O.bf16_bits_to_float(x_bits)
    return float(np.linalg.norm(O.dequant(p, s) - x) / np.linalg.norm(x))


def check_encoder_quark_more_accurate(O, seed=52):
    """The pages: the Quark rule is the more accurate one (0.1141 vs 0.1171
    relative error on real weights). On N(0, 1) blocks the same order holds,
    with both errors near the MXFP4 level (0.08 .. 0.15)."""
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_normal((64, 256)).astype(np.float32)).to(torch.bfloat16)
    hb = x.view(torch.int16).numpy().view(np.uint16)
    e_ocp, e_quark = rel_error(O, hb, "ocp"), rel_error(O, hb, "quark")
    bad = []
    if not (e_quark < e_ocp):
        bad.append(f"Quark {e_quark} not below OCP {e_ocp}")
    if not (0.08 < e_quark < 0.15 and 0.08 < e_ocp < 0.15):
        bad.append(f"errors out of the MXFP4 range: {e_ocp}, {e_quark}")
    return bad


def test_encoder_round_trip():
    assert check_encoder_round_trip(O) == []


def test_encoder_closed_forms():
    assert check_encoder_closed_forms(O) == []


def test_encoder_quark_more_accurate():
    assert check_encoder_quark_more_accurate(O) == []


def _with(**repl):
    ns = types.SimpleNamespace(**{k: getattr(O, k) for k in dir(O) if not k.startswith("__")})
    for k, v in repl.items():
        setattr(ns, k, v)
    for name in ("encode_block", "encode"):
        if name in repl:
            continue
        fn = getattr(O, name)
        g = dict(fn.__globals__)
        g.update(vars(ns))
        setattr(ns, name, types.FunctionType(fn.__code__, g, fn.__name__, fn.__defaults__,
                                             fn.__closure__))
    if "encode_block" in repl and "encode" not in repl:
        fn = O.encode
        g = dict(fn.__globals__)
        g.update(vars(ns))
        ns.encode = types.FunctionType(fn.__code__, g, fn.__name__, fn.__defaults__, fn.__closure__)
    return ns


def _block_variant(exp_off=2, bump=7.0, ties_up=False, keep_neg_zero=True, saturate=True):
    def encode_block(v, rule):
        v = np.asarray(v, dtype=np.float64)
        if not np.all(np.isfinite(v)):
            return np.zeros(v.shape, dtype=np.uint8), 255
        amax = float(np.max(np.abs(v)))
        if amax == 0.0:
            X = -127
        else:
            _, e = math.frexp(amax)
            X = max(e - 1 - exp_off, -127)
            if rule == "quark" and amax / 2.0 ** X >= bump:
                X += 1
            X = min(X, 127)
        codes = np.empty(v.shape, dtype=np.uint8)
        for i, x in enumerate(v.tolist()):
            q = abs(x) / 2.0 ** X
            best = None
            for c in range(8 if saturate else 7):
                d = abs(q - O.E2M1_TABLE[c])
                tie_ok = (c & 1) == 1 if ties_up else (c & 1) == 0
                if best is None or d < best[0] or (d == best[0] and tie_ok):
                    best = (d, c)
            neg = (x < 0) if not keep_neg_zero else math.copysign(1.0, x) < 0
            codes[i] = best[1] | (8 if neg else 0)
        return codes, X + 127
    return encode_block


def test_encoder_pins_catch_planted_mistakes():
    mutants = {
        "exponent floor(log2) - 1": (_with(encode_block=_block_variant(exp_off=1)),
                                     [check_encoder_closed_forms, check_encoder_round_trip]),
        "Quark threshold 6": (_with(encode_block=_block_variant(bump=6.0)),
                              [check_encoder_closed_forms]),
        "ties to the odd mantissa": (_with(encode_block=_block_variant(ties_up=True)),
                                     [check_encoder_closed_forms]),
        "-0 loses its sign": (_with(encode_block=_block_variant(keep_neg_zero=False)),
                              [check_encoder_closed_forms, check_encoder_round_trip]),
        "no 6 (saturates at 4)": (_with(encode_block=_block_variant(saturate=False)),
                                  [check_encoder_closed_forms, check_encoder_round_trip]),
    }
    for name, (m, checks) in mutants.items():
        for check in checks:
            assert check(m) != [], f"{check.__name__} did not catch planted mistake: {name}"
