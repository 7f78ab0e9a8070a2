"""CPU oracle for the routed-expert MXFP4 mixture-of-experts layer.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import this module. The product
path (the C-ABI library and its Python binding) never calls it, and this module
imports nothing from the product package: it shares no code, table or helper
with the CUDA kernels.

What it computes, step by step, each in the plainest form (float64 numpy, one
library matmul per projection):

1. ``route``      stable counting sort of the routes r = t*k + j by expert.
                  ("MXFP4 MoE decode kernels", Design, "Routing inside the
                  kernel": routes are counting-sorted by local expert; routes
                  to experts that are not present are skipped.)
2. ``dequant``    w = E2M1(nibble) * 2^(E8M0 - 127), nibble 2i = low nibble of
                  byte i, one scale per 32 values along the row.
                  ("GLM-5.2 and GLM-5.3 (744B) in MXFP4 on Gaudi 2", What was
                  built, "Byte-exact repack": OCP MXFP4, E2M1 low nibble first,
                  E8M0 scales, blocks of 32; "MXFP4 MoE decode kernels", The
                  bottleneck and Design, "Read the served layout":
                  w13 u8 [E, 2I, K/2], s13 u8 [E, 2I, K/32], w2 u8 [E, K, I/2],
                  s2 u8 [E, K, I/32].)
3. w13 projection g = W_gate x, u = W_up x with the rows of each expert's w13
   stored as [gate; up] ("GLM-5.2 and GLM-5.3", Why it needed a port, item 1;
   "MXFP4 MoE decode kernels", Beyond gpt-oss: SiLU without bias for [gate; up]
   row layouts).
4. SwiGLU h = silu(g) * u, silu(z) = z / (1 + e^-z), then (default) one
   rounding of h to bf16 ("MXFP4 MoE decode kernels", Parity: the reference is
   CPU fp32 with dequantised weights and a bf16 intermediate).
5. w2 projection o = W2 h.
6. Weighted combine y_t = sum over slots j = 0..k-1 of w_tj * o_(t,j)
   ("MXFP4 MoE decode kernels", Design, Fused epilogues: weighted sum per
   token).

All arithmetic is float64; products of E2M1 values, powers of two and bf16
activations are exact there, so the only roundings are the sums (float64) and
the optional bf16 rounding of h.

``forward_oai`` is the gpt-oss form of the same layer ("MXFP4 MoE decode
kernels", Design, "Read the served layout" and "Fused epilogues"): the w13 rows
of each expert interleave gate and up (row 2i = gate i, row 2i + 1 = up i),
f32 biases are added to g, u and o, the activation is SwiGLU-OAI (gate capped
at 7, up clamped to [-7, 7], gate * sigmoid(1.702 gate) * (up + 1)), and the
w2 bias enters each route's output before the routing weight.
"""
from __future__ import annotations

import math

import numpy as np

# --- E2M1 and E8M0 -----------------------------------------------------------
# The 16 E2M1 codes in code order: bit 3 is the sign, bits 2..1 the exponent
# (bias 1), bit 0 the mantissa; code 1 is the subnormal 0.5.
E2M1_TABLE = np.array([
    +0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
], dtype=np.float64)

SCALE_BLOCK = 32  # values per E8M0 scale along the row


def e8m0_value(scale_bytes) -> np.ndarray:
    """2^(s - 127) as float64; the byte 255 is NaN (OCP MX convention)."""
    s = np.asarray(scale_bytes).astype(np.int64)
    v = np.ldexp(np.ones(s.shape, dtype=np.float64), s - 127)
    return np.where(s == 255, np.nan, v)


def unpack_codes(packed) -> np.ndarray:
    """uint8 [..., C/2] -> codes uint8 [..., C]; value 2i is the low nibble of byte i."""
    p = np.asarray(packed, dtype=np.uint8)
    codes = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    codes[..., 0::2] = p & 0x0F
    codes[..., 1::2] = p >> 4
    return codes


def dequant(packed, scale) -> np.ndarray:
    """Packed rows [..., N, C/2] with scales [..., N, C/32] -> float64 [..., N, C]."""
    codes = unpack_codes(packed)
    vals = E2M1_TABLE[codes]
    factor = e8m0_value(scale)
    if factor.shape[-1] * SCALE_BLOCK != vals.shape[-1]:
        raise ValueError("scale count does not match the row length / 32")
    return vals * np.repeat(factor, SCALE_BLOCK, axis=-1)


# --- bf16 --------------------------------------------------------------------
BF16_MAX = float.fromhex("0x1.fe0000p+127")  # (2 - 2^-7) * 2^127


def bf16_bits_to_float(bits) -> np.ndarray:
    """Raw bf16 bit patterns (uint16) -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits: a finite x = m * 2^e (0.5 <= |m| < 1) is
    rounded to a multiple of 2^(e-8), never finer than the smallest subnormal
    2^-133. Results beyond the largest finite bf16 become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    fin = np.isfinite(x)
    xf = x[fin]
    _, e = np.frexp(xf)
    q = np.maximum(e - 8, -133)
    y = np.ldexp(np.rint(np.ldexp(xf, -q)), q)
    big = np.abs(y) > BF16_MAX
    y[big] = np.copysign(np.inf, y[big])
    out[fin] = y
    return out


def float_to_bf16_bits(x) -> np.ndarray:
    """float64 -> bf16 bit patterns after round_to_bf16 (NaN -> 0x7FC0)."""
    r = round_to_bf16(x)
    bits = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    bits[np.isnan(r)] = 0x7FC0
    return bits


# --- routing -------------------------------------------------------------------
def route(topk_ids, E: int) -> dict:
    """Stable counting sort of routes by expert.

    Route r = t*k + j (row-major over topk_ids). Negative ids are padding and
    skipped; ids >= E are counted as invalid and skipped. Returns count[E],
    offset[E+1] (exclusive prefix sum), list (route ids grouped by expert,
    ascending r inside each group), invalid, and touched (experts with a
    non-zero count, ascending).
    """
    flat = np.asarray(topk_ids).reshape(-1).tolist()
    buckets = [[] for _ in range(E)]
    invalid = 0
    for r, e in enumerate(flat):
        if e < 0:
            continue
        if e >= E:
            invalid += 1
            continue
        buckets[e].append(r)
    count = np.array([len(b) for b in buckets], dtype=np.int64)
    offset = np.zeros(E + 1, dtype=np.int64)
    offset[1:] = np.cumsum(count)
    lst = np.array([r for b in buckets for r in b], dtype=np.int64)
    touched = np.array([e for e in range(E) if buckets[e]], dtype=np.int64)
    return dict(count=count, offset=offset, list=lst, invalid=invalid, touched=touched)


# --- the layer -----------------------------------------------------------------
def silu(z):
    return z / (1.0 + np.exp(-z))


def forward(hidden_bits, topk_ids, topk_weights, w13, s13, w2, s2,
            intermediate: str = "bf16", tokens=None) -> np.ndarray:
    """The MoE layer output y [T', K] in float64 (not rounded to bf16).

    hidden_bits: bf16 bit patterns uint16 [T, K]; topk_ids int [T, k];
    topk_weights float32 [T, k]; w13 uint8 [E, 2I, K/2]; s13 uint8 [E, 2I, K/32];
    w2 uint8 [E, K, I/2]; s2 uint8 [E, K, I/32].
    intermediate: "bf16" rounds h to bf16 once (the pages' reference), "fp32"
    keeps it unrounded. tokens: optional list of token indices; each output
    row depends only on its own token's routes, so a subset is computed the
    same way on fewer routes.
    """
    if intermediate not in ("bf16", "fp32"):
        raise ValueError(intermediate)
    ids = np.asarray(topk_ids)
    wts = np.asarray(topk_weights).astype(np.float64)
    xs = bf16_bits_to_float(hidden_bits)
    if tokens is not None:
        tokens = np.asarray(tokens, dtype=np.int64)
        ids, wts, xs = ids[tokens], wts[tokens], xs[tokens]
    T, k = ids.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    K = w2.shape[1]
    rt = route(ids, E)
    o = np.zeros((T * k, K), dtype=np.float64)
    for e in rt["touched"].tolist():
        r = rt["list"][rt["offset"][e]:rt["offset"][e + 1]]
        x_e = xs[r // k]                              # [M_e, K]
        W13 = dequant(w13[e], s13[e])                 # [2I, K], rows [gate; up]
        g = x_e @ W13[:I].T
        u = x_e @ W13[I:].T
        h = silu(g) * u
        if intermediate == "bf16":
            h = round_to_bf16(h)
        W2 = dequant(w2[e], s2[e])                    # [K, I]
        o[r] = h @ W2.T
    y = np.zeros((T, K), dtype=np.float64)
    E_ok = (ids >= 0) & (ids < E)
    for j in range(k):                                # slot order j = 0 .. k-1
        rows = np.arange(T) * k + j
        contrib = wts[:, j:j + 1] * o[rows]
        y += np.where(E_ok[:, j:j + 1], contrib, 0.0)
    return y


# --- the encoder (bf16 -> E2M1 codes + E8M0 scales) ----------------------------
def encode_block(v, rule: str):
    """One block of 32 values (float64, exact bf16 values) -> (32 codes, scale
    byte). ("GLM-5.2 and GLM-5.3 (744B) in MXFP4 on Gaudi 2", What was built,
    "MXFP4 encoder": the OCP shared exponent X = floor(log2(amax)) - 2; the
    Quark rule raises X by one when amax / 2^X >= 7.)
    X is clamped to [-127, 127] (an all-zero block gets X = -127, byte 0); a
    block with a NaN or infinite value gets byte 255 (NaN) and codes 0. Each
    element: q = v / 2^X, the nearest E2M1 magnitude to |q| found by search
    over the 8 magnitudes (|q| > 6 gives 6), ties to the even mantissa (code
    bit 0 clear), and the sign bit of v (-0 stays -0)."""
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        return np.zeros(v.shape, dtype=np.uint8), 255
    amax = float(np.max(np.abs(v)))
    if amax == 0.0:
        X = -127
    else:
        m, e = math.frexp(amax)            # amax = m 2^e, m in [0.5, 1)
        X = max(e - 1 - 2, -127)           # floor(log2(amax)) - 2
        if rule == "quark" and amax / 2.0 ** X >= 7.0:
            X += 1
        elif rule not in ("ocp", "quark"):
            raise ValueError(rule)
        X = min(X, 127)
    codes = np.empty(v.shape, dtype=np.uint8)
    for i, x in enumerate(v.tolist()):
        q = abs(x) / 2.0 ** X
        best = None
        for c in range(8):
            d = abs(q - E2M1_TABLE[c])
            if best is None or d < best[0] or (d == best[0] and (c & 1) == 0):
                best = (d, c)
        codes[i] = best[1] | (8 if math.copysign(1.0, x) < 0 else 0)
    return codes, X + 127


def encode(hidden_bits, rule: str = "ocp"):
    """bf16 bit patterns uint16 [rows, cols] (cols % 32 == 0) -> packed uint8
    [rows, cols/2] (value 2i in the low nibble of byte i) and scales uint8
    [rows, cols/32], block by block with ``encode_block``."""
    x = bf16_bits_to_float(hidden_bits)
    rows, cols = x.shape
    if cols % SCALE_BLOCK:
        raise ValueError("cols must be a multiple of 32")
    codes = np.empty((rows, cols), dtype=np.uint8)
    scale = np.empty((rows, cols // SCALE_BLOCK), dtype=np.uint8)
    for r in range(rows):
        for b in range(cols // SCALE_BLOCK):
            c, s = encode_block(x[r, SCALE_BLOCK * b:SCALE_BLOCK * (b + 1)], rule)
            codes[r, SCALE_BLOCK * b:SCALE_BLOCK * (b + 1)] = c
            scale[r, b] = s
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, scale


# --- the router (logits -> top-k ids and weights) ------------------------------
def topk_route(logits, topk: int, scoring: str, bias=None, n_group: int = 1,
               topk_group: int = 1, bias_in_weights: bool = True):
    """Router step before routing/permute ("MXFP4 MoE decode kernels",
    Design, "Routing inside the kernel" consumes its top-k ids; the workload
    shapes fix the scoring: top-k softmax for the gpt-oss shapes, sigmoid
    scores renormalised over the chosen k for the GLM shapes, an optional
    per-expert bias added to the logits; "GLM-5.2 and GLM-5.3 (744B) in
    MXFP4 on Gaudi 2", Why it needed a port, item 4, names grouped top-k
    without defining it).

    x = float32(logit + bias) (one float32 addition per element, so both
    sides of a comparison take the selection decision on the same values;
    a NaN ranks as -inf).
    Grouped top-k (n_group > 1): the E experts form n_group equal groups of
    consecutive ids; a group's score is its largest x; only the topk_group
    highest-scoring groups (ties to the lower group index) stay eligible.
    The k largest eligible x in order, ties to the lower expert index
    (sigmoid is increasing, so this is the top-k by sigmoid score).
    Weights in float64 from v = x of the chosen, or, with
    bias_in_weights=False (the bias steers the choice only), from their
    unbiased logits (NaN again as -inf): softmax over the chosen v
    ("softmax_topk"), or sigmoid(v) of the chosen divided by their sum
    ("sigmoid_renorm").
    Returns ids int32 [T, k] and weights float64 [T, k]."""
    raw = np.asarray(logits, dtype=np.float32)
    x = raw
    if bias is not None:
        x = (x + np.asarray(bias, dtype=np.float32)[None, :]).astype(np.float32)
    x = np.where(np.isnan(x), np.float32(-np.inf), x)   # NaN ranks as -inf
    T, E = x.shape
    if E % n_group or not 1 <= topk_group <= n_group:
        raise ValueError("n_group must divide E and 1 <= topk_group <= n_group")
    gs = E // n_group
    ids = np.empty((T, topk), dtype=np.int32)
    for t in range(T):
        eligible = range(E)
        if n_group > 1:
            gscore = [max(float(x[t, e]) for e in range(g * gs, (g + 1) * gs))
                      for g in range(n_group)]
            kept = sorted(range(n_group), key=lambda g: (-gscore[g], g))[:topk_group]
            eligible = [e for e in range(E) if e // gs in kept]
        # stable sort on -x: equal values keep ascending expert order
        order = sorted(eligible, key=lambda e: (-float(x[t, e]), e))
        if len(order) < topk:
            raise ValueError("fewer eligible experts than topk")
        ids[t] = order[:topk]
    v = x if bias_in_weights else np.where(np.isnan(raw), np.float32(-np.inf), raw)
    chosen = np.take_along_axis(v, ids.astype(np.int64), axis=1).astype(np.float64)
    if scoring == "softmax_topk":
        z = np.exp(chosen - chosen.max(axis=1, keepdims=True))
        w = z / z.sum(axis=1, keepdims=True)
    elif scoring == "sigmoid_renorm":
        sc = 1.0 / (1.0 + np.exp(-chosen))
        w = sc / sc.sum(axis=1, keepdims=True)
    else:
        raise ValueError(scoring)
    return ids, w


# --- the gpt-oss form ---------------------------------------------------------
OAI_GATE_CAP = 7.0      # gate capped above at 7
OAI_UP_CLAMP = 7.0      # up clamped to [-7, 7]
OAI_ALPHA = 1.702       # gate * sigmoid(1.702 * gate)


def swiglu_oai(g, u):
    """SwiGLU-OAI ("MXFP4 MoE decode kernels", Design, Fused epilogues):
    gate capped at 7 (no lower bound), up clamped to [-7, 7], then
    gate * sigmoid(1.702 * gate) * (up + 1). NaN inputs stay NaN."""
    g = np.minimum(np.asarray(g, dtype=np.float64), OAI_GATE_CAP)
    u = np.clip(np.asarray(u, dtype=np.float64), -OAI_UP_CLAMP, OAI_UP_CLAMP)
    return g * (1.0 / (1.0 + np.exp(-OAI_ALPHA * g))) * (u + 1.0)


def forward_oai(hidden_bits, topk_ids, topk_weights, w13, s13, b13, w2, s2, b2,
                intermediate: str = "bf16", tokens=None) -> np.ndarray:
    """The gpt-oss MoE layer output y [T', K] in float64 (not rounded to bf16).

    As ``forward``, with w13 rows interleaved per expert (row 2i = gate i,
    row 2i + 1 = up i; "Read the served layout": gate and up rows
    interleaved), b13 float32 [E, 2I] in the same row order, b2 float32 [E, K].
    g = W_gate x + b_gate, u = W_up x + b_up (bias added in fp32 before the
    activation), h = swiglu_oai(g, u) (rounded once to bf16 unless
    intermediate == "fp32"), o = W2 h + b2, and y_t = sum over slots j of
    w_tj * o_(t,j): the routing-weighted bias enters once per route.
    """
    if intermediate not in ("bf16", "fp32"):
        raise ValueError(intermediate)
    ids = np.asarray(topk_ids)
    wts = np.asarray(topk_weights).astype(np.float64)
    xs = bf16_bits_to_float(hidden_bits)
    if tokens is not None:
        tokens = np.asarray(tokens, dtype=np.int64)
        ids, wts, xs = ids[tokens], wts[tokens], xs[tokens]
    T, k = ids.shape
    E, twoI, _ = w13.shape
    K = w2.shape[1]
    bias13 = np.asarray(b13, dtype=np.float64)
    bias2 = np.asarray(b2, dtype=np.float64)
    rt = route(ids, E)
    o = np.zeros((T * k, K), dtype=np.float64)
    for e in rt["touched"].tolist():
        r = rt["list"][rt["offset"][e]:rt["offset"][e + 1]]
        x_e = xs[r // k]                              # [M_e, K]
        W13 = dequant(w13[e], s13[e])                 # [2I, K], rows gate0, up0, gate1, ...
        g = x_e @ W13[0::2].T + bias13[e, 0::2]
        u = x_e @ W13[1::2].T + bias13[e, 1::2]
        h = swiglu_oai(g, u)
        if intermediate == "bf16":
            h = round_to_bf16(h)
        W2 = dequant(w2[e], s2[e])                    # [K, I]
        o[r] = h @ W2.T + bias2[e]
    y = np.zeros((T, K), dtype=np.float64)
    E_ok = (ids >= 0) & (ids < E)
    for j in range(k):                                # slot order j = 0 .. k-1
        rows = np.arange(T) * k + j
        contrib = wts[:, j:j + 1] * o[rows]
        y += np.where(E_ok[:, j:j + 1], contrib, 0.0)
    return y


# --- expert-parallel window and per-route outputs --------------------------------
def forward_window(hidden_bits, topk_ids, topk_weights, w13, s13, w2, s2, expert_base: int = 0,
                   per_route: bool = False, intermediate: str = "bf16"):
    """The layer over a window of experts, optionally per route ("MXFP4 MoE
    decode kernels", Design, "Routing inside the kernel": routes to experts on
    other expert-parallel ranks are skipped; Beyond gpt-oss: mxk_w2xr, a
    per-route w2 output for models that apply a per-route operation before the
    token sum).

    The weights hold the E experts with global ids expert_base .. expert_base
    + E - 1; a route whose id lies outside that window is skipped (it adds
    nothing and is not counted as invalid). per_route=False: y [T, K], the sum
    over the window's routes of w_tj o_(t,j). per_route=True: o [T*k, K], row
    t*k + j = W2[e] h of route (t, j), unweighted, zero for skipped routes."""
    ids = np.asarray(topk_ids).astype(np.int64)
    E = w13.shape[0]
    local = ids - expert_base
    inside = (local >= 0) & (local < E)
    # the window's routes only; everything else becomes padding (-1)
    local_ids = np.where(inside, local, -1).astype(np.int32)
    if not per_route:
        return forward(hidden_bits, local_ids, topk_weights, w13, s13, w2, s2, intermediate)
    T, k = ids.shape
    K = w2.shape[1]
    out = np.zeros((T * k, K), dtype=np.float64)
    for j in range(k):
        # slot j alone with weight 1 is route (t, j)'s output
        ids_j = np.full((T, k), -1, dtype=np.int32)
        ids_j[:, j] = local_ids[:, j]
        ones = np.zeros((T, k), dtype=np.float32)
        ones[:, j] = 1.0
        out[np.arange(T) * k + j] = forward(hidden_bits, ids_j, ones, w13, s13, w2, s2,
                                            intermediate)
    return out


def touched_bytes(topk_ids, E: int, K: int, I: int) -> int:
    """Algorithmic HBM bytes of one call: packed bytes + scales of each touched
    expert read once (3*I*K*(1/2 + 1/32) per expert)."""
    n = len(route(topk_ids, E)["touched"])
    return n * (3 * I * K // 2 + 3 * I * K // 32)
