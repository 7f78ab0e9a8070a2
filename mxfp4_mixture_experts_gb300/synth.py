"""Seeded synthetic workloads for the routed-expert MXFP4 MoE layer.

This module only *draws* inputs: packed E2M1 bytes, E8M0 scale bytes, bf16
hidden states and router logits, and turns the logits into the routing tensors
(``topk_ids`` int32, ``topk_weights`` fp32) the way each workload describes.
It holds none of the layer's arithmetic (no dequantisation, no projection, no
SwiGLU, no combine), so both the CUDA path and the CPU oracle can consume the
same inputs without sharing any of the computation they are compared on.

Workloads (shapes follow the "MXFP4 MoE decode kernels" page, "Per-call
timings by variant" and "Prefill"; the real checkpoint layers measured there
are not available, so uniform random packed bytes stand in for them):

* ``single32``   K=I=2880, 32 experts, top-4 softmax-over-top-k, T=1.
* ``gptoss128``  K=I=2880, 128 experts, top-4 softmax-over-top-k, T in 1..32.
* ``glm256``     K=6144, I=2048, 256 experts, top-8 sigmoid + renormalise.
* ``widek256``   K=7168, I=2048, 256 experts, top-8 sigmoid + renormalise,
                 with a per-expert logit bias N(0, 0.5) that skews the load.
* ``prefill256`` the glm256 shape at T=8192 (65,536 token-expert pairs).

Generation order for one (workload, T, seed, layer) is fixed: a numpy
``Generator(PCG64(seed * 1000 + layer))`` draws, in order, hidden [T,K] ~
N(0,1) (fp32, then rounded to bf16 by torch's round-to-nearest-even), logits
[T,E] ~ N(0,1) (fp32), the optional bias [E] (sigma x N(0,1)), w13 bytes
[E,2I,K/2] uniform 0..255, w13 scale bytes [E,2I,K/32] uniform 118..124, w2
bytes [E,K,I/2] and w2 scale bytes [E,K,I/32] likewise. Uniform bytes make
each nibble an independent uniform draw over the 16 E2M1 codes.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

SCALE_LO = 118  # E8M0 scale bytes are drawn uniformly from [118, 124] inclusive
SCALE_HI = 124


@dataclasses.dataclass(frozen=True)
class Shape:
    name: str
    K: int
    I: int
    E: int
    topk: int
    scoring: str          # "softmax_topk" or "sigmoid_renorm"
    bias_sigma: float = 0.0
    tokens: tuple = (1,)


SHAPES = {
    "single32": Shape("single32", 2880, 2880, 32, 4, "softmax_topk", 0.0, (1,)),
    "gptoss128": Shape("gptoss128", 2880, 2880, 128, 4, "softmax_topk", 0.0, (1, 4, 16, 32)),
    "glm256": Shape("glm256", 6144, 2048, 256, 8, "sigmoid_renorm", 0.0, (1, 8, 32)),
    "widek256": Shape("widek256", 7168, 2048, 256, 8, "sigmoid_renorm", 0.5, (1, 2, 4, 8, 16, 32)),
    "prefill256": Shape("prefill256", 6144, 2048, 256, 8, "sigmoid_renorm", 0.0, (8192,)),
}


def custom_shape(K: int, I: int, E: int, topk: int, scoring: str = "softmax_topk",
                 bias_sigma: float = 0.0, name: str = "custom") -> Shape:
    """A small shape of the same family, for tests that must finish in seconds."""
    return Shape(name, K, I, E, topk, scoring, bias_sigma, ())


def select_topk(logits: np.ndarray, topk: int, scoring: str,
                bias: Optional[np.ndarray] = None):
    """Router used to *prepare* inputs (the layer itself starts from ids/weights).

    Scores are taken in float64. Selection is a plain top-k over the scores,
    highest first, ties to the lower expert index. ``softmax_topk`` normalises
    a softmax over the chosen k logits; ``sigmoid_renorm`` renormalises the
    chosen sigmoid scores to sum to one. The optional bias is added to the
    logits before scoring, so it moves both the selection and the weights.
    """
    lg = logits.astype(np.float64)
    if bias is not None:
        lg = lg + bias.astype(np.float64)[None, :]
    T, E = lg.shape
    if scoring == "sigmoid_renorm":
        score = 1.0 / (1.0 + np.exp(-lg))
    elif scoring == "softmax_topk":
        score = lg
    else:
        raise ValueError(scoring)
    order = np.argsort(-score, axis=1, kind="stable")[:, :topk]
    ids = order.astype(np.int32)
    chosen = np.take_along_axis(score, order, axis=1)
    if scoring == "softmax_topk":
        z = np.exp(chosen - chosen.max(axis=1, keepdims=True))
        w = z / z.sum(axis=1, keepdims=True)
    else:
        w = chosen / chosen.sum(axis=1, keepdims=True)
    return ids, w.astype(np.float32)


@dataclasses.dataclass
class Case:
    shape: Shape
    T: int
    hidden: torch.Tensor        # [T, K] bf16
    topk_ids: torch.Tensor      # [T, k] int32
    topk_weights: torch.Tensor  # [T, k] fp32
    w13: torch.Tensor           # [E, 2I, K/2] uint8
    s13: torch.Tensor           # [E, 2I, K/32] uint8
    w2: torch.Tensor            # [E, K, I/2] uint8
    s2: torch.Tensor            # [E, K, I/32] uint8
    logits: torch.Tensor        # [T, E] fp32

    def to(self, device) -> "Case":
        f = lambda t: t.to(device, non_blocking=False)
        return Case(self.shape, self.T, f(self.hidden), f(self.topk_ids),
                    f(self.topk_weights), f(self.w13), f(self.s13), f(self.w2),
                    f(self.s2), f(self.logits))

    def numpy(self) -> dict:
        """Host copies in the oracle's input convention (bf16 as raw uint16 bits)."""
        return dict(
            hidden_bits=self.hidden.cpu().view(torch.int16).numpy().view(np.uint16),
            topk_ids=self.topk_ids.cpu().numpy(),
            topk_weights=self.topk_weights.cpu().numpy(),
            w13=self.w13.cpu().numpy(), s13=self.s13.cpu().numpy(),
            w2=self.w2.cpu().numpy(), s2=self.s2.cpu().numpy())


def _rng(seed: int, layer: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed * 1000 + layer))


def draw_weights_cuda(shape: Shape, seed: int, layer: int, device="cuda"):
    """Weights for timing-chain layers, drawn on the device with torch's CUDA
    generator (seeded like the host path). Not parity-checked."""
    K, I, E = shape.K, shape.I, shape.E
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + layer)
    w13 = torch.randint(0, 256, (E, 2 * I, K // 2), generator=g, dtype=torch.uint8, device=device)
    s13 = torch.randint(SCALE_LO, SCALE_HI + 1, (E, 2 * I, K // 32), generator=g,
                        dtype=torch.uint8, device=device)
    w2 = torch.randint(0, 256, (E, K, I // 2), generator=g, dtype=torch.uint8, device=device)
    s2 = torch.randint(SCALE_LO, SCALE_HI + 1, (E, K, I // 32), generator=g,
                       dtype=torch.uint8, device=device)
    return w13, s13, w2, s2


def draw_activations(shape: Shape, T: int, rng: np.random.Generator):
    """hidden (bf16 tensor), logits (fp32), routing ids/weights, in draw order."""
    K, E, k = shape.K, shape.E, shape.topk
    hidden = torch.from_numpy(rng.standard_normal((T, K), dtype=np.float32)).to(torch.bfloat16)
    logits = rng.standard_normal((T, E), dtype=np.float32)
    bias = None
    if shape.bias_sigma > 0:
        bias = (shape.bias_sigma * rng.standard_normal(E, dtype=np.float32)).astype(np.float32)
    ids, w = select_topk(logits, k, shape.scoring, bias)
    return hidden, torch.from_numpy(logits), torch.from_numpy(ids), torch.from_numpy(w)


def make_case(shape, T: int, seed: int = 0, layer: int = 0,
              weights_device: str = "cpu") -> Case:
    """Draw one layer's inputs in the fixed order described in the module doc.

    ``weights_device="cuda"`` draws the four weight tensors on the device
    instead (see ``draw_weights_cuda``); activations and routing still come
    from the host generator.
    """
    if isinstance(shape, str):
        shape = SHAPES[shape]
    K, I, E = shape.K, shape.I, shape.E
    rng = _rng(seed, layer)
    hidden, logits, ids, w = draw_activations(shape, T, rng)
    if weights_device == "cpu":
        u8 = lambda lo, hi, size: torch.from_numpy(rng.integers(lo, hi + 1, size, dtype=np.uint8))
        w13 = u8(0, 255, (E, 2 * I, K // 2))
        s13 = u8(SCALE_LO, SCALE_HI, (E, 2 * I, K // 32))
        w2 = u8(0, 255, (E, K, I // 2))
        s2 = u8(SCALE_LO, SCALE_HI, (E, K, I // 32))
    else:
        w13, s13, w2, s2 = draw_weights_cuda(shape, seed, layer, weights_device)
    return Case(shape, T, hidden, ids, w, w13, s13, w2, s2, logits)


def draw_biases(shape, seed: int = 0, layer: int = 0, sigma: float = 0.5):
    """f32 biases of the gpt-oss form: b13 [E, 2I] (interleaved gate/up row
    order) and b2 [E, K], N(0, sigma^2), from their own seeded generator (so the
    other inputs of a case are drawn exactly as without biases)."""
    if isinstance(shape, str):
        shape = SHAPES[shape]
    rng = np.random.Generator(np.random.PCG64(7919 * seed + 104729 * layer + 17))
    b13 = (sigma * rng.standard_normal((shape.E, 2 * shape.I))).astype(np.float32)
    b2 = (sigma * rng.standard_normal((shape.E, shape.K))).astype(np.float32)
    return torch.from_numpy(b13), torch.from_numpy(b2)


def hot_routing(T: int, topk: int, E: int, first: int = 0):
    """Every token routed to the same k experts (the pages' "all local"/hot case)."""
    ids = np.tile(np.arange(first, first + topk, dtype=np.int32) % E, (T, 1))
    w = np.full((T, topk), 1.0 / topk, dtype=np.float32)
    return ids, w
