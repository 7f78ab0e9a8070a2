"""Test helpers: seeded cases on the device, oracle calls on host copies,
and the comparison metrics (no arithmetic of the layer itself)."""
import numpy as np
import torch

from mxfp4_mixture_experts_gb300 import synth
from oracle import mxfp4_moe_oracle as O

TOL_REL_L2 = 3e-3   # output gate, rel_l2 over the compared rows, vs both oracle modes


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def oracle_rows(case: synth.Case, tokens=None, intermediate="bf16", biases=None):
    """Oracle output rows for `tokens` (all if None). Only the experts those
    tokens use are copied to the host, relabelled 0..n-1 (the oracle is pinned
    invariant under expert relabelling); padding stays -1 and ids >= E stay
    invalid. biases = (b13, b2) selects the gpt-oss form (interleaved w13)."""
    ids = case.topk_ids.cpu().numpy().astype(np.int64)
    tok = np.arange(ids.shape[0]) if tokens is None else np.asarray(tokens)
    sub = ids[tok]
    E = case.shape.E
    valid = (sub >= 0) & (sub < E)
    used = np.unique(sub[valid])
    n_e = max(len(used), 1)
    remap = np.full(E, -1, dtype=np.int64)
    remap[used] = np.arange(len(used))
    sub_ids = np.where(valid, remap[np.clip(sub, 0, E - 1)], np.where(sub >= E, n_e, -1))
    if len(used):
        idx = torch.as_tensor(used, dtype=torch.long)
        pick = lambda w: w.index_select(0, idx.to(w.device)).cpu().numpy()
    else:
        pick = lambda w: np.zeros((1,) + tuple(w.shape[1:]), dtype=np.uint8)
    w13, s13, w2, s2 = pick(case.w13), pick(case.s13), pick(case.w2), pick(case.s2)
    hb = case.hidden.cpu().view(torch.int16).numpy().view(np.uint16)[tok]
    wts = case.topk_weights.cpu().numpy()[tok]
    if biases is not None:
        if len(used):
            b13, b2 = (b.index_select(0, idx.to(b.device)).cpu().numpy() for b in biases)
        else:
            b13 = np.zeros((1,) + tuple(biases[0].shape[1:]), dtype=np.float32)
            b2 = np.zeros((1,) + tuple(biases[1].shape[1:]), dtype=np.float32)
        return O.forward_oai(hb, sub_ids, wts, w13, s13, b13, w2, s2, b2, intermediate=intermediate)
    return O.forward(hb, sub_ids, wts, w13, s13, w2, s2, intermediate=intermediate)


def compare(y_gpu: torch.Tensor, case: synth.Case, tokens=None, with_gap: bool = False,
            biases=None):
    """(rel_l2 vs bf16-intermediate oracle, rel_l2 vs fp32-intermediate, max abs err)
    and, with_gap, the two oracle modes' own rel_l2 distance."""
    got = bf16_to_f64(y_gpu)
    if tokens is not None:
        got = got[np.asarray(tokens)]
    ref_a = oracle_rows(case, tokens, "bf16", biases)
    ref_b = oracle_rows(case, tokens, "fp32", biases)
    out = (rel_l2(got, ref_a), rel_l2(got, ref_b), float(np.abs(got - ref_a).max()))
    return out + (rel_l2(ref_a, ref_b),) if with_gap else out


def gate(y_gpu: torch.Tensor, case: synth.Case, tokens=None, biases=None):
    """The parity gate. Against the pages' reference (fp32 accumulation with a
    bf16 intermediate h): rel_l2 <= TOL_REL_L2. Against the fp32-intermediate
    reading: rel_l2 <= max(TOL_REL_L2, gap + rel_l2 vs the first), gap being the
    distance of the two oracle modes themselves -- the bf16 rounding of h that
    the layer specifies separates them, by more than the tolerance on short
    reductions with few tokens (triangle inequality). Returns the figures."""
    ra, rb, mx, gap = compare(y_gpu, case, tokens, with_gap=True, biases=biases)
    assert ra <= TOL_REL_L2, (ra, rb, mx, gap)
    assert rb <= max(TOL_REL_L2, gap + ra), (ra, rb, mx, gap)
    return ra, rb, mx
