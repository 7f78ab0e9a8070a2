"""Test helpers: seeded cases on the device, oracle calls on host copies,
and the comparison metrics (no arithmetic of the layer itself)."""
import json
import os

import numpy as np
import torch

from mxfp4_mixture_experts_gb300 import synth
from oracle import mxfp4_moe_oracle as O

TOL_REL_L2 = 3e-3   # output gate, rel_l2 over the compared rows, vs both oracle modes
# Slack over the best bf16 output of the specified computation (below).
IDEAL_SLACK = 1.1


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


def compare(y_gpu: torch.Tensor, case: synth.Case, tokens=None, with_ideal: bool = False,
            biases=None):
    """(rel_l2 vs bf16-intermediate oracle, rel_l2 vs fp32-intermediate, max abs err)
    and, with_ideal, the rel_l2 of the bf16-rounded bf16-intermediate oracle
    output against the fp32-intermediate one."""
    got = bf16_to_f64(y_gpu)
    if tokens is not None:
        got = got[np.asarray(tokens)]
    ref_a = oracle_rows(case, tokens, "bf16", biases)
    ref_b = oracle_rows(case, tokens, "fp32", biases)
    out = (rel_l2(got, ref_a), rel_l2(got, ref_b), float(np.abs(got - ref_a).max()))
    return out + (rel_l2(O.round_to_bf16(ref_a), ref_b),) if with_ideal else out


def log_figures(label: str, **fig):
    """Appends one JSON record of parity figures to $MXFP4_MOE_PARITY_LOG, if set."""
    path = os.environ.get("MXFP4_MOE_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(case=label, **fig)) + "\n")


def gate_figures(ra: float, rb: float, ideal_b: float, strict: bool):
    """The two-mode parity gate on computed figures.

    Mode A, the pages' reference (fp32 accumulation with a bf16 intermediate
    h, "MXFP4 MoE decode kernels", Parity): rel_l2 <= TOL_REL_L2 always.
    Mode B, the unrounded-intermediate reading: rel_l2 <= TOL_REL_L2 as well,
    except on short-reduction shapes where even the best bf16 output of the
    specified computation -- the bf16 rounding of the mode-A result -- lies
    further than that from mode B; there the bound is IDEAL_SLACK times that
    output's own distance. strict (the full-size workload cases) allows no
    such exception."""
    assert ra <= TOL_REL_L2, ("mode A", ra, rb, ideal_b)
    bound_b = TOL_REL_L2 if strict else max(TOL_REL_L2, IDEAL_SLACK * ideal_b)
    assert rb <= bound_b, ("mode B", ra, rb, ideal_b)


def gate(y_gpu: torch.Tensor, case: synth.Case, tokens=None, biases=None, strict: bool = False,
         label: str = ""):
    """The parity gate (gate_figures) against the oracle rows of `tokens`.
    Returns (rel_l2 mode A, rel_l2 mode B, max abs error vs mode A)."""
    ra, rb, mx, ideal_b = compare(y_gpu, case, tokens, with_ideal=True, biases=biases)
    log_figures(label or f"{case.shape.name} T={case.T}", rows=(case.T if tokens is None
                else len(tokens)), rel_l2_a=ra, rel_l2_b=rb, max_abs=mx, ideal_b=ideal_b,
                strict=strict)
    gate_figures(ra, rb, ideal_b, strict)
    return ra, rb, mx
