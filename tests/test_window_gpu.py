"""The expert-window and per-route forms (mxfp4_moe_forward_window) on both
paths vs the CPU oracle's forward_window ("MXFP4 MoE decode kernels", Design,
"Routing inside the kernel": routes of other expert-parallel ranks skipped;
Beyond gpt-oss: a per-route w2 output)."""
import numpy as np
import pytest
import torch

from mxfp4_mixture_experts_gb300 import synth
from helpers import TOL_REL_L2, bf16_to_f64, gate_figures, rel_l2
from oracle import mxfp4_moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_mixture_experts_gb300 import moe
    return moe


def window_case(seed, T, K=320, I=128, E=8, k=3):
    shape = synth.custom_shape(K=K, I=I, E=E, topk=k)
    return synth.make_case(shape, T, seed=seed)


def run_window(moe, case, lo, hi, per_route, path):
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    sl = slice(lo, hi)
    y = moe.forward_window(case.hidden.cuda(), case.topk_ids.cuda(),
                           None if per_route else case.topk_weights.cuda(),
                           case.w13[sl].contiguous().cuda(), case.s13[sl].contiguous().cuda(),
                           case.w2[sl].contiguous().cuda(), case.s2[sl].contiguous().cuda(),
                           expert_base=lo, per_route=per_route, status=status, path=path)
    torch.cuda.synchronize()
    assert int(status[2]) == 0, "a bounded wait inside a kernel gave up"
    assert int(status[0]) == 0, "ids outside the window counted as invalid"
    return y


def oracle_window(case, lo, hi, per_route, mode):
    hb = case.hidden.view(torch.int16).numpy().view(np.uint16)
    sl = slice(lo, hi)
    return O.forward_window(hb, case.topk_ids.numpy(), case.topk_weights.numpy(),
                            case.w13[sl].numpy(), case.s13[sl].numpy(), case.w2[sl].numpy(),
                            case.s2[sl].numpy(), lo, per_route, mode)


def gate_window(y, case, lo, hi, per_route):
    got = bf16_to_f64(y)
    ra_ref = oracle_window(case, lo, hi, per_route, "bf16")
    rb_ref = oracle_window(case, lo, hi, per_route, "fp32")
    ra, rb = rel_l2(got, ra_ref), rel_l2(got, rb_ref)
    gate_figures(ra, rb, rel_l2(O.round_to_bf16(ra_ref), rb_ref), strict=False)
    return got, ra_ref


@pytest.mark.parametrize("path,T", [(1, 9), (1, 32), (2, 60)])
def test_windows_match_the_oracle_and_sum_to_the_layer(moe, path, T):
    case = window_case(300 + T, T)
    ya = run_window(moe, case, 0, 3, False, path)
    yb = run_window(moe, case, 3, 8, False, path)
    gate_window(ya, case, 0, 3, False)
    gate_window(yb, case, 3, 8, False)
    full = O.forward(case.hidden.view(torch.int16).numpy().view(np.uint16), case.topk_ids.numpy(),
                     case.topk_weights.numpy(), case.w13.numpy(), case.s13.numpy(),
                     case.w2.numpy(), case.s2.numpy())
    assert rel_l2(bf16_to_f64(ya) + bf16_to_f64(yb), full) <= 2 * TOL_REL_L2


@pytest.mark.parametrize("path,T", [(1, 7), (1, 32), (2, 50)])
def test_per_route_rows(moe, path, T):
    case = window_case(400 + T, T)
    ids = case.topk_ids.clone()
    ids[1, 0] = -1            # padding
    ids[2, 2] = 5             # outside the window [0, 5) below: skipped
    case.topk_ids = ids
    y = run_window(moe, case, 0, 5, True, path)
    assert tuple(y.shape) == (T * 3, 320)
    got, ref = gate_window(y, case, 0, 5, True)
    skipped = [(t, j) for t in range(T) for j in range(3)
               if not (0 <= int(ids[t, j]) < 5)]
    assert skipped
    for t, j in skipped:
        assert np.all(got[t * 3 + j] == 0) and np.all(ref[t * 3 + j] == 0)


def test_window_of_all_experts_is_the_layer(moe):
    case = window_case(500, 12)
    y = run_window(moe, case, 0, 8, False, 1)
    yf = moe.forward(case.hidden.cuda(), case.topk_ids.cuda(), case.topk_weights.cuda(),
                     case.w13.cuda(), case.s13.cuda(), case.w2.cuda(), case.s2.cuda(), path=1)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), yf.view(torch.int16))
