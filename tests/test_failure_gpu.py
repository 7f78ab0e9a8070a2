"""Failure reporting of the decode kernel's bounded waits, exercised without
faulting or hanging the GPU: the test-only switch mxfp4_moe_test_skip_grid_arrival
keeps one CTA from arriving at the grid barrier between the two phases, so
every CTA's wait on that barrier runs out its bound. The call must report it
(status[2] names the waits, status[3] a CTA), leave the workspace's counters
at zero, and the next call on the same workspace must be correct."""
import pytest
import torch

from mxfp4_mixture_experts_gb300 import synth
from helpers import gate

pytestmark = pytest.mark.gpu

# status[2] bits of the decode kernel's consumer warps (bits 8..15): bit 7 of
# the field marks a consumer failure, bit 1 the phase-2 grid wait, bit 5 the
# combine's grid wait
CONSUMER_FAIL = 128 << 8
GRID_WAIT_PHASE2 = 2 << 8
GRID_WAIT_COMBINE = 32 << 8


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_mixture_experts_gb300 import moe
    return moe


def skip_arrival(moe, cta):
    moe.lib().mxfp4_moe_test_skip_grid_arrival(cta)


@pytest.mark.parametrize("cta", [0, 151])
def test_missing_arrival_is_reported_and_the_workspace_stays_usable(moe, cta):
    shape = synth.custom_shape(K=2880, I=2880, E=16, topk=4)
    case = synth.make_case(shape, 8, seed=90 + cta)
    g = case.to("cuda")
    ws = moe.new_workspace(8, shape.K, shape.I, shape.E, shape.topk)
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    skip_arrival(moe, min(cta, nsm - 1))
    try:
        moe.forward(g.hidden, g.topk_ids, g.topk_weights, g.w13, g.s13, g.w2, g.s2,
                    workspace=ws, status=status, path=1)
        torch.cuda.synchronize()
    finally:
        skip_arrival(moe, -1)
    s2 = int(status[2])
    assert s2 & CONSUMER_FAIL, hex(s2)
    assert s2 & GRID_WAIT_PHASE2, hex(s2)
    assert s2 & GRID_WAIT_COMBINE, hex(s2)
    assert 1 <= int(status[3]) <= nsm
    # the kernel's last CTA reset the grid counters on its way out
    assert torch.count_nonzero(ws[:moe.workspace_zero_bytes()]).item() == 0
    # the same workspace, not cleared by the caller, serves the next call
    status.zero_()
    y = moe.forward(g.hidden, g.topk_ids, g.topk_weights, g.w13, g.s13, g.w2, g.s2,
                    workspace=ws, status=status, path=1)
    torch.cuda.synchronize()
    assert int(status[2]) == 0 and int(status[3]) == 0
    gate(y, case)
