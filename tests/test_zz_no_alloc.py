"""mxfp4_moe_forward_noalloc, the forward call for callers that cannot
allocate device memory (it runs on a fixed device array compiled into the
library), must give the same layer output as mxfp4_moe_forward, bit for bit:
both run the same deterministic kernels. Called through the C ABI, two calls
in a row on each path, and once more after a call whose bounded waits ran
out (the array's counters must be left at zero for the next call). Kept in a
file of its own that pytest collects last."""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_mixture_experts_gb300 import moe
    f = moe.lib().mxfp4_moe_forward_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, i32, vp]
    f.restype = i32
    return moe, f


def _call(moe, f, case, path, status):
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    s = case.shape
    out = torch.full((case.T, s.K), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = f(P(case.hidden), P(case.topk_ids), P(case.topk_weights), P(case.w13), P(case.s13),
           P(case.w2), P(case.s2), case.T, s.K, s.I, s.E, s.topk, P(out), P(status), path,
           stream)
    assert rc == 0, moe.strerror(rc)
    torch.cuda.synchronize()
    return out


def _same(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("path", [1, 2])
def test_noalloc_matches_forward_two_calls_in_a_row(path):
    moe, f = _noalloc_fn()
    from mxfp4_mixture_experts_gb300 import synth
    shapes = [synth.custom_shape(K=2880, I=2880, E=16, topk=4, name="a"),
              synth.custom_shape(K=1024, I=512, E=8, topk=2, name="b")]
    T0 = 5 if path == 1 else 40
    for call, shape in enumerate(shapes):
        case = synth.make_case(shape, T=T0 + call, seed=40 + call).to("cuda")
        ref = moe.forward(case.hidden, case.topk_ids, case.topk_weights, case.w13, case.s13,
                          case.w2, case.s2, path=path)
        status = torch.zeros(4, dtype=torch.int32, device="cuda")
        out = _call(moe, f, case, path, status)
        assert int(status[2]) == 0
        assert _same(out, ref)


def test_noalloc_after_a_call_whose_waits_ran_out():
    moe, f = _noalloc_fn()
    from mxfp4_mixture_experts_gb300 import synth
    shape = synth.custom_shape(K=2880, I=2880, E=16, topk=4, name="c")
    case = synth.make_case(shape, T=7, seed=45).to("cuda")
    ref = moe.forward(case.hidden, case.topk_ids, case.topk_weights, case.w13, case.s13,
                      case.w2, case.s2, path=1)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    moe.lib().mxfp4_moe_test_skip_grid_arrival(3)
    try:
        _call(moe, f, case, 1, status)
    finally:
        moe.lib().mxfp4_moe_test_skip_grid_arrival(-1)
    assert int(status[2]) != 0, "the missing arrival was not reported"
    # a stale grid counter would let the next call pass its barriers early
    for _ in range(2):
        status.zero_()
        out = _call(moe, f, case, 1, status)
        assert int(status[2]) == 0
        assert _same(out, ref)


def test_noalloc_rejects_sizes_beyond_its_array():
    moe, f = _noalloc_fn()
    nul = ctypes.c_void_p(0x1000)
    # 8192 tokens of the glm256 shape need far more than the fixed array
    rc = f(nul, nul, nul, nul, nul, nul, nul, 8192, 6144, 2048, 256, 8, nul, None, 2, None)
    assert rc == moe.ERR_WORKSPACE
