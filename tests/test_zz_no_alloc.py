"""mxfp4_moe_forward_noalloc, the forward call for callers that cannot
allocate device memory (it runs on a fixed device array compiled into the
library), must give the same layer output as mxfp4_moe_forward. Called
through the C ABI, twice in a row. Kept in a file of its own that pytest
collects last."""
import ctypes

import pytest
import torch

from helpers import TOL_REL_L2, bf16_to_f64, rel_l2

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


def test_noalloc_matches_forward_two_calls_in_a_row():
    moe, f = _noalloc_fn()
    from mxfp4_mixture_experts_gb300 import synth
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    shapes = [synth.custom_shape(K=2880, I=2880, E=16, topk=4, name="a"),
              synth.custom_shape(K=1024, I=512, E=8, topk=2, name="b")]
    for call, shape in enumerate(shapes):
        case = synth.make_case(shape, T=5 + call, seed=40 + call).to("cuda")
        ref = moe.forward(case.hidden, case.topk_ids, case.topk_weights, case.w13, case.s13,
                          case.w2, case.s2, path=1)
        out = torch.full_like(ref, float("nan"))
        status = torch.zeros(4, dtype=torch.int32, device="cuda")
        K, I, E, k = shape.K, shape.I, shape.E, shape.topk
        rc = f(P(case.hidden), P(case.topk_ids), P(case.topk_weights), P(case.w13),
               P(case.s13), P(case.w2), P(case.s2), case.T, K, I, E, k, P(out), P(status), 1,
               stream)
        assert rc == 0, moe.strerror(rc)
        torch.cuda.synchronize()
        assert int(status[2]) == 0
        assert rel_l2(bf16_to_f64(out), bf16_to_f64(ref)) <= TOL_REL_L2


def test_noalloc_rejects_sizes_beyond_its_array():
    moe, f = _noalloc_fn()
    from mxfp4_mixture_experts_gb300 import moe as m
    nul = ctypes.c_void_p(0x1000)
    # 8192 tokens of the glm256 shape need far more than the fixed array
    rc = f(nul, nul, nul, nul, nul, nul, nul, 8192, 6144, 2048, 256, 8, nul, None, 2, None)
    assert rc == m.ERR_WORKSPACE
