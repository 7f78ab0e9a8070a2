"""Guard bands around the output and the workspace (the substitute for a
memory sanitizer): both paths at full size write nothing outside `out` and
the workspace, leave their inputs unmodified and leave the workspace's
bookkeeping bytes at zero."""
import numpy as np
import pytest
import torch

from mxfp4_mixture_experts_gb300 import synth

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes of guard band on each side (keeps 256-byte alignment)
PATTERN = 0xA5


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_mixture_experts_gb300 import moe
    return moe


def guarded(nbytes: int):
    buf = torch.full((nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
    return buf, buf[GUARD:GUARD + nbytes]


def guards_intact(buf) -> bool:
    return bool((buf[:GUARD] == PATTERN).all() and (buf[-GUARD:] == PATTERN).all())


@pytest.mark.parametrize("name,T,path", [("gptoss128", 32, 1), ("glm256", 32, 1),
                                         ("widek256", 1, 1), ("gptoss128", 2048, 2)])
def test_writes_stay_inside_out_and_workspace(moe, name, T, path):
    shape = synth.SHAPES[name]
    hidden, logits, ids, w = synth.draw_activations(
        shape, T, np.random.Generator(np.random.PCG64(77 + T)))
    w13, s13, w2, s2 = synth.draw_weights_cuda(shape, seed=0, layer=0)
    x, ids, w = hidden.cuda(), ids.cuda(), w.cuda()
    keep = [t.clone() for t in (x, ids, w, s13, s2)]
    w13_sum, w2_sum = int(w13.sum(dtype=torch.int64)), int(w2.sum(dtype=torch.int64))
    out_buf, out_bytes = guarded(T * shape.K * 2)
    out = out_bytes.view(torch.bfloat16).view(T, shape.K)
    n_ws = moe.workspace_size(T, shape.K, shape.I, shape.E, shape.topk)
    ws_buf, ws = guarded(n_ws)
    ws.zero_()
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    for _ in range(2):
        moe.forward(x, ids, w, w13, s13, w2, s2, out=out, workspace=ws, status=status, path=path)
    torch.cuda.synchronize()
    assert int(status[2]) == 0
    assert guards_intact(out_buf), "a write landed next to the output"
    assert guards_intact(ws_buf), "a write landed next to the workspace"
    assert torch.count_nonzero(ws[:moe.workspace_zero_bytes()]).item() == 0, \
        "bookkeeping bytes not left at zero"
    assert torch.isfinite(out.float()).all()
    for a, b in zip(keep, (x, ids, w, s13, s2)):
        assert torch.equal(a, b), "an input was modified"
    assert int(w13.sum(dtype=torch.int64)) == w13_sum and int(w2.sum(dtype=torch.int64)) == w2_sum
    del w13, s13, w2, s2, ws_buf, keep
    torch.cuda.empty_cache()
