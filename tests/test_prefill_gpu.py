"""Prefill path (tensor-core grouped GEMMs) vs the CPU oracle.

Small shapes are compared on every output element and span one and several
m-tiles per expert, ragged m- and n-tiles (K % 128 == 64 leaves a half w2
tile), experts with no tokens and the routing edge cases; the many-token
workload shape runs at full size (T = 8192, the launch configuration the
benchmark times) and is compared on sampled tokens the oracle computes one
by one, plus the properties that hold at any size."""
import numpy as np
import pytest
import torch

from mxfp4_mixture_experts_gb300 import synth
from helpers import TOL_REL_L2, compare, gate
from oracle import mxfp4_moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_mixture_experts_gb300 import moe
    return moe


def run(moe, case, path=2, workspace=None, status=None):
    g = case.to("cuda")
    if status is None:
        status = torch.zeros(4, dtype=torch.int32, device="cuda")
    y = moe.forward(g.hidden, g.topk_ids, g.topk_weights, g.w13, g.s13, g.w2, g.s2,
                    workspace=workspace, status=status, path=path)
    torch.cuda.synchronize()
    assert int(status[2]) == 0, f"a bounded wait inside a kernel gave up: {int(status[2]):#x}"
    return y


def assert_close(y, case, tokens=None):
    return gate(y, case, tokens)


SMALL = synth.custom_shape(K=256, I=128, E=8, topk=3, name="psmall")


@pytest.mark.parametrize("K,I,E,k,T", [
    (256, 128, 8, 3, 50),       # one m-tile per expert
    (384, 192, 4, 2, 300),      # ~150 tokens per expert: second m-tile ragged
    (192, 64, 2, 1, 700),       # two m-pairs per expert; K % 128 == 64
    (2880, 2880, 4, 2, 40),     # the 2880-wide expert shape
    (6144, 2048, 3, 2, 33),     # the 6144 x 2048 expert shape
    (128, 256, 64, 2, 40),      # most experts empty
])
def test_shapes_all_elements(moe, K, I, E, k, T):
    shape = synth.custom_shape(K=K, I=I, E=E, topk=k)
    case = synth.make_case(shape, T, seed=K + I + T)
    assert_close(run(moe, case), case)


def test_auto_path_above_32_tokens(moe):
    case = synth.make_case(SMALL, 33, seed=3)
    assert_close(run(moe, case, path=0), case)


@pytest.mark.parametrize("T", [1, 8, 32])
def test_few_tokens_on_prefill_path(moe, T):
    """The prefill path is valid at decode sizes too (one short m-tile)."""
    case = synth.make_case(SMALL, T, seed=40 + T)
    assert_close(run(moe, case), case)


def test_hot_routing_several_m_pairs(moe):
    """Every token on the same experts: 600 tokens each = 3 ragged m-pairs."""
    case = synth.make_case(SMALL, 600, seed=11)
    ids, w = synth.hot_routing(600, SMALL.topk, SMALL.E, first=5)
    case.topk_ids, case.topk_weights = torch.from_numpy(ids), torch.from_numpy(w)
    assert_close(run(moe, case), case)


def test_padding_invalid_and_duplicates(moe):
    case = synth.make_case(SMALL, 70, seed=12)
    ids = case.topk_ids.clone()
    ids[0, 1] = -1          # padding
    ids[1, :] = -1          # a token with no route at all -> zero row
    ids[2, 2] = 99          # invalid: counted, skipped
    ids[3, 1] = ids[3, 0]   # the same expert twice for one token
    case.topk_ids = ids
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    y = run(moe, case, status=status)
    assert int(status[0]) == 1
    assert torch.all(y[1] == 0)
    rt = O.route(ids.numpy(), SMALL.E)
    assert int(status[1]) == len(rt["touched"])
    assert_close(y, case)


def test_nothing_routed_gives_zeros(moe):
    case = synth.make_case(SMALL, 40, seed=13)
    case.topk_ids = torch.full_like(case.topk_ids, -1)
    y = run(moe, case)
    assert torch.all(y == 0)


def test_wide_scale_range(moe):
    case = synth.make_case(SMALL, 45, seed=14)
    gen = torch.Generator().manual_seed(5)
    for name in ("s13", "s2"):
        t = getattr(case, name)
        setattr(case, name, torch.randint(100, 141, t.shape, generator=gen, dtype=torch.uint8))
    assert_close(run(moe, case), case)


def test_scale_255_is_nan(moe):
    case = synth.make_case(SMALL, 40, seed=15)
    e = int(case.topk_ids[0, 0])
    case.s2 = case.s2.clone()
    case.s2[e, 7, 0] = 255           # one w2 block of expert e -> NaN in output column 7
    y = run(moe, case)
    assert torch.isnan(y[0, 7]).item()
    assert not torch.isnan(y[0, 8]).item()


def test_deterministic_and_chain_independent(moe):
    case = synth.make_case(SMALL, 170, seed=16)
    other = synth.make_case(SMALL, 90, seed=17)
    ws = moe.new_workspace(170, SMALL.K, SMALL.I, SMALL.E, SMALL.topk)
    y1 = run(moe, case, workspace=ws).clone()
    run(moe, other, workspace=ws)
    y2 = run(moe, case, workspace=ws).clone()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


def test_many_tiles_per_cta_deterministic(moe):
    """~13 GEMM1 tiles per CTA with only 8 k-stages each: the shared-memory
    rings wrap across many tile boundaries. Three runs must be bit-identical
    (a ring hazard shows up as run-to-run differences) and sampled tokens
    must meet the gate."""
    shape = synth.custom_shape(K=512, I=512, E=128, topk=4, scoring="sigmoid_renorm")
    case = synth.make_case(shape, 16384, seed=21)
    ys = [run(moe, case).clone() for _ in range(3)]
    for y in ys[1:]:
        assert torch.equal(ys[0].view(torch.int16), y.view(torch.int16))
    assert_close(ys[0], case, [0, 1, 5000, 9999, 16383])


def test_decode_and_prefill_agree(moe):
    """Both paths on the same 32 tokens meet the gate against the oracle and
    lie within twice the gate of each other."""
    case = synth.make_case(synth.custom_shape(512, 256, 16, 4), 32, seed=18)
    yd = run(moe, case, path=1).float()
    yp = run(moe, case, path=2).float()
    assert_close(yp, case)
    assert (torch.linalg.norm(yd - yp) / torch.linalg.norm(yd)).item() <= 2 * TOL_REL_L2


def test_negative_control_swapped_gate_up(moe):
    case = synth.make_case(synth.custom_shape(512, 256, 4, 2), 64, seed=19)
    I = 256
    sw = synth.Case(case.shape, case.T, case.hidden, case.topk_ids, case.topk_weights,
                    torch.cat([case.w13[:, I:], case.w13[:, :I]], 1).contiguous(),
                    torch.cat([case.s13[:, I:], case.s13[:, :I]], 1).contiguous(),
                    case.w2, case.s2, case.logits)
    ra, _, _ = compare(run(moe, sw), case)
    assert ra > 0.1


@pytest.mark.parametrize("name,T,tokens", [
    ("prefill256", 8192, tuple(range(0, 8192, 32))),   # 256 tokens over all 256 experts
    ("gptoss128", 2048, (0, 2047)),
])
def test_full_size_sampled_tokens(moe, name, T, tokens):
    shape = synth.SHAPES[name]
    hidden, logits, ids, w = synth.draw_activations(
        shape, T, np.random.Generator(np.random.PCG64(T)))
    w13, s13, w2, s2 = synth.draw_weights_cuda(shape, seed=0, layer=0)
    case = synth.Case(shape, T, hidden, ids, w, w13, s13, w2, s2, logits)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    y = run(moe, case, status=status)
    assert torch.isfinite(y).all()
    rt = O.route(ids.numpy(), shape.E)
    assert int(status[1]) == len(rt["touched"]) and int(status[0]) == 0
    gate(y, case, list(tokens), strict=True, label=f"{name} T={T} prefill")
    del case, w13, s13, w2, s2
    torch.cuda.empty_cache()
