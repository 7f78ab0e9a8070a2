"""Decode path (1..32 tokens) vs the CPU oracle.

Small shapes span several row tiles, a ragged k-step and several stream-K
splits, and are compared on every output element; the four workload shapes
are run at full size (the launch configuration the benchmark times) and
compared on sampled tokens the oracle computes one by one, plus properties
that hold at any size (touched-expert count, finiteness)."""
import numpy as np
import pytest
import torch

from mxfp4_mixture_experts_gb300 import synth
from helpers import compare, gate
from oracle import mxfp4_moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_mixture_experts_gb300 import moe
    return moe


def run(moe, case, path=1, workspace=None, status=None):
    g = case.to("cuda")
    if status is None:
        status = torch.zeros(4, dtype=torch.int32, device="cuda")
    y = moe.forward(g.hidden, g.topk_ids, g.topk_weights, g.w13, g.s13, g.w2, g.s2,
                    workspace=workspace, status=status, path=path)
    torch.cuda.synchronize()
    assert int(status[2]) == 0, "a bounded wait inside a kernel gave up"
    return y


def assert_close(y, case, tokens=None):
    return gate(y, case, tokens)


SMALL = synth.custom_shape(K=320, I=128, E=8, topk=3, name="small")   # 10 k-blocks: ragged stage


@pytest.mark.parametrize("T", [1, 2, 5, 8, 9, 17, 32])
def test_small_all_elements(moe, T):
    case = synth.make_case(SMALL, T, seed=T)
    y = run(moe, case)
    assert_close(y, case)


@pytest.mark.parametrize("K,I,E,k", [(64, 64, 2, 1), (64, 64, 4, 4), (2880, 2880, 3, 2),
                                     (7168, 64, 5, 3), (128, 2048, 6, 2), (576, 192, 3, 3)])
def test_shapes_all_elements(moe, K, I, E, k):
    shape = synth.custom_shape(K=K, I=I, E=E, topk=k)
    case = synth.make_case(shape, 3, seed=K + I)
    assert_close(run(moe, case), case)


def test_hot_routing_many_token_groups(moe):
    """Every token on the same experts: 32 tokens per expert = 4 token groups."""
    case = synth.make_case(SMALL, 32, seed=11)
    ids, w = synth.hot_routing(32, SMALL.topk, SMALL.E, first=2)
    case.topk_ids, case.topk_weights = torch.from_numpy(ids), torch.from_numpy(w)
    assert_close(run(moe, case), case)


def test_rows_beyond_staging_read_from_global(moe):
    """32 tokens on the same 2 experts with K = 7168: each CTA's items need 32
    activation rows of 14 KB, more than shared memory holds, so most B rows are
    read from global memory and converted on the fly."""
    shape = synth.custom_shape(K=7168, I=128, E=4, topk=2)
    case = synth.make_case(shape, 32, seed=20)
    ids, w = synth.hot_routing(32, 2, 4, first=1)
    case.topk_ids, case.topk_weights = torch.from_numpy(ids), torch.from_numpy(w)
    assert_close(run(moe, case), case)


def test_scale_zero_is_two_to_minus_127(moe):
    """E8M0 byte 0 (2^-127, a subnormal factor) in a few blocks: the exact
    general conversion path."""
    case = synth.make_case(SMALL, 3, seed=21)
    e = int(case.topk_ids[0, 0])
    case.s13 = case.s13.clone()
    case.s13[e, :4, 0] = 0
    case.s2 = case.s2.clone()
    case.s2[e, :4, 1] = 0
    assert_close(run(moe, case), case)


def test_padding_invalid_and_duplicates(moe):
    case = synth.make_case(SMALL, 6, seed=12)
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


def test_expert_named_in_every_slot(moe):
    """All 32 tokens name expert 3 in both slots: 64 routes for one expert,
    more than one item's token batch (32), so the expert's items run twice."""
    shape = synth.custom_shape(K=320, I=128, E=8, topk=2)
    case = synth.make_case(shape, 32, seed=22)
    case.topk_ids = torch.full((32, 2), 3, dtype=torch.int32)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    y = run(moe, case, status=status)
    assert int(status[1]) == 1
    assert_close(y, case)


def test_nothing_routed_gives_zeros(moe):
    case = synth.make_case(SMALL, 4, seed=13)
    case.topk_ids = torch.full_like(case.topk_ids, -1)
    y = run(moe, case)
    assert torch.all(y == 0)


def test_wide_scale_range(moe):
    """Scale bytes from 100 to 140 (outputs spanning ~12 orders of magnitude
    per block), so the exact scale multiply matters."""
    case = synth.make_case(SMALL, 5, seed=14)
    gen = torch.Generator().manual_seed(5)
    for name in ("s13", "s2"):
        t = getattr(case, name)
        setattr(case, name, torch.randint(100, 141, t.shape, generator=gen, dtype=torch.uint8))
    assert_close(run(moe, case), case)


def test_scale_255_is_nan(moe):
    case = synth.make_case(SMALL, 2, seed=15)
    e = int(case.topk_ids[0, 0])
    case.s2 = case.s2.clone()
    case.s2[e, 7, 0] = 255           # one w2 block of expert e -> NaN in output row 7
    y = run(moe, case)
    assert torch.isnan(y[0, 7]).item()
    assert not torch.isnan(y[0, 8]).item()


def test_deterministic_and_chain_independent(moe):
    case = synth.make_case(SMALL, 17, seed=16)
    other = synth.make_case(SMALL, 9, seed=17)
    ws = moe.new_workspace(32, SMALL.K, SMALL.I, SMALL.E, SMALL.topk)
    y1 = run(moe, case, workspace=ws).clone()
    run(moe, other, workspace=ws)
    y2 = run(moe, case, workspace=ws).clone()
    y3 = run(moe, case, workspace=ws).clone()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))


def test_negative_control_swapped_gate_up(moe):
    """The test has power: feeding [up; gate] instead of [gate; up] fails the
    gate by far on the workloads' statistics."""
    case = synth.make_case(synth.custom_shape(512, 256, 4, 2), 4, seed=18)
    I = 256
    sw = synth.Case(case.shape, case.T, case.hidden, case.topk_ids, case.topk_weights,
                    torch.cat([case.w13[:, I:], case.w13[:, :I]], 1).contiguous(),
                    torch.cat([case.s13[:, I:], case.s13[:, :I]], 1).contiguous(),
                    case.w2, case.s2, case.logits)
    y = run(moe, sw)
    ra, _, _ = compare(y, case)
    assert ra > 0.1


# full size, the launch configuration the benchmark times; at T = 32 every
# row of the three large shapes is compared, elsewhere the first and last token
FULL = [("single32", 1), ("gptoss128", 1), ("gptoss128", 4), ("gptoss128", 16),
        ("gptoss128", 32), ("glm256", 1), ("glm256", 8), ("glm256", 32), ("widek256", 1),
        ("widek256", 2), ("widek256", 4), ("widek256", 8), ("widek256", 16), ("widek256", 32)]


@pytest.fixture(scope="module")
def full_weights():
    cache = {}

    def get(name):
        if name not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            cache[name] = synth.draw_weights_cuda(synth.SHAPES[name], seed=0, layer=0)
        return cache[name]
    yield get
    cache.clear()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,T", FULL)
def test_full_size_sampled_tokens(moe, full_weights, name, T):
    shape = synth.SHAPES[name]
    rng = np.random.default_rng(0)
    hidden, logits, ids, w = synth.draw_activations(shape, T, np.random.Generator(np.random.PCG64(T)))
    w13, s13, w2, s2 = full_weights(name)
    case = synth.Case(shape, T, hidden, ids, w, w13, s13, w2, s2, logits)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    y = run(moe, case, status=status)
    assert torch.isfinite(y).all()
    rt = O.route(ids.numpy(), shape.E)
    assert int(status[1]) == len(rt["touched"]) and int(status[0]) == 0
    tokens = None if T == 32 else sorted({0, T - 1})
    gate(y, case, tokens, strict=True, label=f"{name} T={T} decode")


def test_wide_activation_range_in_every_block(moe):
    """Hidden values spread over 2^-24 .. 2^24 inside every 32-value block (the
    per-row power-of-two prescale to f16 keeps every element within 2^-31 of
    the row maximum exact)."""
    shape = synth.custom_shape(K=1024, I=256, E=8, topk=2)
    case = synth.make_case(shape, 6, seed=30)
    gen = torch.Generator().manual_seed(9)
    mag = torch.pow(2.0, torch.randint(-24, 25, case.hidden.shape, generator=gen).float())
    case.hidden = (case.hidden.float() * mag).to(torch.bfloat16)
    assert_close(run(moe, case), case)


def test_one_token_one_expert_full_width(moe):
    """One token on one expert with K = I = 2880: the smallest real decode
    call, every CTA's items belong to the same expert."""
    shape = synth.custom_shape(K=2880, I=2880, E=4, topk=1)
    case = synth.make_case(shape, 1, seed=31)
    assert_close(run(moe, case), case)
