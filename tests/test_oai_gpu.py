"""The gpt-oss form of the layer ("MXFP4 MoE decode kernels", Design:
interleaved gate/up rows, f32 biases, SwiGLU-OAI, routing-weighted w2 bias per
route) on the decode and prefill paths vs the CPU oracle's forward_oai.

Small shapes span several row tiles, a ragged last stage, several token groups
and rows read from the global scratch (decode), one and several m-tiles per
expert and a half w2 tile (prefill), compared on every output element; the
gpt-oss-120b layer (K = I = 2880, 128 experts, top-4) runs at full size on
sampled tokens on both paths."""
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


def run_oai(moe, case, biases, status=None):
    g = case.to("cuda")
    b13, b2 = (b.to("cuda") for b in biases)
    if status is None:
        status = torch.zeros(4, dtype=torch.int32, device="cuda")
    y = moe.forward_oai(g.hidden, g.topk_ids, g.topk_weights, g.w13, g.s13, b13, g.w2, g.s2, b2,
                        status=status)
    torch.cuda.synchronize()
    assert int(status[2]) == 0, "a bounded wait inside a kernel gave up"
    return y


SMALL = synth.custom_shape(K=320, I=128, E=8, topk=3, name="small")


@pytest.mark.parametrize("T", [1, 5, 17, 32])
def test_oai_small_all_elements(moe, T):
    case = synth.make_case(SMALL, T, seed=200 + T)
    b = synth.draw_biases(SMALL, seed=T)
    gate(run_oai(moe, case, b), case, biases=b)


@pytest.mark.parametrize("K,I,E,k", [(64, 64, 2, 1), (2880, 2880, 3, 2), (7168, 64, 5, 3),
                                     (128, 2048, 6, 2), (576, 192, 3, 3)])
def test_oai_shapes_all_elements(moe, K, I, E, k):
    shape = synth.custom_shape(K=K, I=I, E=E, topk=k)
    case = synth.make_case(shape, 3, seed=K + 2 * I)
    b = synth.draw_biases(shape, seed=K)
    gate(run_oai(moe, case, b), case, biases=b)


def test_oai_many_token_groups(moe):
    """Every token on the same experts: 32 tokens per expert = 4 token groups."""
    case = synth.make_case(SMALL, 32, seed=211)
    ids, w = synth.hot_routing(32, SMALL.topk, SMALL.E, first=2)
    case.topk_ids, case.topk_weights = torch.from_numpy(ids), torch.from_numpy(w)
    b = synth.draw_biases(SMALL, seed=11)
    gate(run_oai(moe, case, b), case, biases=b)


def test_oai_rows_beyond_staging(moe):
    """K = 7168, 32 tokens on 2 experts: most activation rows come from the f16
    scratch in global memory."""
    shape = synth.custom_shape(K=7168, I=128, E=4, topk=2)
    case = synth.make_case(shape, 32, seed=220)
    ids, w = synth.hot_routing(32, 2, 4, first=1)
    case.topk_ids, case.topk_weights = torch.from_numpy(ids), torch.from_numpy(w)
    b = synth.draw_biases(shape, seed=20)
    gate(run_oai(moe, case, b), case, biases=b)


def test_oai_zero_weights_give_the_weighted_w2_bias(moe):
    """All weight codes 0: each route's output is its expert's b2, so y_t is
    the routing-weighted sum of b2 rows (a padding slot adds nothing)."""
    case = synth.make_case(SMALL, 6, seed=230)
    case.w13 = torch.zeros_like(case.w13)
    case.w2 = torch.zeros_like(case.w2)
    ids = case.topk_ids.clone()
    ids[2, 1] = -1
    case.topk_ids = ids
    b13, b2 = synth.draw_biases(SMALL, seed=30)
    y = run_oai(moe, case, (b13, b2)).float().cpu().numpy()
    want = np.zeros((6, SMALL.K))
    for t in range(6):
        for j in range(SMALL.topk):
            e = int(ids[t, j])
            if e >= 0:
                want[t] += float(case.topk_weights[t, j]) * b2[e].double().numpy()
    assert np.abs(y - want).max() <= 2.0 ** -7 * np.abs(want).max()
    gate(torch.from_numpy(y).to(torch.bfloat16), case, biases=(b13, b2))


def test_oai_clamps_reached(moe):
    """The synthetic weights drive gates past the cap and ups past the clamp
    (checked on the host), and the outputs still match the oracle."""
    case = synth.make_case(synth.custom_shape(K=2880, I=256, E=4, topk=2), 4, seed=240)
    x = O.bf16_bits_to_float(case.hidden.view(torch.int16).numpy().view(np.uint16))
    e = int(case.topk_ids[0, 0])
    W = O.dequant(case.w13[e].numpy(), case.s13[e].numpy())
    g, u = x[0] @ W[0::2].T, x[0] @ W[1::2].T
    assert (g > 7).any() and (np.abs(u) > 7).any()
    b = synth.draw_biases(case.shape, seed=40)
    gate(run_oai(moe, case, b), case, biases=b)


def test_oai_nan_scale_reaches_the_routed_tokens(moe):
    """Scale byte 255 (NaN) in one gate-row block of expert e: h of that pair
    is NaN, so every output of the tokens routed to e is NaN and the others
    stay finite, as in the oracle."""
    case = synth.make_case(SMALL, 6, seed=250)
    e = int(case.topk_ids[0, 0])
    case.s13 = case.s13.clone()
    case.s13[e, 2 * 3, 1] = 255              # gate row of pair 3, block 1
    b = synth.draw_biases(SMALL, seed=50)
    y = run_oai(moe, case, b).float().cpu().numpy()
    hb = case.hidden.view(torch.int16).numpy().view(np.uint16)
    ref = O.forward_oai(hb, case.topk_ids.numpy(), case.topk_weights.numpy(), case.w13.numpy(),
                        case.s13.numpy(), b[0].numpy(), case.w2.numpy(), case.s2.numpy(),
                        b[1].numpy())
    assert np.array_equal(np.isnan(y), np.isnan(ref))
    assert np.isnan(y[0]).all()
    ok = np.where(~np.isnan(ref).any(axis=1))[0]
    assert len(ok) > 0
    ra, _, _ = compare(torch.from_numpy(y).to(torch.bfloat16), case, tokens=ok, biases=b)
    assert ra <= 3e-3


def test_oai_negative_control_blocked_rows(moe):
    """The test has power: feeding [gate; up] blocks to the interleaved form
    fails the gate by far."""
    shape = synth.custom_shape(K=512, I=256, E=4, topk=2)
    case = synth.make_case(shape, 4, seed=260)
    b = synth.draw_biases(shape, seed=60)
    blocked = synth.Case(case.shape, case.T, case.hidden, case.topk_ids, case.topk_weights,
                         torch.cat([case.w13[:, 0::2], case.w13[:, 1::2]], 1).contiguous(),
                         torch.cat([case.s13[:, 0::2], case.s13[:, 1::2]], 1).contiguous(),
                         case.w2, case.s2, case.logits)
    y = run_oai(moe, blocked, b)
    ra, _, _ = compare(y, case, biases=b)
    assert ra > 0.1


@pytest.mark.parametrize("T", [1, 32])
def test_oai_gptoss128_full_size_sampled_tokens(moe, T):
    shape = synth.SHAPES["gptoss128"]
    hidden, logits, ids, w = synth.draw_activations(shape, T, np.random.Generator(np.random.PCG64(T)))
    w13, s13, w2, s2 = synth.draw_weights_cuda(shape, seed=0, layer=0)
    case = synth.Case(shape, T, hidden, ids, w, w13, s13, w2, s2, logits)
    b = synth.draw_biases(shape, seed=0)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    y = run_oai(moe, case, b, status=status)
    assert torch.isfinite(y).all()
    rt = O.route(ids.numpy(), shape.E)
    assert int(status[1]) == len(rt["touched"])
    gate(y, case, sorted({0, T - 1}), biases=b, strict=True)
    del w13, s13, w2, s2
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# the gpt-oss form on the prefill path (tensor-core grouped GEMMs)
# ---------------------------------------------------------------------------
def run_oai_path(moe, case, biases, path):
    g = case.to("cuda")
    b13, b2 = (b.to("cuda") for b in biases)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    y = moe.forward_oai(g.hidden, g.topk_ids, g.topk_weights, g.w13, g.s13, b13, g.w2, g.s2, b2,
                        status=status, path=path)
    torch.cuda.synchronize()
    assert int(status[2]) == 0, f"a bounded wait inside a kernel gave up: {int(status[2]):#x}"
    return y


@pytest.mark.parametrize("K,I,E,k,T", [
    (256, 128, 8, 3, 50),       # one m-tile per expert
    (384, 192, 4, 2, 300),      # a ragged second m-tile
    (192, 64, 2, 1, 700),       # K % 128 == 64: a half w2 tile
    (2880, 2880, 4, 2, 40),     # the gpt-oss-120b expert shape
])
def test_oai_prefill_all_elements(moe, K, I, E, k, T):
    shape = synth.custom_shape(K=K, I=I, E=E, topk=k)
    case = synth.make_case(shape, T, seed=3 * K + I + T)
    b = synth.draw_biases(shape, seed=K + T)
    gate(run_oai_path(moe, case, b, 2), case, biases=b)


def test_oai_prefill_and_decode_agree(moe):
    """Both paths on the same 32 tokens meet the gate against the oracle and
    lie within twice the gate of each other."""
    shape = synth.custom_shape(512, 256, 16, 4)
    case = synth.make_case(shape, 32, seed=270)
    b = synth.draw_biases(shape, seed=70)
    yd = run_oai_path(moe, case, b, 1).float()
    yp = run_oai_path(moe, case, b, 2)
    gate(yp, case, biases=b)
    yp = yp.float()
    assert (torch.linalg.norm(yd - yp) / torch.linalg.norm(yd)).item() <= 2 * 3e-3


def test_oai_auto_path_above_32_tokens(moe):
    shape = synth.custom_shape(K=256, I=128, E=8, topk=3)
    case = synth.make_case(shape, 40, seed=280)
    b = synth.draw_biases(shape, seed=80)
    gate(run_oai_path(moe, case, b, 0), case, biases=b)


def test_oai_prefill_gptoss128_full_size_sampled_tokens(moe):
    shape = synth.SHAPES["gptoss128"]
    T = 2048
    hidden, logits, ids, w = synth.draw_activations(shape, T, np.random.Generator(np.random.PCG64(T)))
    w13, s13, w2, s2 = synth.draw_weights_cuda(shape, seed=0, layer=0)
    case = synth.Case(shape, T, hidden, ids, w, w13, s13, w2, s2, logits)
    b = synth.draw_biases(shape, seed=0)
    y = run_oai_path(moe, case, b, 0)
    assert torch.isfinite(y).all()
    gate(y, case, [0, 1023, 2047], biases=b, strict=True)
    del case, w13, s13, w2, s2
    torch.cuda.empty_cache()
