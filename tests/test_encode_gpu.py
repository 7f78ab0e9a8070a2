"""The MXFP4 encoder vs the CPU oracle's encode: packed bytes and scale bytes
bit-exact under both exponent rules, on random blocks spanning the whole bf16
range, on blocks whose codes follow from the rules by hand, on a value round
trip through the library's dequant, and on a full gpt-oss-120b w13 expert."""
import numpy as np
import pytest
import torch

from oracle import mxfp4_moe_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_mixture_experts_gb300 import moe
    return moe


def bits_of(x: torch.Tensor) -> np.ndarray:
    return x.cpu().view(torch.int16).numpy().view(np.uint16)


def check(moe, x: torch.Tensor, rule: str, rows=None):
    p, s = moe.encode(x.cuda(), rule)
    torch.cuda.synchronize()
    hb = bits_of(x)
    if rows is not None:
        hb = hb[rows]
        p, s = p[rows], s[rows]
    rp, rs = O.encode(hb, rule)
    gp, gs = p.cpu().numpy(), s.cpu().numpy()
    assert np.array_equal(gs, rs), np.argwhere(gs != rs)[:5]
    assert np.array_equal(gp, rp), np.argwhere(gp != rp)[:5]


@pytest.mark.parametrize("rule", ["ocp", "quark"])
def test_encode_random_blocks_all_magnitudes(moe, rule):
    g = torch.Generator().manual_seed(61)
    x = torch.randn(48, 512, generator=g)
    # each 32-value block at its own power of two, 2^-140 .. 2^120
    e = torch.randint(-140, 121, (48, 16), generator=g).float()
    x = (x * torch.pow(2.0, e).repeat_interleave(32, dim=1)).to(torch.bfloat16)
    check(moe, x, rule)


@pytest.mark.parametrize("rule", ["ocp", "quark"])
def test_encode_special_blocks(moe, rule):
    blocks = [
        [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -6.0, -0.75],   # midpoints
        [6.0, 0.251953125, 0.7578125],                               # just above
        [7.0, 1.0], [6.9375, -3.0], [1.0, 0.125, -0.375],
        [0.0, -0.0], [], [2.0 ** -133, -2.0 ** -130],                # zeros, subnormals
        [1.9921875 * 2.0 ** 127, -1.0],                              # the largest bf16
        [1.0, float("nan")], [float("inf"), 2.0], [-float("inf")],   # non-finite
        [-1e-30, 1e30],                                              # sign of a flushed value
    ]
    x = torch.zeros(len(blocks), 32)
    for r, b in enumerate(blocks):
        if b:
            x[r, :len(b)] = torch.tensor(b)
    check(moe, x.to(torch.bfloat16), rule)


def test_encode_round_trip_through_dequant(moe):
    """Representable values (random codes and scales, dequantised by the
    library) encode back to the same values."""
    g = torch.Generator().manual_seed(62)
    packed = torch.randint(0, 256, (32, 256), generator=g, dtype=torch.uint8).cuda()
    scale = torch.randint(90, 160, (32, 16), generator=g, dtype=torch.uint8).cuda()
    x = moe.dequant(packed, scale)
    for rule in ("ocp", "quark"):
        p, s = moe.encode(x, rule)
        y = moe.dequant(p, s)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), x.view(torch.int16))


def test_encode_gptoss_expert_full_size(moe):
    """One gpt-oss-120b w13 expert ([2I, K] = [5760, 2880], N(0, 0.02)),
    sampled rows vs the oracle, both rules."""
    g = torch.Generator().manual_seed(63)
    x = (0.02 * torch.randn(5760, 2880, generator=g)).to(torch.bfloat16)
    for rule in ("ocp", "quark"):
        check(moe, x, rule, rows=[0, 1, 2879, 2880, 5759])
