"""Weight dequantisation of both paths vs the oracle, bit for bit: the decode
kernels' conversion (hardware E2M1 -> f16, fp32 scale multiply) and the
prefill GEMM's operand-A construction (E2M1 fields placed in bf16 bits, exact
bf16 multiplies -- the device routine that feeds the GEMM's tensor memory),
each exported through mxfp4_moe_dequant_form. NaN is compared as NaN."""
import numpy as np
import pytest
import torch

from mxfp4_mixture_experts_gb300 import synth
from oracle import mxfp4_moe_oracle as O

pytestmark = pytest.mark.gpu

FORMS = ["decode", "prefill"]


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_mixture_experts_gb300 import moe
    return moe


def bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def check_bits(got_bits, ref_vals):
    want = O.float_to_bf16_bits(ref_vals)
    nan = np.isnan(ref_vals)
    g = got_bits
    assert np.all(((g[nan] & 0x7F80) == 0x7F80) & ((g[nan] & 0x7F) != 0)), "NaN expected"
    bad = (g != want) & ~nan
    assert not bad.any(), f"{bad.sum()} mismatches, first at {np.argwhere(bad)[:3]}"


def dq(moe, packed, scale, form):
    out = moe.dequant(torch.as_tensor(packed, device="cuda"), torch.as_tensor(scale, device="cuda"),
                      form=form)
    torch.cuda.synchronize()
    return bits(out)


@pytest.mark.parametrize("form", FORMS)
def test_all_codes_all_scales(moe, form):
    # row s holds codes 0..15 twice with scale byte s: all 16 x 256 combinations,
    # including byte 0 (subnormal products), bytes above 128 (two multiplies in
    # the prefill form), 254 (overflow to inf) and 255 (NaN)
    codes = np.tile(np.arange(16, dtype=np.uint8), 2)
    row = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    packed = np.tile(row, (256, 1))
    scale = np.arange(256, dtype=np.uint8)[:, None]
    check_bits(dq(moe, packed, scale, form), O.dequant(packed, scale))


@pytest.mark.parametrize("form", FORMS)
def test_every_code_in_every_nibble_position(moe, form):
    """Each of the 16 codes at each of the 32 positions of a block (the
    prefill form places nibbles by shifts that depend on the position)."""
    codes = (np.arange(32)[None, :] + np.arange(16)[:, None]) % 16   # [16, 32]
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    packed = np.tile(packed, (3, 1))
    scale = np.repeat(np.array([0, 127, 200], dtype=np.uint8), 16)[:, None]
    check_bits(dq(moe, packed, scale, form), O.dequant(packed, scale))


@pytest.mark.parametrize("form", FORMS)
def test_random_rows_many_blocks(moe, form):
    rng = np.random.default_rng(3)
    packed = rng.integers(0, 256, size=(333, 2880 // 2), dtype=np.uint8)
    scale = rng.integers(0, 256, size=(333, 2880 // 32), dtype=np.uint8)
    check_bits(dq(moe, packed, scale, form), O.dequant(packed, scale))


@pytest.mark.parametrize("form", FORMS)
def test_full_size_experts_first_middle_last(moe, form):
    """glm256-shaped w13 and w2 at full size: experts 0, 127, 255 (the pages'
    prefill check compares first, middle and last experts)."""
    shape = synth.SHAPES["glm256"]
    w13, s13, w2, s2 = synth.draw_weights_cuda(shape, seed=0, layer=0)
    for e in (0, 127, 255):
        for wq, ws in ((w13, s13), (w2, s2)):
            out = moe.dequant(wq[e].contiguous(), ws[e].contiguous(), form=form)
            torch.cuda.synchronize()
            check_bits(bits(out), O.dequant(wq[e].cpu().numpy(), ws[e].cpu().numpy()))
    del w13, s13, w2, s2
    torch.cuda.empty_cache()
