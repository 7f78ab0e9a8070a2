"""mxfp4_moe_dequant (same register decode as the decode/prefill kernels)
vs the oracle: bf16 bits identical, NaN compared as NaN."""
import numpy as np
import pytest
import torch

from mxfp4_mixture_experts_gb300 import synth
from oracle import mxfp4_moe_oracle as O

pytestmark = pytest.mark.gpu


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


def test_all_codes_all_scales(moe):
    # row s holds codes 0..15 twice with scale byte s: all 16 x 256 combinations
    codes = np.tile(np.arange(16, dtype=np.uint8), 2)
    row = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
    packed = np.tile(row, (256, 1))
    scale = np.arange(256, dtype=np.uint8)[:, None]
    out = moe.dequant(torch.as_tensor(packed, device="cuda"), torch.as_tensor(scale, device="cuda"))
    torch.cuda.synchronize()
    check_bits(bits(out), O.dequant(packed, scale))


def test_random_rows_many_blocks(moe):
    rng = np.random.default_rng(3)
    packed = rng.integers(0, 256, size=(333, 2880 // 2), dtype=np.uint8)
    scale = rng.integers(0, 256, size=(333, 2880 // 32), dtype=np.uint8)
    out = moe.dequant(torch.as_tensor(packed, device="cuda"), torch.as_tensor(scale, device="cuda"))
    torch.cuda.synchronize()
    check_bits(bits(out), O.dequant(packed, scale))


def test_full_size_experts_first_middle_last(moe):
    """glm256-shaped w13 and w2 at full size: experts 0, 127, 255 (the pages'
    prefill check compares first, middle and last experts)."""
    shape = synth.SHAPES["glm256"]
    w13, s13, w2, s2 = synth.draw_weights_cuda(shape, seed=0, layer=0)
    for e in (0, 127, 255):
        for wq, ws in ((w13, s13), (w2, s2)):
            out = moe.dequant(wq[e].contiguous(), ws[e].contiguous())
            torch.cuda.synchronize()
            check_bits(bits(out), O.dequant(wq[e].cpu().numpy(), ws[e].cpu().numpy()))
    del w13, s13, w2, s2
    torch.cuda.empty_cache()
