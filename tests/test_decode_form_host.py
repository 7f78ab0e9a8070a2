"""Host-only checks of the decode kernel's form choice (no GPU): every decode
T of a layer shape runs one form when the shape's largest T runs a 10- to
12-warp form (calls of mixed T then run the same code), the rows-starved wide
shapes fall back to the 7-consumer + producer form, and shapes outside the
decode path are refused."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from mxfp4_mixture_experts_gb300 import moe, synth  # noqa: E402

SMEM = 232448   # opt-in shared memory per block on the target GPU (227 KB)


def form(name, T, smem=SMEM):
    s = synth.SHAPES[name]
    return moe.decode_form(T, s.K, s.I, s.E, s.topk, smem)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    try:
        moe.lib()
    except Exception as e:  # the library is built by __graft_entry__.build()
        pytest.skip(f"library not built: {e}")


def test_gpt_oss_shape_runs_one_form_for_every_t():
    forms = {form("gptoss128", T) for T in range(1, 33)}
    assert len(forms) == 1
    (cw,) = forms
    assert 10 <= cw <= 12


def test_wide_shapes_fall_back_to_the_producer_form_at_large_t():
    for name in ("glm256", "widek256"):
        assert form(name, 32) == 7
        assert form(name, 1) >= 10          # one token's rows fit next to 10+ consumer warps
    # the largest T runs the producer form, so each T keeps the form it needs
    assert form("single32", 32) == 7
    assert form("single32", 1) == 12


def test_less_shared_memory_never_picks_more_warps_at_the_largest_t():
    # (at smaller T a smaller budget can give more warps: once the largest T
    # no longer fits a 10- to 12-warp form, each T takes the form it needs)
    for name in ("gptoss128", "glm256", "widek256", "single32"):
        prev = form(name, 32)
        for smem in (200 * 1024, 160 * 1024, 120 * 1024, 80 * 1024):
            cw = form(name, 32, smem)
            assert cw <= prev or cw == 0, (name, smem, cw, prev)
            prev = cw
    # and a budget too small for every form is reported as 0
    assert form("widek256", 32, 64 * 1024) == 0


def test_the_shape_rule_gives_way_when_the_largest_t_loses_the_wide_forms():
    # gpt-oss at 200 KB: T = 32 no longer fits 10 to 12 warps, so T = 1 takes its own form
    assert form("gptoss128", 32, 200 * 1024) < 10
    assert form("gptoss128", 1, 200 * 1024) >= 10


def test_shapes_outside_the_decode_path_are_refused():
    s = synth.SHAPES["gptoss128"]
    assert moe.decode_form(0, s.K, s.I, s.E, s.topk) == -1
    assert moe.decode_form(33, s.K, s.I, s.E, s.topk) == -1
    assert moe.decode_form(32, 2880 + 32, s.I, s.E, s.topk) == -1     # K % 64
    assert moe.decode_form(32, s.K, s.I, 256, 33) == -1                # topk > 32
    assert moe.decode_form(32, s.K, s.I, 2, 4) == -1                   # topk > E
    assert moe.decode_form(32, s.K, s.I, 1025, 4) == -1                # E > 1024
