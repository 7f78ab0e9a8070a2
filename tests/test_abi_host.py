"""The C-ABI library loads, exports what include/mxfp4_moe.h declares, and
rejects bad arguments on the host before touching the GPU (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxfp4_moe.h")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from mxfp4_mixture_experts_gb300 import moe
    return moe.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mxfp4_moe_\w+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("mxfp4_moe_route", "mxfp4_moe_route_ws", "mxfp4_moe_router", "mxfp4_moe_router_grouped",
              "mxfp4_moe_forward", "mxfp4_moe_forward_oai",
              "mxfp4_moe_forward_window",
              "mxfp4_moe_dequant", "mxfp4_moe_dequant_form", "mxfp4_moe_encode",
              "mxfp4_moe_workspace_size", "mxfp4_moe_strerror"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    from mxfp4_mixture_experts_gb300 import moe
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)", out))
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(L, n)


def test_header_compiles_as_plain_c(tmp_path):
    c = tmp_path / "t.c"
    c.write_text('#include "mxfp4_moe.h"\nint main(void){return mxfp4_moe_version()>0?0:1;}\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-c", "-I", os.path.dirname(HEADER),
                        str(c), "-o", str(tmp_path / "t.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_version_and_strerror(L):
    from mxfp4_mixture_experts_gb300 import moe
    assert moe.version() == 100
    for code in range(7):
        assert len(moe.strerror(code)) > 0
    assert moe.strerror(99) == "unknown error code"


def test_workspace_size(L):
    from mxfp4_mixture_experts_gb300 import moe
    a = moe.workspace_size(32, 2880, 2880, 128, 4)
    b = moe.workspace_size(1, 2880, 2880, 128, 4)
    assert a > b > 0
    assert a % 256 == 0
    assert moe.workspace_size(1, 2881, 2880, 128, 4) == 0      # K not a multiple of 32
    assert moe.workspace_size(1, 2880, 2880, 2048, 4) == 0     # E above the limit
    assert moe.workspace_size(1, 2880, 2880, 8, 9) == 0        # topk > E
    assert moe.workspace_size(-1, 2880, 2880, 8, 2) == 0


VP = ctypes.c_void_p


def fwd(L, **kw):
    a = dict(hidden=VP(0x10000), ids=VP(0x20000), wts=VP(0x30000), w13=VP(0x40000),
             s13=VP(0x50000), w2=VP(0x60000), s2=VP(0x70000), T=4, K=64, I=64, E=4, topk=2,
             out=VP(0x80000), status=None, ws=VP(0x100000), ws_bytes=1 << 40, path=1,
             stream=None)
    a.update(kw)
    return L.mxfp4_moe_forward(a["hidden"], a["ids"], a["wts"], a["w13"], a["s13"], a["w2"],
                               a["s2"], a["T"], a["K"], a["I"], a["E"], a["topk"], a["out"],
                               a["status"], a["ws"], a["ws_bytes"], a["path"], a["stream"])


def test_forward_rejects_bad_arguments_without_a_gpu(L):
    from mxfp4_mixture_experts_gb300 import moe as m
    assert fwd(L, hidden=None) == m.ERR_ARG
    assert fwd(L, w2=None) == m.ERR_ARG
    assert fwd(L, out=None) == m.ERR_ARG
    assert fwd(L, path=3) == m.ERR_ARG
    assert fwd(L, K=65) == m.ERR_SHAPE
    assert fwd(L, I=48) == m.ERR_SHAPE
    assert fwd(L, topk=0) == m.ERR_SHAPE
    assert fwd(L, topk=5) == m.ERR_SHAPE          # topk > E
    assert fwd(L, E=0) == m.ERR_SHAPE
    assert fwd(L, T=-1) == m.ERR_SHAPE
    assert fwd(L, T=33, path=1) == m.ERR_SHAPE    # decode limited to 32 tokens
    assert fwd(L, K=96, I=96, T=40, path=2) == m.ERR_SHAPE   # prefill needs multiples of 64
    assert fwd(L, K=96, I=64, T=4, path=1) == m.ERR_SHAPE    # decode needs multiples of 64 too
    assert fwd(L, K=64, I=96, T=4, path=1) == m.ERR_SHAPE
    assert fwd(L, hidden=VP(0x10008)) == m.ERR_ALIGN
    assert fwd(L, w13=VP(0x40004)) == m.ERR_ALIGN
    assert fwd(L, s2=VP(0x70001)) == m.ERR_ALIGN
    assert fwd(L, out=VP(0x80002)) == m.ERR_ALIGN
    assert fwd(L, ws=VP(0x100080)) == m.ERR_ALIGN
    assert fwd(L, ws=None) == m.ERR_WORKSPACE
    need = L.mxfp4_moe_workspace_size(4, 64, 64, 4, 2)
    assert fwd(L, ws_bytes=need - 1) == m.ERR_WORKSPACE
    assert fwd(L, T=0) == m.OK                    # nothing to do, nothing enqueued


def fwd_oai(L, **kw):
    a = dict(hidden=VP(0x10000), ids=VP(0x20000), wts=VP(0x30000), w13=VP(0x40000),
             s13=VP(0x50000), b13=VP(0x58000), w2=VP(0x60000), s2=VP(0x70000), b2=VP(0x78000),
             T=4, K=64, I=64, E=4, topk=2, out=VP(0x80000), status=None, ws=VP(0x100000),
             ws_bytes=1 << 40, path=1, stream=None)
    a.update(kw)
    return L.mxfp4_moe_forward_oai(a["hidden"], a["ids"], a["wts"], a["w13"], a["s13"], a["b13"],
                                   a["w2"], a["s2"], a["b2"], a["T"], a["K"], a["I"], a["E"],
                                   a["topk"], a["out"], a["status"], a["ws"], a["ws_bytes"],
                                   a["path"], a["stream"])


def test_forward_oai_rejects_bad_arguments_without_a_gpu(L):
    from mxfp4_mixture_experts_gb300 import moe as m
    assert fwd_oai(L, b13=None) == m.ERR_ARG
    assert fwd_oai(L, b2=None) == m.ERR_ARG
    assert fwd_oai(L, hidden=None) == m.ERR_ARG
    assert fwd_oai(L, path=3) == m.ERR_ARG
    assert fwd_oai(L, b13=VP(0x58002)) == m.ERR_ALIGN
    assert fwd_oai(L, b2=VP(0x78001)) == m.ERR_ALIGN
    assert fwd_oai(L, w13=VP(0x40004)) == m.ERR_ALIGN
    assert fwd_oai(L, K=65) == m.ERR_SHAPE
    assert fwd_oai(L, T=33, path=1) == m.ERR_SHAPE    # decode limited to 32 tokens
    assert fwd_oai(L, K=96, I=96, T=40, path=2) == m.ERR_SHAPE   # prefill needs multiples of 64
    assert fwd_oai(L, K=96, I=64) == m.ERR_SHAPE
    assert fwd_oai(L, ws=None) == m.ERR_WORKSPACE
    need = L.mxfp4_moe_workspace_size(4, 64, 64, 4, 2)
    assert fwd_oai(L, ws_bytes=need - 1) == m.ERR_WORKSPACE
    assert fwd_oai(L, T=0) == m.OK


def test_router_rejects_bad_arguments_without_a_gpu(L):
    from mxfp4_mixture_experts_gb300 import moe as m
    R = L.mxfp4_moe_router
    ok = dict(lg=VP(0x1000), b=None, T=4, E=64, k=4, sc=0, ids=VP(0x2000), w=VP(0x3000))

    def call(**kw):
        a = dict(ok, **kw)
        return R(a["lg"], a["b"], a["T"], a["E"], a["k"], a["sc"], a["ids"], a["w"], None)
    assert call(E=0) == m.ERR_SHAPE
    assert call(E=1025) == m.ERR_SHAPE
    assert call(k=0) == m.ERR_SHAPE
    assert call(k=33, E=64) == m.ERR_SHAPE
    assert call(k=9, E=8) == m.ERR_SHAPE
    assert call(T=-1) == m.ERR_SHAPE
    assert call(sc=2) == m.ERR_ARG
    assert call(lg=None) == m.ERR_ARG
    assert call(ids=None) == m.ERR_ARG
    assert call(w=VP(0x3002)) == m.ERR_ALIGN
    assert call(b=VP(0x4001)) == m.ERR_ALIGN
    assert call(T=0) == m.OK


def test_router_grouped_rejects_bad_arguments_without_a_gpu(L):
    from mxfp4_mixture_experts_gb300 import moe as m
    R = L.mxfp4_moe_router_grouped
    ok = dict(lg=VP(0x1000), b=None, T=4, E=64, k=4, sc=1, ng=8, tg=2, bw=1, ids=VP(0x2000),
              w=VP(0x3000))

    def call(**kw):
        a = dict(ok, **kw)
        return R(a["lg"], a["b"], a["T"], a["E"], a["k"], a["sc"], a["ng"], a["tg"], a["bw"],
                 a["ids"], a["w"], None)
    assert call(ng=0) == m.ERR_SHAPE
    assert call(ng=33, E=66) == m.ERR_SHAPE
    assert call(ng=6) == m.ERR_SHAPE            # 64 % 6 != 0
    assert call(tg=0) == m.ERR_SHAPE
    assert call(tg=9) == m.ERR_SHAPE
    assert call(k=17, tg=2) == m.ERR_SHAPE      # 2 groups of 8 hold 16 experts
    assert call(k=0) == m.ERR_SHAPE
    assert call(E=1025, ng=1, tg=1) == m.ERR_SHAPE
    assert call(bw=2) == m.ERR_ARG
    assert call(sc=5) == m.ERR_ARG
    assert call(lg=None) == m.ERR_ARG
    assert call(ids=VP(0x2001)) == m.ERR_ALIGN
    assert call(T=0) == m.OK
    assert call(T=0, k=16, tg=2, ng=8, bw=0) == m.OK


def test_encode_rejects_bad_arguments_without_a_gpu(L):
    from mxfp4_mixture_experts_gb300 import moe as m
    enc = L.mxfp4_moe_encode
    assert enc(VP(0x1000), 4, 48, 0, VP(0x2000), VP(0x3000), None) == m.ERR_SHAPE
    assert enc(VP(0x1000), 4, 16, 0, VP(0x2000), VP(0x3000), None) == m.ERR_SHAPE
    assert enc(VP(0x1000), -1, 64, 0, VP(0x2000), VP(0x3000), None) == m.ERR_SHAPE
    assert enc(VP(0x1000), 4, 64, 2, VP(0x2000), VP(0x3000), None) == m.ERR_ARG
    assert enc(None, 4, 64, 0, VP(0x2000), VP(0x3000), None) == m.ERR_ARG
    assert enc(VP(0x1000), 4, 64, 1, VP(0x2000), None, None) == m.ERR_ARG
    assert enc(VP(0x1008), 4, 64, 0, VP(0x2000), VP(0x3000), None) == m.ERR_ALIGN
    assert enc(VP(0x1000), 4, 64, 0, VP(0x2002), VP(0x3000), None) == m.ERR_ALIGN
    assert enc(VP(0x1000), 0, 64, 0, VP(0x2000), VP(0x3000), None) == m.OK


def test_forward_window_rejects_bad_arguments_without_a_gpu(L):
    from mxfp4_mixture_experts_gb300 import moe as m

    def call(base=0, per_route=0, wts=VP(0x30000), path=1, **kw):
        a = dict(hidden=VP(0x10000), ids=VP(0x20000), w13=VP(0x40000), s13=VP(0x50000),
                 w2=VP(0x60000), s2=VP(0x70000), T=4, K=64, I=64, E=4, topk=2, out=VP(0x80000),
                 ws=VP(0x100000), ws_bytes=1 << 40)
        a.update(kw)
        return L.mxfp4_moe_forward_window(a["hidden"], a["ids"], wts, a["w13"], a["s13"], a["w2"],
                                          a["s2"], a["T"], a["K"], a["I"], a["E"], a["topk"], base,
                                          per_route, a["out"], None, a["ws"], a["ws_bytes"], path,
                                          None)
    assert call(base=-1) == m.ERR_ARG
    assert call(per_route=2) == m.ERR_ARG
    assert call(wts=None) == m.ERR_ARG            # weights needed for the token sums
    assert call(path=3) == m.ERR_ARG
    assert call(K=65) == m.ERR_SHAPE
    assert call(T=33, path=1) == m.ERR_SHAPE
    assert call(out=VP(0x80008)) == m.ERR_ALIGN
    assert call(ws=None) == m.ERR_WORKSPACE
    assert call(T=0) == m.OK


def test_route_and_dequant_reject_bad_arguments(L):
    from mxfp4_mixture_experts_gb300 import moe as m
    r = L.mxfp4_moe_route(VP(0x1000), 4, 0, 8, VP(0x2000), VP(0x3000), VP(0x4000), None, None)
    assert r == m.ERR_SHAPE
    r = L.mxfp4_moe_route(VP(0x1000), 4, 2, 8, None, VP(0x3000), VP(0x4000), None, None)
    assert r == m.ERR_ARG
    r = L.mxfp4_moe_route(None, 4, 2, 8, VP(0x2000), VP(0x3000), VP(0x4000), None, None)
    assert r == m.ERR_ARG
    assert L.mxfp4_moe_dequant(VP(0x1000), VP(0x2000), 4, 48, VP(0x3000), None) == m.ERR_SHAPE
    assert L.mxfp4_moe_dequant(VP(0x1008), VP(0x2000), 4, 64, VP(0x3000), None) == m.ERR_ALIGN
    assert L.mxfp4_moe_dequant(None, VP(0x2000), 4, 64, VP(0x3000), None) == m.ERR_ARG
    assert L.mxfp4_moe_dequant(VP(0x1000), VP(0x2000), 0, 64, VP(0x3000), None) == m.OK
    for form in (1, 2):
        f = L.mxfp4_moe_dequant_form
        assert f(VP(0x1000), VP(0x2000), 4, 48, form, VP(0x3000), None) == m.ERR_SHAPE
        assert f(VP(0x1008), VP(0x2000), 4, 64, form, VP(0x3000), None) == m.ERR_ALIGN
        assert f(VP(0x1000), VP(0x2000), 0, 64, form, VP(0x3000), None) == m.OK
    for form in (0, 3, -1):
        assert L.mxfp4_moe_dequant_form(VP(0x1000), VP(0x2000), 4, 64, form, VP(0x3000),
                                        None) == m.ERR_ARG


def test_noalloc_array_holds_the_decode_workspace_of_every_workload_shape(L):
    """The fixed array of mxfp4_moe_forward_noalloc fits the decode path of
    the four decode workload shapes at their largest token count (T = 32)."""
    from mxfp4_mixture_experts_gb300 import synth
    src = open(HEADER).read()
    m = re.search(r"#define\s+MXFP4_MOE_NOALLOC_BYTES\s+\((\d+)u\s*\*\s*(\d+)u\s*\*\s*(\d+)u\)", src)
    assert m, "MXFP4_MOE_NOALLOC_BYTES not found"
    cap = int(m.group(1)) * int(m.group(2)) * int(m.group(3))
    for name in ("single32", "gptoss128", "glm256", "widek256"):
        s = synth.SHAPES[name]
        need = L.mxfp4_moe_workspace_size(32, s.K, s.I, s.E, s.topk)
        assert 0 < need <= cap, (name, need, cap)


def test_workspace_zero_prefix_is_fixed_and_inside_every_workspace(L):
    from mxfp4_mixture_experts_gb300 import moe
    z = moe.workspace_zero_bytes()
    assert 0 < z <= 16 * 1024 and z % 256 == 0
    for T in (1, 7, 32, 33, 8192):
        assert L.mxfp4_moe_workspace_size(T, 2880, 2880, 128, 4) > z


def test_route_ws_rejects_bad_arguments(L):
    from mxfp4_mixture_experts_gb300 import moe as m
    n = L.mxfp4_moe_route_workspace_size(8192, 8, 256)
    assert n > 0 and L.mxfp4_moe_route_workspace_size(1, 0, 8) == 0
    f = L.mxfp4_moe_route_ws
    assert f(VP(0x1000), 4, 2, 8, VP(0x2000), VP(0x3000), VP(0x4000), None, None, 0, None) == \
        m.ERR_WORKSPACE
    assert f(VP(0x1000), 4, 2, 8, VP(0x2000), VP(0x3000), VP(0x4000), None, VP(0x5008), n,
             None) == m.ERR_ALIGN
    assert f(VP(0x1000), 4, 0, 8, VP(0x2000), VP(0x3000), VP(0x4000), None, VP(0x5000), n,
             None) == m.ERR_SHAPE
