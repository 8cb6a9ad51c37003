"""Host-side checks of the C ABI that need no GPU: the library builds, loads
and exports every symbol include/w4.h declares, and argument validation
returns its documented status before anything is launched."""
import ctypes
import os
import re

import pytest

import int4_weight_quantized_w4_gb300 as w4
from int4_weight_quantized_w4_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "w4.h")
FAKE = ctypes.c_void_p(1 << 20)    # 16-byte aligned, never dereferenced: validation fails first
ODD = ctypes.c_void_p((1 << 20) + 4)


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return w4.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:w4_status|const char\*|void|size_t)\s+(w4\w*)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("w4_quant_act_per_token", "w4a8_gemm", "w4a16_gemm", "w4afp8_moe_grouped_gemm"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"libw4.so does not export {n}"
    assert set(names) == set(w4.EXPORTED_SYMBOLS), "binding signatures out of sync with the header"


def test_status_strings(lib):
    assert lib.w4_status_string(0) == b"W4_OK"
    assert lib.w4_status_string(4) == b"W4_ERR_DTYPE"
    assert lib.w4_status_string(99) == b"W4_ERR_UNKNOWN"


def gemm(lib, **kw):
    a = dict(qx=FAKE, sx=FAKE, qw=FAKE, ws=FAKE, wdt=w4.W4_FP16, group=128, bias=None, y=FAKE,
             M=16, N=256, K=256, work=None, work_bytes=0)
    a.update(kw)
    return lib.w4a8_gemm(a["qx"], a["sx"], a["qw"], a["ws"], a["wdt"], a["group"], a["bias"], a["y"],
                         a["M"], a["N"], a["K"], a["work"], a["work_bytes"], None)


def test_w4a8_validation(lib):
    assert gemm(lib, wdt=w4.W4_BF16) == w4.W4_ERR_DTYPE          # the fp16-scale rule
    assert b"fp16" in lib.w4_last_error()
    assert gemm(lib, N=260) == w4.W4_ERR_ALIGN                    # N % 8
    assert gemm(lib, K=252) == w4.W4_ERR_ALIGN                    # K % 8
    assert gemm(lib, group=96) == w4.W4_ERR_GROUP                 # does not divide K
    assert gemm(lib, group=0) == w4.W4_ERR_GROUP
    assert gemm(lib, group=-2) == w4.W4_ERR_GROUP
    assert gemm(lib, K=264, group=-1) == w4.W4_ERR_UNSUPPORTED    # K % 16 for the MMA tiles
    assert gemm(lib, K=256, group=8) == w4.W4_ERR_UNSUPPORTED     # group % 16
    assert gemm(lib, M=-1) == w4.W4_ERR_SHAPE
    assert gemm(lib, qx=None) == w4.W4_ERR_NULL
    assert gemm(lib, y=ODD) == w4.W4_ERR_ALIGN
    assert gemm(lib, M=0) == w4.W4_OK                             # empty: no-op, no launch
    assert lib.w4_last_error() == b""
    # workspace: missing, too small, misaligned
    need = lib.w4_workspace_bytes(w4.W4_OP_W4A8, 16, 256, 256, 128)
    assert need == 16 * 256 * 2
    assert gemm(lib) == w4.W4_ERR_WORKSPACE
    assert gemm(lib, work=FAKE, work_bytes=need - 1) == w4.W4_ERR_WORKSPACE
    assert gemm(lib, work=ODD, work_bytes=need) == w4.W4_ERR_WORKSPACE


def test_w4a8_partials_validation(lib):
    assert lib.w4a8_group_partials(FAKE, FAKE, 128, None, 16, 256, 256, FAKE, 1 << 20, None) == w4.W4_ERR_NULL
    assert lib.w4a8_group_partials(FAKE, FAKE, 100, FAKE, 16, 256, 256, FAKE, 1 << 20, None) == w4.W4_ERR_GROUP
    assert lib.w4a8_group_partials(FAKE, FAKE, -1, FAKE, 16, 256, 32768, FAKE, 1 << 30, None) == w4.W4_ERR_UNSUPPORTED


def test_w4a16_validation(lib):
    def call(**kw):
        a = dict(x=FAKE, qw=FAKE, ws=FAKE, wdt=w4.W4_FP16, z=None, group=128, bias=None, y=FAKE,
                 M=1, N=256, K=256)
        a.update(kw)
        return lib.w4a16_gemm(a["x"], a["qw"], a["ws"], a["wdt"], a["z"], a["group"], a["bias"], a["y"],
                              a["M"], a["N"], a["K"], None)
    assert call(wdt=w4.W4_INT8) == w4.W4_ERR_DTYPE
    assert call(group=16) == w4.W4_ERR_UNSUPPORTED
    assert call(group=32) == w4.W4_ERR_UNSUPPORTED
    assert call(K=288, group=-1) == w4.W4_ERR_UNSUPPORTED         # K % 64
    assert call(K=131072, group=128) == w4.W4_ERR_UNSUPPORTED     # a row of x does not fit in shared memory
    assert call(N=12) == w4.W4_ERR_ALIGN
    assert call(group=3) == w4.W4_ERR_GROUP
    assert call(x=None) == w4.W4_ERR_NULL
    assert call(qw=ODD) == w4.W4_ERR_ALIGN
    assert call(ws=ctypes.c_void_p((1 << 20) + 8)) == w4.W4_ERR_ALIGN   # scales and zeros arrive by TMA
    assert call(z=ctypes.c_void_p((1 << 20) + 8)) == w4.W4_ERR_ALIGN
    assert call(M=0) == w4.W4_OK


def test_quant_validation(lib):
    def call(**kw):
        a = dict(x=FAKE, xdt=w4.W4_BF16, M=4, K=256, qdt=w4.W4_INT8, q=FAKE, s=FAKE)
        a.update(kw)
        return lib.w4_quant_act_per_token(a["x"], a["xdt"], a["M"], a["K"], a["qdt"], a["q"], a["s"], None)
    assert call(xdt=w4.W4_INT8) == w4.W4_ERR_DTYPE
    assert call(xdt=w4.W4_FP16, M=0) == w4.W4_OK               # fp16 activations are accepted
    assert call(qdt=w4.W4_BF16) == w4.W4_ERR_DTYPE
    assert call(K=12) == w4.W4_ERR_ALIGN
    assert call(K=0) == w4.W4_ERR_SHAPE
    assert call(q=None) == w4.W4_ERR_NULL
    assert call(x=ODD) == w4.W4_ERR_ALIGN
    assert call(M=0) == w4.W4_OK


def test_moe_validation(lib):
    def call(**kw):
        a = dict(qx=FAKE, sx=FAKE, off=FAKE, E=64, qw=FAKE, ws=FAKE, wdt=w4.W4_FP16, group=128, y=FAKE,
                 R=32, N=256, K=256, work=FAKE, work_bytes=1 << 20)
        a.update(kw)
        return lib.w4afp8_moe_grouped_gemm(a["qx"], a["sx"], a["off"], a["E"], a["qw"], a["ws"], a["wdt"],
                                           a["group"], a["y"], a["R"], a["N"], a["K"], a["work"], a["work_bytes"],
                                           None)
    assert call(E=0) == w4.W4_ERR_SHAPE
    assert call(wdt=w4.W4_BF16) == w4.W4_ERR_DTYPE
    assert call(off=None) == w4.W4_ERR_NULL
    assert call(group=24) == w4.W4_ERR_GROUP
    assert call(K=272, group=16) == w4.W4_ERR_UNSUPPORTED        # K % 32 for the 3-D weight map
    assert call(work=None) == w4.W4_ERR_WORKSPACE
    assert call(R=0) == w4.W4_OK


def test_selftest_rejects_bad_limit(lib):
    assert lib.w4_selftest_bounded_wait(0, None) == w4.W4_ERR_SHAPE


def test_weight_tools_validation(lib):
    def q(**kw):
        a = dict(w=FAKE, wdt=w4.W4_BF16, N=4, K=256, group=128, packed=FAKE, scale=FAKE, zero=FAKE)
        a.update(kw)
        return lib.w4_quantize_groupwise(a["w"], a["wdt"], a["N"], a["K"], a["group"], a["packed"], a["scale"],
                                         a["zero"], None)
    assert q(wdt=w4.W4_INT8) == w4.W4_ERR_DTYPE
    assert q(group=96) == w4.W4_ERR_GROUP                    # does not divide K
    assert q(group=0) == w4.W4_ERR_GROUP
    assert q(K=257, group=-1) == w4.W4_ERR_UNSUPPORTED       # two codes per byte need K even ...
    assert q(K=255, group=5) == w4.W4_ERR_UNSUPPORTED        # ... and an even group
    assert q(w=None) == w4.W4_ERR_NULL
    assert q(w=ctypes.c_void_p((1 << 20) + 2)) == w4.W4_ERR_ALIGN
    assert q(N=-1) == w4.W4_ERR_SHAPE
    assert q(N=0) == w4.W4_OK
    assert lib.w4_repack_s4_to_uint4b8(FAKE, FAKE, -1, None) == w4.W4_ERR_SHAPE
    assert lib.w4_repack_s4_to_uint4b8(None, FAKE, 64, None) == w4.W4_ERR_NULL
    assert lib.w4_repack_s4_to_uint4b8(ODD, FAKE, 64, None) == w4.W4_ERR_ALIGN
    assert lib.w4_repack_s4_to_uint4b8(FAKE, FAKE, 0, None) == w4.W4_OK


def test_w4a8_bf16in_validation(lib):
    def call(**kw):
        a = dict(x=FAKE, qw=FAKE, ws=FAKE, wdt=w4.W4_FP16, group=128, bias=None, y=FAKE, sx=FAKE,
                 M=16, N=256, K=256, work=FAKE, work_bytes=1 << 20)
        a.update(kw)
        return lib.w4a8_gemm_bf16in(a["x"], a["qw"], a["ws"], a["wdt"], a["group"], a["bias"], a["y"], a["sx"],
                                    a["M"], a["N"], a["K"], a["work"], a["work_bytes"], None)
    assert call(wdt=w4.W4_BF16) == w4.W4_ERR_DTYPE
    assert call(sx=None) == w4.W4_ERR_NULL
    assert call(x=ODD) == w4.W4_ERR_ALIGN
    assert call(group=96) == w4.W4_ERR_GROUP
    assert call(K=264, group=-1) == w4.W4_ERR_UNSUPPORTED
    assert call(work=None) == w4.W4_ERR_WORKSPACE
    assert call(M=0) == w4.W4_OK


def test_embedding_validation(lib):
    def gat(**kw):
        a = dict(ids=FAKE, T=4, table=FAKE, sc=FAKE, z=FAKE, V=100, D=256, group=128, out=FAKE)
        a.update(kw)
        return lib.w4_embedding_gather(a["ids"], a["T"], a["table"], a["sc"], a["z"], a["V"], a["D"], a["group"],
                                       a["out"], None)
    assert gat(group=96) == w4.W4_ERR_GROUP
    assert gat(D=252, group=-1) == w4.W4_ERR_ALIGN
    assert gat(V=0) == w4.W4_ERR_SHAPE
    assert gat(ids=None) == w4.W4_ERR_NULL
    assert gat(out=ODD) == w4.W4_ERR_ALIGN
    assert gat(T=0) == w4.W4_OK

    def head(**kw):
        a = dict(h=FAKE, M=1, table=FAKE, sc=FAKE, z=FAKE, V=100, D=256, group=128, y=FAKE)
        a.update(kw)
        return lib.w4_lm_head_gemv(a["h"], a["M"], a["table"], a["sc"], a["z"], a["V"], a["D"], a["group"],
                                   a["y"], None)
    assert head(D=264, group=-1) == w4.W4_ERR_UNSUPPORTED      # rows read 32 codes at a time
    assert head(D=8320, group=128) == w4.W4_ERR_UNSUPPORTED    # 8 rows of h must fit in shared memory
    assert head(D=8192, group=128, M=0) == w4.W4_OK           # tensor-core form: fp16 h
    assert head(D=8192, group=64, M=0) == w4.W4_ERR_UNSUPPORTED
    assert head(D=5792, group=32, M=0) == w4.W4_OK            # the longest row that fits
    assert head(D=5824, group=32, M=0) == w4.W4_ERR_UNSUPPORTED
    assert head(table=ODD) == w4.W4_ERR_ALIGN
    assert head(M=0) == w4.W4_OK


def test_moe_glue_validation(lib):
    def route(**kw):
        a = dict(lg=FAKE, f32=1, T=100, E=64, k=8, ren=0, ids=FAKE, w=FAKE, off=FAKE, rt=FAKE, ro=FAKE, ws=FAKE,
                 wsb=1 << 20)
        a.update(kw)
        return lib.w4_moe_route(a["lg"], a["f32"], a["T"], a["E"], a["k"], a["ren"], a["ids"], a["w"], a["off"],
                                a["rt"], a["ro"], a["ws"], a["wsb"], None)
    assert route(E=1025) == w4.W4_ERR_UNSUPPORTED
    assert route(k=65, E=128) == w4.W4_ERR_SHAPE
    assert route(k=9, E=8) == w4.W4_ERR_SHAPE
    assert route(ids=None) == w4.W4_ERR_NULL
    assert route(ws=None) == w4.W4_ERR_WORKSPACE
    need = lib.w4_workspace_bytes(w4.W4_OP_MOE_ROUTE, 100, 64, 1, 0)
    assert need == 64 * 4                                   # one 256-token tile x 64 experts
    assert route(wsb=need - 1) == w4.W4_ERR_WORKSPACE
    assert route(T=0) == w4.W4_OK

    assert lib.w4_moe_gather_quant_fp8(FAKE, 10, 260, FAKE, 5, FAKE, FAKE, None) == w4.W4_ERR_ALIGN
    assert lib.w4_moe_gather_quant_fp8(FAKE, 10, 256, None, 5, FAKE, FAKE, None) == w4.W4_ERR_NULL
    assert lib.w4_moe_gather_quant_fp8(FAKE, 10, 256, FAKE, 0, FAKE, FAKE, None) == w4.W4_OK

    def moe_in(**kw):
        a = dict(x=FAKE, T=64, rt=FAKE, off=FAKE, E=8, qw=FAKE, sw=FAKE, sdt=w4.W4_FP16, group=128, y=FAKE, sx=FAKE,
                 R=128, N=256, K=256, ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return lib.w4afp8_moe_gemm_bf16in(a["x"], a["T"], a["rt"], a["off"], a["E"], a["qw"], a["sw"], a["sdt"],
                                          a["group"], a["y"], a["sx"], a["R"], a["N"], a["K"], a["ws"], a["wsb"], None)
    assert moe_in(rt=None) == w4.W4_ERR_SHAPE               # without row_token R must equal T
    assert moe_in(sdt=w4.W4_BF16) == w4.W4_ERR_DTYPE
    assert moe_in(K=240, group=-1) == w4.W4_ERR_UNSUPPORTED
    assert moe_in(wsb=16) == w4.W4_ERR_WORKSPACE
    assert moe_in(x=ODD) == w4.W4_ERR_ALIGN
    assert moe_in(R=0, T=0, rt=None) == w4.W4_OK

    assert lib.w4_moe_silu_mul_quant_fp8(FAKE, 4, 12, FAKE, FAKE, None, None) == w4.W4_ERR_ALIGN
    assert lib.w4_moe_silu_mul_quant_fp8(FAKE, 4, 16, FAKE, FAKE, ODD, None) == w4.W4_ERR_ALIGN
    assert lib.w4_moe_silu_mul_quant_fp8(FAKE, 0, 16, FAKE, FAKE, None, None) == w4.W4_OK

    assert lib.w4_moe_combine(FAKE, 16, 12, FAKE, FAKE, 2, 8, FAKE, None) == w4.W4_ERR_ALIGN
    assert lib.w4_moe_combine(FAKE, 16, 16, FAKE, None, 2, 8, FAKE, None) == w4.W4_ERR_NULL
    assert lib.w4_moe_combine(FAKE, 16, 16, FAKE, FAKE, 2, 0, FAKE, None) == w4.W4_ERR_SHAPE
    assert lib.w4_moe_combine(FAKE, 16, 16, FAKE, FAKE, 0, 8, FAKE, None) == w4.W4_OK


def test_w4a16_host_entry_validation(lib):
    def call(**kw):
        a = dict(xh=FAKE, xd=FAKE, qw=FAKE, ws=FAKE, wdt=w4.W4_FP16, z=None, group=128, b=None, yd=FAKE, yh=FAKE,
                 M=1, N=256, K=256)
        a.update(kw)
        return lib.w4a16_gemm_host(a["xh"], a["xd"], a["qw"], a["ws"], a["wdt"], a["z"], a["group"], a["b"], a["yd"],
                                   a["yh"], a["M"], a["N"], a["K"], None)
    assert call(xh=None) == w4.W4_ERR_NULL
    assert call(yh=None) == w4.W4_ERR_NULL
    assert call(xd=None) == w4.W4_ERR_NULL
    assert call(xd=ODD) == w4.W4_ERR_ALIGN
    assert call(wdt=w4.W4_INT8) == w4.W4_ERR_DTYPE
    assert call(group=96) == w4.W4_ERR_GROUP
    assert call(M=0, xh=None, yh=None) == w4.W4_OK


@pytest.mark.parametrize("M,N,K,group,extra", [
    (4096, 11008, 4096, 128, 8 * 11 * 128 * 256 * 4),    # 1,376 tiles: the last wave's 8 in 11 K parts
    (16384, 3072, 3072, -1, 16 * 8 * 128 * 256 * 4),     # 1,536 tiles: the last 16 in 8 parts
    (4096, 4096, 4096, 128, 56 * 2 * 128 * 256 * 4),     # 512 tiles: the last 56 in 2 parts
    (512, 4096, 4096, 128, 2 * 512 * 4096 * 4),          # 64 tiles: every tile in 2 parts
    (300, 264, 2048, 128, 4 * 300 * 264 * 4),            # 6 tiles: every tile in 4 parts
    (1024, 4096, 4096, 128, 0),                          # 128 tiles: one wave, no split
    (2048, 11008, 4096, 128, 0),                         # 688 tiles: the last wave over half full, no split
    (300, 10240, 1024, 128, 0),                          # a last-wave split would not pay at K = 1024
])
def test_w4a8_split_plans(lib, M, N, K, group, extra):
    """The W4A8 workspace holds the widened activations (M K 2 bytes) plus the
    fp32 partial sums of the plan the GEMM takes: none, every tile split along
    K, or only the last wave's tiles split (compact [tile][part][256][128]).
    The plan is fixed arithmetic over a 152-SM GB300, so it is the same here."""
    assert lib.w4_workspace_bytes(w4.W4_OP_W4A8, M, N, K, group) == M * K * 2 + extra
