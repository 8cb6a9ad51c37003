"""Host-side argument checks of the Python binding, run without a GPU.

The library reaches most tensors through bare pointers and cannot see their
sizes, so the binding checks that every such tensor has the shape, dtype and
device the call implies, and raises ValueError before the library is called.
A stand-in library records which calls get through; CPU tensors stand in for
device tensors (``is_cuda`` is patched), host buffers are marked as such.
"""
import pytest
import torch

import int4_weight_quantized_w4_gb300 as w4


class _FakeLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if name == "w4_workspace_bytes":
            return lambda *a: 1 << 16
        if name == "w4_last_error":
            return lambda: b""
        if name == "w4_status_string":
            return lambda s: b"W4_OK"

        def call(*a):
            self.calls.append(name)
            return w4.W4_OK
        return call


class _Stream:
    cuda_stream = 0


@pytest.fixture
def lib(monkeypatch):
    fake = _FakeLib()
    monkeypatch.setattr(w4, "_lib", fake)
    monkeypatch.setattr(torch.Tensor, "is_cuda", property(lambda self: not getattr(self, "_host", False)))
    monkeypatch.setattr(torch.cuda, "current_stream", lambda *a, **k: _Stream())
    return fake


def _t(shape, dtype):
    return torch.zeros(shape, dtype=dtype)


def _host(shape, dtype):
    t = torch.zeros(shape, dtype=dtype)
    t._host = True
    return t


def _rejects(lib, fn, *a, match=None, **k):
    before = len(lib.calls)
    with pytest.raises(ValueError, match=match):
        fn(*a, **k)
    assert len(lib.calls) == before, "the library was called despite a bad argument"


# ---- dense W4A8 ----------------------------------------------------------

M, K, N, G = 4, 256, 64, 2   # group 128


def _w4a8_args():
    return (_t((M, K), torch.int8), _t((M,), torch.float32), _t((K // 8, N), torch.int32),
            _t((G, N), torch.float16))


def test_w4a8_valid_call_reaches_library(lib):
    y = w4.w4a8_gemm(*_w4a8_args(), 128, bias=_t((N,), torch.bfloat16))
    assert lib.calls == ["w4a8_gemm"] and tuple(y.shape) == (M, N) and y.dtype == torch.bfloat16


def test_w4a8_bf16_scales_are_left_to_the_library(lib):
    """The library itself rejects bf16 scales for W4A8 (W4_ERR_DTYPE); the
    binding passes them on with their dtype code."""
    qx, sx, qw, _ = _w4a8_args()
    w4.w4a8_gemm(qx, sx, qw, _t((G, N), torch.bfloat16), 128)
    assert lib.calls == ["w4a8_gemm"]


@pytest.mark.parametrize("what", ["x_scale_shape", "x_scale_dtype", "scale_rows", "scale_dtype", "bias_dtype",
                                  "bias_shape", "y_shape", "y_dtype", "qweight_rows", "y_noncontig"])
def test_w4a8_rejects(lib, what):
    qx, sx, qw, sw = _w4a8_args()
    kw = {}
    if what == "x_scale_shape":
        sx = _t((M, 1), torch.float32)
    elif what == "x_scale_dtype":
        sx = _t((M,), torch.float16)
    elif what == "scale_rows":
        sw = _t((G + 1, N), torch.float16)
    elif what == "scale_dtype":
        sw = _t((G, N), torch.float32)
    elif what == "bias_dtype":
        kw["bias"] = _t((N,), torch.float32)
    elif what == "bias_shape":
        kw["bias"] = _t((N + 8,), torch.bfloat16)
    elif what == "y_shape":
        kw["y"] = _t((M, N + 1), torch.bfloat16)
    elif what == "y_dtype":
        kw["y"] = _t((M, N), torch.float16)
    elif what == "qweight_rows":
        qw = _t((K // 8 + 1, N), torch.int32)
    elif what == "y_noncontig":
        kw["y"] = _t((N, M), torch.bfloat16).t()
    _rejects(lib, w4.w4a8_gemm, qx, sx, qw, sw, 128, **kw)


def test_w4a8_bad_group_is_left_to_the_library(lib):
    """A group that does not divide K gives no scale shape to check: the
    library reports W4_ERR_GROUP."""
    qx, sx, qw, _ = _w4a8_args()
    w4.w4a8_gemm(qx, sx, qw, _t((3, N), torch.float16), 100)
    assert lib.calls == ["w4a8_gemm"]


def test_w4a8_per_channel_scales(lib):
    qx, sx, qw, _ = _w4a8_args()
    w4.w4a8_gemm(qx, sx, qw, _t((1, N), torch.float16), -1)
    _rejects(lib, w4.w4a8_gemm, qx, sx, qw, _t((G, N), torch.float16), -1)
    assert lib.calls == ["w4a8_gemm"]


def test_w4a8_device_mismatch(lib):
    qx, sx, qw, sw = _w4a8_args()
    _rejects(lib, w4.w4a8_gemm, qx, torch.zeros((M,), dtype=torch.float32, device="meta"), qw, sw, 128,
             match="the call runs on")


def test_w4a8_variants(lib):
    qx, sx, qw, sw = _w4a8_args()
    x = _t((M, K), torch.bfloat16)
    w4.w4a8_gemm_bf16in(x, qw, sw, 128)
    w4.w4a8_gemm_noalloc(qx, sx, qw, sw, 128)
    p = w4.w4a8_group_partials(qx, qw, 128)
    assert tuple(p.shape) == (M, G, N) and p.dtype == torch.int32
    assert lib.calls == ["w4a8_gemm_bf16in", "w4a8_gemm_noalloc", "w4a8_group_partials"]
    _rejects(lib, w4.w4a8_gemm_bf16in, x, qw, sw, 128, x_scale=_t((M + 1,), torch.float32))
    _rejects(lib, w4.w4a8_gemm_noalloc, qx, sx, qw, sw, 128, bias=_t((N,), torch.float16))
    _rejects(lib, w4.w4a8_group_partials, qx, qw, 128, out=_t((M, G + 1, N), torch.int32))
    _rejects(lib, w4.w4a8_gemm, qx, sx, qw, sw, 128, workspace=_t((64, 64), torch.uint8).t())


def test_quant_outputs(lib):
    x = _t((M, K), torch.bfloat16)
    w4.w4_quant_act_per_token(x, "int8", q=_t((M, K), torch.int8))
    w4.w4_quant_act_per_token(x, "fp8", q=_t((M, K), torch.uint8))
    assert lib.calls == ["w4_quant_act_per_token"] * 2
    _rejects(lib, w4.w4_quant_act_per_token, x, "int8", q=_t((M, K), torch.uint8))
    _rejects(lib, w4.w4_quant_act_per_token, x, "fp8", scale=_t((M,), torch.float16))


# ---- W4A16 ---------------------------------------------------------------

def test_w4a16_zeros_and_scales(lib):
    x, qw = _t((1, K), torch.bfloat16), _t((K // 8, N), torch.int32)
    w4.w4a16_gemm(x, qw, _t((G, N), torch.bfloat16), 128, zeros=_t((G, N), torch.bfloat16))
    assert lib.calls == ["w4a16_gemm"]
    _rejects(lib, w4.w4a16_gemm, x, qw, _t((G, N), torch.float16), 128, zeros=_t((G, N), torch.float16))
    _rejects(lib, w4.w4a16_gemm, x, qw, _t((G, N), torch.float16), 128, zeros=_t((G - 1, N), torch.bfloat16))
    _rejects(lib, w4.w4a16_gemm, x, qw, _t((G * 2, N), torch.float16), 128)


def test_w4a16_host_entry(lib):
    qw, sw = _t((K // 8, N), torch.int32), _t((G, N), torch.float16)
    xh, yh = _host((2, K), torch.bfloat16), _host((2, N), torch.bfloat16)
    xd, yd = _t((2, K), torch.bfloat16), _t((2, N), torch.bfloat16)
    w4.w4a16_gemm_host(xh, xd, qw, sw, 128, yd, yh)
    assert lib.calls == ["w4a16_gemm_host"]
    _rejects(lib, w4.w4a16_gemm_host, xd, xd, qw, sw, 128, yd, yh, match="CPU tensor")
    _rejects(lib, w4.w4a16_gemm_host, xh, xd, qw, sw, 128, _t((2, N + 1), torch.bfloat16), yh)
    _rejects(lib, w4.w4a16_gemm_host, xh, xd, _t((K // 8 + 1, N), torch.int32), sw, 128, yd, yh)


# ---- grouped experts and the MoE glue ----------------------------------

E, R, KE, NE = 4, 40, 256, 64


def test_moe_grouped(lib):
    qx, sx = _t((R, KE), torch.uint8), _t((R,), torch.float32)
    off, qw, sw = _t((E + 1,), torch.int32), _t((E, NE, KE // 8), torch.int32), _t((E, NE, KE // 128), torch.float16)
    w4.w4afp8_moe_grouped_gemm(qx, sx, off, qw, sw, 128)
    x = _t((R, KE), torch.bfloat16)
    w4.w4afp8_moe_gemm_bf16in(x, None, off, qw, sw, 128)
    w4.w4afp8_moe_gemm_bf16in(x, _t((2 * R,), torch.int32), off, qw, sw, 128)
    assert lib.calls == ["w4afp8_moe_grouped_gemm"] + ["w4afp8_moe_gemm_bf16in"] * 2
    _rejects(lib, w4.w4afp8_moe_grouped_gemm, qx, sx, _t((E + 1,), torch.int64), qw, sw, 128)
    _rejects(lib, w4.w4afp8_moe_grouped_gemm, qx, sx, off, qw, _t((E, NE, 1), torch.float16), 128)
    _rejects(lib, w4.w4afp8_moe_gemm_bf16in, x, _t((R,), torch.int64), off, qw, sw, 128)
    _rejects(lib, w4.w4afp8_moe_gemm_bf16in, x, None, off, qw, sw, 128, y=_t((R, NE), torch.float32))


def test_moe_glue(lib):
    T, k, H = 10, 2, 64
    out = w4.w4_moe_route(_t((T, E), torch.float32), k)
    assert [tuple(o.shape) for o in out] == [(T, k), (T, k), (E + 1,), (T * k,), (T, k)]
    bad = list(out)
    bad[1] = _t((T, k), torch.float16)
    _rejects(lib, w4.w4_moe_route, _t((T, E), torch.float32), k, out=tuple(bad))
    w4.w4_moe_gather_quant_fp8(_t((T, H), torch.bfloat16), _t((T * k,), torch.int32))
    _rejects(lib, w4.w4_moe_gather_quant_fp8, _t((T, H), torch.bfloat16), _t((T * k,), torch.int64))
    w4.w4_moe_silu_mul_quant_fp8(_t((R, 2 * H), torch.bfloat16), act=_t((R, H), torch.bfloat16))
    _rejects(lib, w4.w4_moe_silu_mul_quant_fp8, _t((R, 2 * H + 1), torch.bfloat16))
    _rejects(lib, w4.w4_moe_silu_mul_quant_fp8, _t((R, 2 * H), torch.bfloat16), act=_t((R, 2 * H), torch.bfloat16))
    w4.w4_moe_combine(_t((R, H), torch.bfloat16), _t((T, k), torch.float32), _t((T, k), torch.int32))
    _rejects(lib, w4.w4_moe_combine, _t((R, H), torch.bfloat16), _t((T, k + 1), torch.float32),
             _t((T, k), torch.int32))
    _rejects(lib, w4.w4_moe_combine, _t((R, H), torch.bfloat16), _t((T, k), torch.float32),
             _t((T, k), torch.int64))
    assert lib.calls == ["w4_moe_route", "w4_moe_gather_quant_fp8", "w4_moe_silu_mul_quant_fp8", "w4_moe_combine"]


# ---- weight tools and the vocab table -------------------------------------

def test_quantize_groupwise_outputs(lib):
    w = _t((N, K), torch.bfloat16)
    pk, sc, z = w4.w4_quantize_groupwise(w, 64)
    assert (tuple(pk.shape), tuple(sc.shape), sc.dtype) == ((N, K // 2), (N, K // 64), torch.float32)
    _rejects(lib, w4.w4_quantize_groupwise, w, 64, scale=_t((N, K // 128), torch.float32))
    _rejects(lib, w4.w4_quantize_groupwise, w, 64, zero=_t((N, K // 64), torch.bfloat16))
    assert lib.calls == ["w4_quantize_groupwise"]


V, D = 100, 256


def test_table_scales_must_be_fp32(lib):
    """The page's checkpoint keeps the table's scale and zero in bf16; the
    library reads fp32, so bf16 tensors (half the bytes) are refused rather
    than read past their end."""
    table, h = _t((V, D // 2), torch.uint8), _t((1, D), torch.bfloat16)
    sc, z = _t((V, D // 64), torch.float32), _t((V, D // 64), torch.float32)
    w4.w4_lm_head_gemv(h, table, sc, z, 64)
    w4.w4_embedding_gather(_t((3,), torch.int32), table, sc, z, 64)
    assert lib.calls == ["w4_lm_head_gemv", "w4_embedding_gather"]
    _rejects(lib, w4.w4_lm_head_gemv, h, table, sc.bfloat16(), z.bfloat16(), 64, match="dtype")
    _rejects(lib, w4.w4_lm_head_gemv, h, table, _t((V, D // 128), torch.float32), z, 64)
    _rejects(lib, w4.w4_embedding_gather, _t((3,), torch.int32), table, sc, z.bfloat16(), 64)
    _rejects(lib, w4.w4_embedding_gather, _t((3,), torch.int64), table, sc, z, 64)
    _rejects(lib, w4.w4_lm_head_gemv, h, table, sc, z, 64, y=_t((1, V + 1), torch.bfloat16))
