"""int4-weight quantized linear layer for NVIDIA GB300 (sm_103a).

A thin ctypes binding over the C ABI in ``include/w4.h`` (``libw4.so``). Each
function has the name of the C entry point it calls and only marshals
arguments: it checks tensor shapes and dtypes, allocates outputs with PyTorch
when the caller passes none, and passes raw device pointers plus the current
CUDA stream. Every step of the computation runs in the library's kernels;
there is no fallback. If ``libw4.so`` has not been built the first call raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

__all__ = [
    "W4Error", "load", "library_path",
    "w4_quant_act_per_token", "w4a8_gemm", "w4a8_gemm_bf16in", "w4a8_gemm_noalloc", "w4a8_group_partials", "w4a16_gemm",
    "w4a16_gemm_host", "w4afp8_moe_grouped_gemm", "w4_quantize_groupwise", "w4_repack_s4_to_uint4b8",
    "w4_embedding_gather", "w4_lm_head_gemv",
    "w4_moe_route", "w4_moe_gather_quant_fp8", "w4afp8_moe_gemm_bf16in", "w4_moe_silu_mul_quant_fp8",
    "w4_moe_combine",
    "w4_device_status", "w4_selftest_bounded_wait", "apply_weights", "MIN_TOKENS_FOR_INT8",
    "W4_OK", "W4_ERR_NULL", "W4_ERR_ALIGN", "W4_ERR_GROUP", "W4_ERR_DTYPE",
    "W4_ERR_UNSUPPORTED", "W4_ERR_SHAPE", "W4_ERR_CUDA", "W4_ERR_TIMEOUT", "W4_ERR_WORKSPACE",
    "W4_OP_W4A8", "W4_OP_W4AFP8_MOE", "W4_OP_MOE_ROUTE", "w4_workspace_bytes", "EXPORTED_SYMBOLS",
]

(W4_OK, W4_ERR_NULL, W4_ERR_ALIGN, W4_ERR_GROUP, W4_ERR_DTYPE, W4_ERR_UNSUPPORTED,
 W4_ERR_SHAPE, W4_ERR_CUDA, W4_ERR_TIMEOUT, W4_ERR_WORKSPACE) = range(10)
W4_BF16, W4_FP16, W4_INT8, W4_FP8_E4M3 = range(4)
W4_OP_W4A8, W4_OP_W4AFP8_MOE, W4_OP_MOE_ROUTE = range(3)

_DIR = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_DIR, "libw4.so")

_P, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
# name -> (restype, argtypes); mirrors include/w4.h
_SIGNATURES = {
    "w4_quant_act_per_token": (_I32, [_P, _I32, _I64, _I64, _I32, _P, _P, _P]),
    "w4_workspace_bytes": (_SZ, [_I32, _I64, _I64, _I64, _I32]),
    "w4a8_gemm": (_I32, [_P, _P, _P, _P, _I32, _I32, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "w4a8_group_partials": (_I32, [_P, _P, _I32, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "w4a8_gemm_bf16in": (_I32, [_P, _P, _P, _I32, _I32, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "w4a8_gemm_noalloc": (_I32, [_P, _P, _P, _P, _I32, _I32, _P, _P, _I64, _I64, _I64, _P]),
    "w4a16_gemm": (_I32, [_P, _P, _P, _I32, _P, _I32, _P, _P, _I64, _I64, _I64, _P]),
    "w4a16_gemm_host": (_I32, [_P, _P, _P, _P, _I32, _P, _I32, _P, _P, _P, _I64, _I64, _I64, _P]),
    "w4afp8_moe_grouped_gemm": (_I32, [_P, _P, _P, _I32, _P, _P, _I32, _I32, _P, _I64, _I64, _I64, _P, _SZ, _P]),
    "w4_quantize_groupwise": (_I32, [_P, _I32, _I64, _I64, _I32, _P, _P, _P, _P]),
    "w4_repack_s4_to_uint4b8": (_I32, [_P, _P, _I64, _P]),
    "w4_embedding_gather": (_I32, [_P, _I64, _P, _P, _P, _I64, _I64, _I32, _P, _P]),
    "w4_lm_head_gemv": (_I32, [_P, _I64, _P, _P, _P, _I64, _I64, _I32, _P, _P]),
    "w4_moe_route": (_I32, [_P, _I32, _I64, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "w4_moe_gather_quant_fp8": (_I32, [_P, _I64, _I64, _P, _I64, _P, _P, _P]),
    "w4afp8_moe_gemm_bf16in": (_I32, [_P, _I64, _P, _P, _I32, _P, _P, _I32, _I32, _P, _P, _I64, _I64, _I64, _P, _SZ,
                                      _P]),
    "w4_moe_silu_mul_quant_fp8": (_I32, [_P, _I64, _I64, _P, _P, _P, _P]),
    "w4_moe_combine": (_I32, [_P, _I64, _I64, _P, _P, _I64, _I32, _P, _P]),
    "w4_last_error": (ctypes.c_char_p, []),
    "w4_status_string": (ctypes.c_char_p, [_I32]),
    "w4_device_status": (_I32, [_P]),
    "w4_selftest_bounded_wait": (_I32, [_I64, _P]),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_lib = None


class W4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def load() -> ctypes.CDLL:
    """Load ``libw4.so`` (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise RuntimeError(f"{library_path} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(library_path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def _check(status: int, what: str):
    if status != W4_OK:
        lib = load()
        msg = lib.w4_last_error().decode() or lib.w4_status_string(status).decode()
        raise W4Error(status, f"{what}: {lib.w4_status_string(status).decode()}: {msg}")


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda2d(t, name, dtypes):
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dim() == 2 and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous 2-D CUDA tensor")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} must have dtype in {dtypes}, got {t.dtype}")


def _expect(t, name, shape, dtypes, device, optional=False):
    """``t`` is read or written through a bare pointer, so the library cannot
    see its size: it must be a contiguous CUDA tensor on ``device`` with this
    exact ``shape`` (None: any) and a dtype in ``dtypes`` (None: any)."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, the call runs on {device}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} must have dtype in {dtypes}, got {t.dtype}")


def _groups(K, group):
    """Groups along K: 1 for ``group == -1``, ``K / group`` for a group that
    divides K, None for any other group (the library reports it as
    W4_ERR_GROUP, so the scale shapes are then not checked here)."""
    if group == -1:
        return 1
    if group > 0 and K % group == 0:
        return K // group
    return None


_F32, _I32T, _BF16T = (torch.float32,), (torch.int32,), (torch.bfloat16,)
_SCALE_T = (torch.float16, torch.bfloat16)   # the library rejects what a path does not take
_FP8_T = (torch.float8_e4m3fn, torch.uint8)


def _scale_dtype(t):
    return {torch.float16: W4_FP16, torch.bfloat16: W4_BF16}.get(t.dtype, -1)


def w4_workspace_bytes(op: int, M: int, N: int, K: int, group: int) -> int:
    """Device workspace in bytes that ``op`` (W4_OP_W4A8 / W4_OP_W4AFP8_MOE) needs."""
    return int(load().w4_workspace_bytes(op, M, N, K, group))


def _workspace(ws, op, M, N, K, group, device):
    need = w4_workspace_bytes(op, M, N, K, group)
    if ws is None:
        ws = torch.empty((max(need, 16),), dtype=torch.uint8, device=device)
    _expect(ws, "workspace", None, None, device)   # the library checks its size in bytes
    return ws, ws.numel() * ws.element_size()


def _dense_weight_args(what, qweight, w_scale, K, group, device, zeros=None, bias=None):
    """GPTQ ``qweight [K/8, N]`` int32, ``w_scale [G, N]``, optional bf16
    ``zeros [G, N]`` and ``bias [N]``; returns N."""
    _cuda2d(qweight, "qweight", _I32T)
    N = qweight.shape[1]
    if qweight.shape[0] * 8 != K or not isinstance(w_scale, torch.Tensor) or w_scale.dim() != 2 \
            or w_scale.shape[1] != N:
        raise ValueError(f"inconsistent shapes for {what}")
    G = _groups(K, group)
    gshape = None if G is None else (G, N)
    _expect(qweight, "qweight", None, None, device)
    _expect(w_scale, "w_scale", gshape, _SCALE_T, device)
    _expect(zeros, "zeros", gshape, _BF16T, device, optional=True)
    _expect(bias, "bias", (N,), _BF16T, device, optional=True)
    return N


def _expert_weight_args(what, qweight, w_scale, expert_offsets, K, group, device):
    """Compressed-tensors ``qweight [E, N, K/8]`` int32, ``w_scale [E, N, G]``
    and int32 ``expert_offsets [E + 1]``; returns (E, N)."""
    if not isinstance(qweight, torch.Tensor) or qweight.dim() != 3 or not qweight.is_contiguous() \
            or qweight.dtype != torch.int32:
        raise ValueError("qweight must be a contiguous int32 [E, N, K/8] tensor")
    E, N = qweight.shape[0], qweight.shape[1]
    if qweight.shape[2] * 8 != K or not isinstance(w_scale, torch.Tensor) or w_scale.dim() != 3 \
            or w_scale.shape[:2] != (E, N):
        raise ValueError(f"inconsistent shapes for {what}")
    G = _groups(K, group)
    _expect(qweight, "qweight", None, None, device)
    _expect(w_scale, "w_scale", None if G is None else (E, N, G), _SCALE_T, device)
    _expect(expert_offsets, "expert_offsets", (E + 1,), _I32T, device)
    return E, N


def w4_quant_act_per_token(x, q_dtype: str = "int8", q=None, scale=None, stream=None):
    """Per-token symmetric quantization of bf16 or fp16 ``x [M, K]``; returns
    ``(q, scale)`` with q int8 (``q_dtype="int8"``) or float8_e4m3fn (``"fp8"``)
    and fp32 scales."""
    _cuda2d(x, "x", (torch.bfloat16, torch.float16))
    M, K = x.shape
    if q_dtype == "int8":
        qd, tdt = W4_INT8, torch.int8
    elif q_dtype == "fp8":
        qd, tdt = W4_FP8_E4M3, torch.float8_e4m3fn
    else:
        raise ValueError("q_dtype must be 'int8' or 'fp8'")
    q = torch.empty((M, K), dtype=tdt, device=x.device) if q is None else q
    scale = torch.empty((M,), dtype=torch.float32, device=x.device) if scale is None else scale
    _expect(q, "q", (M, K), (torch.int8,) if qd == W4_INT8 else _FP8_T, x.device)
    _expect(scale, "scale", (M,), _F32, x.device)
    xd = W4_FP16 if x.dtype == torch.float16 else W4_BF16
    _check(load().w4_quant_act_per_token(_ptr(x), xd, M, K, qd, _ptr(q), _ptr(scale),
                                         _stream(stream, x.device)), "w4_quant_act_per_token")
    return q, scale


def w4a8_gemm(qx, x_scale, qweight, w_scale, group: int, bias=None, y=None, workspace=None, stream=None):
    """W4A8 linear: int8 ``qx [M, K]`` with fp32 ``x_scale [M]`` times GPTQ
    ``qweight [K/8, N]`` with fp16 ``w_scale [G, N]``; returns bf16 ``y [M, N]``.
    ``workspace`` (bytes from ``w4_workspace_bytes``) is allocated if not given."""
    _cuda2d(qx, "qx", (torch.int8,))
    M, K = qx.shape
    N = _dense_weight_args("w4a8_gemm", qweight, w_scale, K, group, qx.device, bias=bias)
    _expect(x_scale, "x_scale", (M,), _F32, qx.device)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=qx.device) if y is None else y
    _expect(y, "y", (M, N), _BF16T, qx.device)
    ws, wsb = _workspace(workspace, W4_OP_W4A8, M, N, K, group, qx.device)
    _check(load().w4a8_gemm(_ptr(qx), _ptr(x_scale), _ptr(qweight), _ptr(w_scale), _scale_dtype(w_scale),
                            group, _ptr(bias), _ptr(y), M, N, K, _ptr(ws), wsb, _stream(stream, qx.device)),
           "w4a8_gemm")
    return y


def w4a8_gemm_bf16in(x, qweight, w_scale, group: int, bias=None, y=None, x_scale=None, workspace=None, stream=None):
    """W4A8 linear from bf16 ``x [M, K]``: per-token int8 quantization fused into
    the GEMM's activation pass. Returns ``(y bf16 [M, N], x_scale f32 [M])``."""
    _cuda2d(x, "x", (torch.bfloat16,))
    M, K = x.shape
    N = _dense_weight_args("w4a8_gemm_bf16in", qweight, w_scale, K, group, x.device, bias=bias)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device) if y is None else y
    x_scale = torch.empty((M,), dtype=torch.float32, device=x.device) if x_scale is None else x_scale
    _expect(y, "y", (M, N), _BF16T, x.device)
    _expect(x_scale, "x_scale", (M,), _F32, x.device)
    ws, wsb = _workspace(workspace, W4_OP_W4A8, M, N, K, group, x.device)
    _check(load().w4a8_gemm_bf16in(_ptr(x), _ptr(qweight), _ptr(w_scale), _scale_dtype(w_scale), group, _ptr(bias),
                                   _ptr(y), _ptr(x_scale), M, N, K, _ptr(ws), wsb, _stream(stream, x.device)),
           "w4a8_gemm_bf16in")
    return y, x_scale


def w4a8_gemm_noalloc(qx, x_scale, qweight, w_scale, group: int, bias=None, y=None, stream=None):
    """``w4a8_gemm`` without a workspace argument: for callers that cannot
    allocate device memory, it uses the library's built-in 32 MiB workspace
    (M * K <= 16,777,216). Calls that may overlap on the GPU share that
    workspace and must be serialized by the caller."""
    _cuda2d(qx, "qx", (torch.int8,))
    M, K = qx.shape
    N = _dense_weight_args("w4a8_gemm_noalloc", qweight, w_scale, K, group, qx.device, bias=bias)
    _expect(x_scale, "x_scale", (M,), _F32, qx.device)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=qx.device) if y is None else y
    _expect(y, "y", (M, N), _BF16T, qx.device)
    # the built-in workspace is looked up on the current device: make qx's current
    with torch.cuda.device(qx.device) if qx.device.type == "cuda" else contextlib.nullcontext():
        st = load().w4a8_gemm_noalloc(_ptr(qx), _ptr(x_scale), _ptr(qweight), _ptr(w_scale), _scale_dtype(w_scale),
                                      group, _ptr(bias), _ptr(y), M, N, K, _stream(stream, qx.device))
    _check(st, "w4a8_gemm_noalloc")
    return y


def w4a8_group_partials(qx, qweight, group: int, out=None, workspace=None, stream=None):
    """Integer group partials ``P [M, G, N]`` (int32) of the W4A8 product."""
    _cuda2d(qx, "qx", (torch.int8,))
    _cuda2d(qweight, "qweight", _I32T)
    M, K = qx.shape
    N = qweight.shape[1]
    if qweight.shape[0] * 8 != K:
        raise ValueError("inconsistent shapes for w4a8_group_partials")
    _expect(qweight, "qweight", None, None, qx.device)
    G = _groups(K, group)
    out = torch.empty((M, G or 0, N), dtype=torch.int32, device=qx.device) if out is None else out
    _expect(out, "out", None if G is None else (M, G, N), _I32T, qx.device)
    ws, wsb = _workspace(workspace, W4_OP_W4A8, M, N, K, group, qx.device)
    _check(load().w4a8_group_partials(_ptr(qx), _ptr(qweight), group, _ptr(out), M, N, K, _ptr(ws), wsb,
                                      _stream(stream, qx.device)), "w4a8_group_partials")
    return out


def w4a16_gemm(x, qweight, w_scale, group: int, zeros=None, bias=None, y=None, stream=None):
    """W4A16 linear: bf16 ``x [M, K]`` times GPTQ ``qweight [K/8, N]`` with fp16
    or bf16 ``w_scale [G, N]`` and optional bf16 ``zeros [G, N]``."""
    _cuda2d(x, "x", (torch.bfloat16,))
    M, K = x.shape
    N = _dense_weight_args("w4a16_gemm", qweight, w_scale, K, group, x.device, zeros=zeros, bias=bias)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device) if y is None else y
    _expect(y, "y", (M, N), _BF16T, x.device)
    _check(load().w4a16_gemm(_ptr(x), _ptr(qweight), _ptr(w_scale), _scale_dtype(w_scale), _ptr(zeros), group,
                             _ptr(bias), _ptr(y), M, N, K, _stream(stream, x.device)), "w4a16_gemm")
    return y


def w4a16_gemm_host(x_host, x_dev, qweight, w_scale, group: int, y_dev, y_host, zeros=None, bias=None, stream=None):
    """``w4a16_gemm`` from and to host memory: copies ``x_host`` (page-locked bf16
    ``[M, K]`` CPU tensor) into ``x_dev``, runs the GEMM into ``y_dev`` and copies
    it into ``y_host`` (page-locked bf16 ``[M, N]``), all queued on the stream;
    ``y_host`` is valid once the stream is synchronized."""
    for t, name in ((x_host, "x_host"), (y_host, "y_host")):
        if not isinstance(t, torch.Tensor) or t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 2 \
                or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous 2-D bf16 CPU tensor")
    _cuda2d(x_dev, "x_dev", (torch.bfloat16,))
    M, K = x_host.shape
    N = _dense_weight_args("w4a16_gemm_host", qweight, w_scale, K, group, x_dev.device, zeros=zeros, bias=bias)
    if tuple(x_dev.shape) != (M, K) or tuple(y_host.shape) != (M, N):
        raise ValueError("inconsistent shapes for w4a16_gemm_host")
    _expect(y_dev, "y_dev", (M, N), _BF16T, x_dev.device)
    _check(load().w4a16_gemm_host(_ptr(x_host), _ptr(x_dev), _ptr(qweight), _ptr(w_scale), _scale_dtype(w_scale),
                                  _ptr(zeros), group, _ptr(bias), _ptr(y_dev), _ptr(y_host), M, N, K,
                                  _stream(stream, x_dev.device)), "w4a16_gemm_host")
    return y_host


def w4afp8_moe_grouped_gemm(qx, x_scale, expert_offsets, qweight, w_scale, group: int, y=None, workspace=None,
                            stream=None):
    """Grouped expert linear: e4m3 ``qx [R, K]`` (rows grouped by expert, as
    float8_e4m3fn or uint8 codes), fp32 ``x_scale [R]``, int32 device
    ``expert_offsets [E+1]``, ``qweight [E, N, K/8]``, fp16 ``w_scale [E, N, G]``."""
    _cuda2d(qx, "qx", _FP8_T)
    R, K = qx.shape
    E, N = _expert_weight_args("w4afp8_moe_grouped_gemm", qweight, w_scale, expert_offsets, K, group, qx.device)
    _expect(x_scale, "x_scale", (R,), _F32, qx.device)
    y = torch.empty((R, N), dtype=torch.bfloat16, device=qx.device) if y is None else y
    _expect(y, "y", (R, N), _BF16T, qx.device)
    ws, wsb = _workspace(workspace, W4_OP_W4AFP8_MOE, R, N, K, group, qx.device)
    _check(load().w4afp8_moe_grouped_gemm(_ptr(qx), _ptr(x_scale), _ptr(expert_offsets), E, _ptr(qweight),
                                          _ptr(w_scale), _scale_dtype(w_scale), group, _ptr(y), R, N, K,
                                          _ptr(ws), wsb, _stream(stream, qx.device)), "w4afp8_moe_grouped_gemm")
    return y


def w4_moe_route(logits, top_k: int, renormalize: bool = False, out=None, workspace=None, stream=None):
    """Top-k routing of router ``logits [T, E]`` (bf16 or fp32). Returns
    ``(topk_ids int32 [T,k], topk_weights fp32 [T,k], offsets int32 [E+1],
    row_token int32 [T*k], row_of int32 [T,k])``; ``out`` may pass that tuple
    preallocated."""
    _cuda2d(logits, "logits", (torch.bfloat16, torch.float32))
    T, E = logits.shape
    dev = logits.device
    if out is None:
        out = (torch.empty((T, top_k), dtype=torch.int32, device=dev),
               torch.empty((T, top_k), dtype=torch.float32, device=dev),
               torch.zeros((E + 1,), dtype=torch.int32, device=dev),
               torch.empty((T * top_k,), dtype=torch.int32, device=dev),
               torch.empty((T, top_k), dtype=torch.int32, device=dev))
    ids, wts, off, rt, ro = out
    _expect(ids, "topk_ids", (T, top_k), _I32T, dev)
    _expect(wts, "topk_weights", (T, top_k), _F32, dev)
    _expect(off, "offsets", (E + 1,), _I32T, dev)
    _expect(rt, "row_token", (T * top_k,), _I32T, dev)
    _expect(ro, "row_of", (T, top_k), _I32T, dev)
    ws, wsb = _workspace(workspace, W4_OP_MOE_ROUTE, T, E, 1, 0, dev)
    _check(load().w4_moe_route(_ptr(logits), int(logits.dtype == torch.float32), T, E, top_k, int(bool(renormalize)),
                               _ptr(ids), _ptr(wts), _ptr(off), _ptr(rt), _ptr(ro), _ptr(ws), wsb,
                               _stream(stream, dev)), "w4_moe_route")
    return out


def w4_moe_gather_quant_fp8(x, row_token, q=None, scale=None, stream=None):
    """Rows ``x[row_token[r]]`` of bf16 ``x [T, K]`` quantized per row to e4m3;
    returns ``(q float8_e4m3fn [R, K], scale fp32 [R])``."""
    _cuda2d(x, "x", (torch.bfloat16,))
    T, K = x.shape
    _expect(row_token, "row_token", None, _I32T, x.device)
    R = row_token.numel()
    q = torch.empty((R, K), dtype=torch.float8_e4m3fn, device=x.device) if q is None else q
    scale = torch.empty((R,), dtype=torch.float32, device=x.device) if scale is None else scale
    _expect(q, "q", (R, K), _FP8_T, x.device)
    _expect(scale, "scale", (R,), _F32, x.device)
    _check(load().w4_moe_gather_quant_fp8(_ptr(x), T, K, _ptr(row_token), R, _ptr(q), _ptr(scale),
                                          _stream(stream, x.device)), "w4_moe_gather_quant_fp8")
    return q, scale


def w4afp8_moe_gemm_bf16in(x, row_token, expert_offsets, qweight, w_scale, group: int, y=None, x_scale=None,
                           workspace=None, stream=None):
    """Grouped expert linear from bf16 token rows: row r is ``x[row_token[r]]``
    (``row_token`` None: row r is token r), quantized per row to e4m3 inside
    the call. Returns ``(y bf16 [R, N], x_scale fp32 [R])``."""
    _cuda2d(x, "x", (torch.bfloat16,))
    T, K = x.shape
    _expect(row_token, "row_token", None, _I32T, x.device, optional=True)
    R = T if row_token is None else row_token.numel()
    E, N = _expert_weight_args("w4afp8_moe_gemm_bf16in", qweight, w_scale, expert_offsets, K, group, x.device)
    y = torch.empty((R, N), dtype=torch.bfloat16, device=x.device) if y is None else y
    x_scale = torch.empty((R,), dtype=torch.float32, device=x.device) if x_scale is None else x_scale
    _expect(y, "y", (R, N), _BF16T, x.device)
    _expect(x_scale, "x_scale", (R,), _F32, x.device)
    ws, wsb = _workspace(workspace, W4_OP_W4AFP8_MOE, R, N, K, group, x.device)
    _check(load().w4afp8_moe_gemm_bf16in(_ptr(x), T, _ptr(row_token), _ptr(expert_offsets), E, _ptr(qweight),
                                         _ptr(w_scale), _scale_dtype(w_scale), group, _ptr(y), _ptr(x_scale), R, N,
                                         K, _ptr(ws), wsb, _stream(stream, x.device)), "w4afp8_moe_gemm_bf16in")
    return y, x_scale


def w4_moe_silu_mul_quant_fp8(h, q=None, scale=None, act=None, stream=None):
    """``silu(gate) * up`` of the bf16 gate_up output ``h [R, 2I]``, quantized per
    row to e4m3; returns ``(q [R, I], scale [R])``, and writes the bf16
    activations to ``act`` when given."""
    _cuda2d(h, "h", (torch.bfloat16,))
    R, I2 = h.shape
    if I2 % 2:
        raise ValueError("h must hold gate and up halves of equal width")
    I = I2 // 2
    q = torch.empty((R, I), dtype=torch.float8_e4m3fn, device=h.device) if q is None else q
    scale = torch.empty((R,), dtype=torch.float32, device=h.device) if scale is None else scale
    _expect(q, "q", (R, I), _FP8_T, h.device)
    _expect(scale, "scale", (R,), _F32, h.device)
    _expect(act, "act", (R, I), _BF16T, h.device, optional=True)
    _check(load().w4_moe_silu_mul_quant_fp8(_ptr(h), R, I, _ptr(q), _ptr(scale), _ptr(act),
                                            _stream(stream, h.device)), "w4_moe_silu_mul_quant_fp8")
    return q, scale


def w4_moe_combine(y, topk_weights, row_of, out=None, stream=None):
    """``out[t] = sum_j topk_weights[t, j] * y[row_of[t, j]]`` for bf16 ``y [R, H]``;
    returns bf16 ``[T, H]``."""
    _cuda2d(y, "y", (torch.bfloat16,))
    R, H = y.shape
    _cuda2d(row_of, "row_of", _I32T)
    T, k = row_of.shape
    _expect(row_of, "row_of", None, None, y.device)
    _expect(topk_weights, "topk_weights", (T, k), _F32, y.device)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device) if out is None else out
    _expect(out, "out", (T, H), _BF16T, y.device)
    _check(load().w4_moe_combine(_ptr(y), R, H, _ptr(topk_weights), _ptr(row_of), T, k, _ptr(out),
                                 _stream(stream, y.device)), "w4_moe_combine")
    return out


def w4_quantize_groupwise(w, group: int, packed=None, scale=None, zero=None, stream=None):
    """Min/max 4-bit group quantization of bf16 or fp16 ``w [N, K]``; returns
    ``(packed uint8 [N, K/2], scale f32 [N, G], zero f32 [N, G])``."""
    _cuda2d(w, "w", (torch.bfloat16, torch.float16))
    N, K = w.shape
    G = 1 if group == -1 else (K // group if group > 0 else 0)
    packed = torch.empty((N, K // 2), dtype=torch.uint8, device=w.device) if packed is None else packed
    scale = torch.empty((N, G), dtype=torch.float32, device=w.device) if scale is None else scale
    zero = torch.empty((N, G), dtype=torch.float32, device=w.device) if zero is None else zero
    _expect(packed, "packed", (N, K // 2), (torch.uint8,), w.device)
    gshape = (N, G) if _groups(K, group) is not None else None
    _expect(scale, "scale", gshape, _F32, w.device)
    _expect(zero, "zero", gshape, _F32, w.device)
    wdt = W4_FP16 if w.dtype == torch.float16 else W4_BF16
    _check(load().w4_quantize_groupwise(_ptr(w), wdt, N, K, group, _ptr(packed), _ptr(scale), _ptr(zero),
                                        _stream(stream, w.device)), "w4_quantize_groupwise")
    return packed, scale, zero


def w4_repack_s4_to_uint4b8(src, dst=None, stream=None):
    """Signed int4 pairs (any contiguous 1-byte or int32 tensor) -> uint4b8 by
    XOR 0x88 on every byte; ``dst`` may be ``src`` (in place)."""
    if not src.is_cuda or not src.is_contiguous():
        raise ValueError("src must be a contiguous CUDA tensor")
    dst = torch.empty_like(src) if dst is None else dst
    n = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != n:
        raise ValueError("dst must hold as many bytes as src")
    _check(load().w4_repack_s4_to_uint4b8(_ptr(src), _ptr(dst), n, _stream(stream, src.device)),
           "w4_repack_s4_to_uint4b8")
    return dst


def _table_args(table, scale, zero, group):
    """The quantized vocab table: packed uint8 ``[V, D/2]`` with fp32 scale and
    zero ``[V, G]``. A checkpoint's bf16 scale and zero are widened once with
    ``.float()`` (exact). Returns (V, D)."""
    _cuda2d(table, "table", (torch.uint8,))
    V, D = table.shape[0], table.shape[1] * 2
    G = _groups(D, group)
    gshape = None if G is None else (V, G)
    _expect(scale, "scale", gshape, _F32, table.device)
    _expect(zero, "zero", gshape, _F32, table.device)
    return V, D


def w4_embedding_gather(ids, table, scale, zero, group: int, out=None, stream=None):
    """Rows ``ids`` (int32 [T]) of the quantized table (packed uint8 [V, D/2],
    f32 scale/zero [V, G]) dequantized to bf16 ``[T, D]``."""
    V, D = _table_args(table, scale, zero, group)
    _expect(ids, "ids", None, _I32T, table.device)
    T = ids.numel()
    out = torch.empty((T, D), dtype=torch.bfloat16, device=table.device) if out is None else out
    _expect(out, "out", (T, D), _BF16T, table.device)
    _check(load().w4_embedding_gather(_ptr(ids), T, _ptr(table), _ptr(scale), _ptr(zero), V, D, group, _ptr(out),
                                      _stream(stream, table.device)), "w4_embedding_gather")
    return out


def w4_lm_head_gemv(h, table, scale, zero, group: int, y=None, stream=None):
    """Tied output head: bf16 ``h [M, D]`` against the quantized table
    (packed uint8 [V, D/2], f32 scale/zero [V, G]); returns bf16 ``[M, V]``."""
    _cuda2d(h, "h", (torch.bfloat16,))
    M, D = h.shape
    V, Dt = _table_args(table, scale, zero, group)
    if Dt != D:
        raise ValueError("table and h disagree on D")
    _expect(h, "h", None, None, table.device)
    y = torch.empty((M, V), dtype=torch.bfloat16, device=h.device) if y is None else y
    _expect(y, "y", (M, V), _BF16T, h.device)
    _check(load().w4_lm_head_gemv(_ptr(h), M, _ptr(table), _ptr(scale), _ptr(zero), V, D, group, _ptr(y),
                                  _stream(stream, h.device)), "w4_lm_head_gemv")
    return y


# [INC] INCXPUW4A8LinearMethod._MIN_TOKENS_FOR_INT8: below this token count the
# per-token quantization does not pay off and the call takes the W4A16 path.
MIN_TOKENS_FOR_INT8 = 512


def apply_weights(x, qweight, w_scale, group: int, bias=None, zeros=None, stream=None):
    """The int4 linear layer with the per-call path choice of [INC]
    ``INCXPUW4A8LinearMethod.apply_weights``: ``x [..., K]`` (bf16 or fp16)
    times GPTQ ``qweight [K/8, N]``; returns bf16 ``[..., N]``.

    From ``MIN_TOKENS_FOR_INT8`` tokens up, activations are quantized per token
    to int8 and the W4A8 GEMM runs (fp16 scales, no zeros); below it, the
    W4A16 GEMM runs on the bf16 activations. fp16 activations always take the
    int8 path (the W4A16 kernels read bf16), so they need fp16 scales and no
    zeros.
    """
    K = x.shape[-1]
    x2 = x.reshape(-1, K)
    M = x2.shape[0]
    int8_path = x2.dtype == torch.float16 or (M >= MIN_TOKENS_FOR_INT8 and zeros is None
                                              and w_scale.dtype == torch.float16)
    if int8_path:
        if zeros is not None:
            raise ValueError("the W4A8 path has no zeros; asymmetric weights need bf16 activations")
        if x2.dtype == torch.bfloat16:
            y, _ = w4a8_gemm_bf16in(x2, qweight, w_scale, group, bias=bias, stream=stream)
        else:
            q, sx = w4_quant_act_per_token(x2, "int8", stream=stream)
            y = w4a8_gemm(q, sx, qweight, w_scale, group, bias=bias, stream=stream)
    else:
        y = w4a16_gemm(x2, qweight, w_scale, group, zeros=zeros, bias=bias, stream=stream)
    return y.reshape(*x.shape[:-1], y.shape[-1])


def w4_device_status(stream=None, device=None) -> int:
    """Synchronize the stream and return (and clear) the kernels' status word."""
    return int(load().w4_device_status(_stream(stream, device)))


def w4_selftest_bounded_wait(spin_limit: int, stream=None, device=None):
    _check(load().w4_selftest_bounded_wait(int(spin_limit), _stream(stream, device)), "w4_selftest_bounded_wait")
