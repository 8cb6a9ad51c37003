"""Plain, slow reference for what the int4-weight linear layer computes.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this file. Every function is numpy in float64 / int64; a dense matmul
is used as a library step only where its result is exact or where float64 is
the stated precision, and each such use says which.

Sources, cited by page title and section:
  [INC]  vLLM API docs, ``inc.schemes.inc_w4a8_linear``:
         ``INCXPUW4A8LinearMethod`` (class docstring, ``create_weights``,
         ``process_weights_after_loading``, ``apply_weights``).
  [CT]   vLLM v0.10.1.1 API docs, ``compressed_tensors_w4a8_int``:
         ``CompressedTensorsW4A8Int.__init__`` / ``create_weights``.
  [FP8]  vLLM API docs, ``quantization.w4afp8``: ``W4AFP8Config.__init__``,
         ``get_checkpoint_weight_mapper``, ``_repack_signed_int4_to_uint4b8``.
  [ZEN]  vLLM API docs, ``kernels.linear.mixed_precision.zentorch``:
         ``ZentorchWNA16LinearKernel`` (``can_implement``,
         ``_zentorch_woq_eligible``, ``_maybe_process_da8w4_weights``).
  [OMNI] vllm-omni ``quantization/cpu_int4.py``: module docstring,
         ``pack_nibbles``, ``unpack_nibbles``, ``quantize_groupwise``,
         ``CPUInt4EmbeddingMethod.embedding``.

Readings where the pages are silent (each is listed in the design notes):
  * The per-token quantizer's formula is not printed ([INC] ``apply_weights``
    calls an opaque ``dynamic_per_token_int8_quant_ref(x, True, 8)``). Reading:
    symmetric, ``s = amax / 127`` in fp32 (``s = 1`` when ``amax == 0``),
    ``q = clamp(round_half_even(x / s), -127, 127)`` with an IEEE fp32 divide.
  * "8-bit float" activations ([FP8] ``input_quant``) are e4m3fn, max 448:
    ``s = amax / 448``, ``q = e4m3(x / s)`` rounded to nearest even and
    saturated to +-448.
  * The activation scale stays fp32 (the [INC] page narrows it to fp16 for
    the XPU kernel; that is a property of that kernel).
  * The asymmetric zero is the additive float zero of [OMNI]:
    ``w = (q - 8) * scale + zero``.
  * Outputs are the fp32 result ``r`` of the exact (fp64) computation; the
    stored bf16 output is ``r`` rounded to nearest even.
  * The MoE layer around the grouped GEMM ([FP8] module docstring and
    ``get_quant_method``: the int4 weights serve the routed experts; no
    routing or activation formula is printed). Reading, the plain top-k MoE
    layer: per token a softmax over the router logits; the k experts with the
    largest logits (ties to the lower expert index); weight = the softmax
    value, divided by the sum over the k chosen when renormalizing. Rows
    (token, expert) sorted by expert, then token. Between the GEMMs
    ``act = silu(gate) * up`` with ``gate`` the first half of the gate_up
    output columns, computed in fp32 and rounded to bf16, then quantized per
    row to e4m3 as the first GEMM's input was. The output of token t is
    ``sum_j w[t, j] * y[row(t, j)]``.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against values fixed by the pages or by mathematics (exhaustive layout checks,
worked ties, closed forms, brute force). No function is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_to_f64", "f32_to_bf16_bits", "bf16_bits_to_f32",
    "e4m3_decode", "e4m3_encode",
    "effective_group",
    "unpack_gptq", "unpack_ct", "pack_nibbles", "unpack_nibbles",
    "repack_signed_int4_to_uint4b8",
    "quant_int8_per_token", "quant_fp8_per_token",
    "w4a8_group_partials", "w4a8_linear",
    "w4a16_linear", "moe_grouped_linear",
    "quantize_groupwise", "dequant_rows", "embedding_rows", "lm_head_logits",
    "moe_route", "moe_gather_quant_fp8", "silu_mul_bf16", "silu_mul_quant_fp8", "moe_combine",
]

# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact: bf16 is the top half of fp32)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    with np.errstate(invalid="ignore"):
        return bf16_bits_to_f32(bits).astype(np.float64)


def f32_to_bf16_bits(r: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest, ties to even (finite inputs)."""
    u = np.ascontiguousarray(r, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """e4m3fn code -> float64: 1 sign, 4 exponent (bias 7), 3 mantissa bits;
    exponent 0 is subnormal (m * 2^-9); 0x7F / 0xFF are NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e.astype(np.float64) - 10))
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return sign * mag


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """float -> e4m3fn code, round to nearest even, saturate to +-448.

    The grid spacing in the binade ``[2^e, 2^(e+1))`` is ``2^(e-3)`` for
    ``e >= -6`` and ``2^-9`` below (subnormals). Dividing by the spacing is
    exact, so rounding the quotient half-to-even rounds the mantissa
    half-to-even.
    """
    v = np.asarray(v, dtype=np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    a = np.minimum(a, 448.0)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    step = np.exp2(e - 3.0)
    n = np.rint(a / step)               # numpy rint: round half to even
    val = n * step                       # may step up into the next binade
    # encode val exactly
    with np.errstate(divide="ignore"):
        ev = np.floor(np.log2(np.where(val > 0, val, 1.0)))
    normal = val >= 2.0 ** -6
    E = np.where(normal, ev + 7, 0).astype(np.int64)
    Mn = np.where(normal, val / np.exp2(ev) * 8 - 8, val / 2.0 ** -9)
    code = (E << 3) | Mn.astype(np.int64)
    code = np.where(val == 0, 0, code)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


# ---------------------------------------------------------------------------
# layouts
# ---------------------------------------------------------------------------

def effective_group(group: int, K: int) -> int:
    """[CT] ``create_weights``: group -1 means one group spanning the input
    dimension; any other group must divide it ([ZEN] ``can_implement``)."""
    if group == -1:
        return K
    if group <= 0 or K % group != 0:
        raise ValueError(f"group {group} does not divide K={K}")
    return group


def unpack_gptq(qweight: np.ndarray) -> np.ndarray:
    """GPTQ "NT" qweight int32 ``[K/8, N]`` -> codes uint8 ``[K, N]``.

    [INC] class docstring / ``apply_weights`` (``qweight.shape[1]`` is N) and
    [ZEN] ``_zentorch_woq_eligible`` (GPTQ packs 8 values per int32 along the
    input dim). Nibble j of word i (bits 4j..4j+3) is input row 8i + j; this
    is the little-endian byte stream of [ZEN] ``_maybe_process_da8w4_weights``
    with the low nibble first as in [OMNI] ``pack_nibbles``.
    """
    w = np.asarray(qweight).view(np.uint32)
    kb, n = w.shape
    out = np.empty((kb * 8, n), dtype=np.uint8)
    for j in range(8):
        out[j::8, :] = ((w >> np.uint32(4 * j)) & np.uint32(0xF)).astype(np.uint8)
    return out


def unpack_ct(qweight: np.ndarray) -> np.ndarray:
    """Compressed-tensors packed weight int32 ``[..., N, K/8]`` -> codes ``[..., N, K]``
    ([ZEN] ``_zentorch_woq_eligible``: ``input_dim == packed_dim == 1``)."""
    w = np.asarray(qweight).view(np.uint32)
    out = np.empty(w.shape[:-1] + (w.shape[-1] * 8,), dtype=np.uint8)
    for j in range(8):
        out[..., j::8] = ((w >> np.uint32(4 * j)) & np.uint32(0xF)).astype(np.uint8)
    return out


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[OMNI] ``pack_nibbles``: codes ``[N, K]`` in 0..15 -> uint8 ``[N, K/2]``,
    byte j = w[2j] | w[2j+1] << 4."""
    c = np.asarray(codes).astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << np.uint8(4))).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """[OMNI] ``unpack_nibbles``: uint8 ``[N, K/2]`` -> codes ``[N, K]``."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty((p.shape[0], p.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = p & 0x0F
    out[:, 1::2] = p >> 4
    return out


def repack_signed_int4_to_uint4b8(packed_s4: np.ndarray) -> np.ndarray:
    """[FP8] ``_repack_signed_int4_to_uint4b8``: signed int4 packed two per
    int8 -> ``uint4b8`` packed eight per int32, by XOR 0x88 on every byte
    (adds 8 mod 16 to both nibbles), then a reinterpretation as int32."""
    b = np.ascontiguousarray(packed_s4).view(np.uint8) ^ np.uint8(0x88)
    return b.view(np.int32)


# ---------------------------------------------------------------------------
# per-token activation quantization
# ---------------------------------------------------------------------------

def _activations_f32(x) -> np.ndarray:
    """Activations as float32 (exact): bf16 bit patterns (uint16), or fp16
    values (float16; [INC] class docstring: the activations may be bf16 or
    fp16)."""
    x = np.asarray(x)
    if x.dtype == np.float16:
        return x.astype(np.float32)
    return bf16_bits_to_f32(x)


def quant_int8_per_token(x_bits: np.ndarray):
    """Dynamic per-token symmetric int8 ([INC] class docstring and
    ``apply_weights``: ``dynamic_per_token_int8_quant_ref(x, True, 8)``).

    Returns ``(q int8 [M,K], s float32 [M])`` with, per row,
    ``s = fp32(amax / 127)`` (1 if amax is 0) and
    ``q = clamp(rne(fp32(x / s)), -127, 127)``. ``x_bits``: bf16 bit
    patterns, or a float16 array for fp16 activations.
    """
    x = _activations_f32(x_bits)
    amax = np.max(np.abs(x), axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    s = (amax / np.float32(127.0)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    v = (x / s[:, None]).astype(np.float32)
    q = np.clip(np.rint(v), -127, 127).astype(np.int8)
    return q, s


def quant_fp8_per_token(x_bits: np.ndarray):
    """Dynamic per-token symmetric 8-bit float ([FP8] ``W4AFP8Config.__init__``:
    ``input_quant`` num_bits=8, type float, symmetric, strategy token, dynamic).

    Returns ``(q uint8 e4m3fn codes [M,K], s float32 [M])``:
    ``s = fp32(amax / 448)`` (1 if amax is 0), ``q = e4m3(fp32(x / s))``.
    ``x_bits``: bf16 bit patterns, or a float16 array for fp16 activations.
    """
    x = _activations_f32(x_bits)
    amax = np.max(np.abs(x), axis=1) if x.shape[1] else np.zeros(x.shape[0], np.float32)
    s = (amax / np.float32(448.0)).astype(np.float32)
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    v = (x / s[:, None]).astype(np.float32)
    return e4m3_encode(v), s


# ---------------------------------------------------------------------------
# the linear layers
# ---------------------------------------------------------------------------

def _exact_int_matmul(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """a @ b for integer-valued float64 operands whose every partial sum is an
    integer below 2^53 in magnitude: float64 represents each exactly, so the
    library matmul returns the exact integer product in any summation order."""
    bound = np.max(np.abs(a), initial=0) * np.max(np.abs(b), initial=0) * a.shape[-1]
    assert bound < 2.0 ** 53, "partial sums would leave the exact range of float64"
    return a @ b


def w4a8_group_partials(qx: np.ndarray, qweight: np.ndarray, group: int) -> np.ndarray:
    """Integer group partials of the W4A8 layer, int64 ``[M, G, N]``:
    ``P[m,g,n] = sum_{k in g} qx[m,k] * (code[k,n] - 8)``.

    [INC] ``apply_weights``: int8 activations times the uint4b8 GPTQ weight,
    with scales applied per group ([CT] ``create_weights`` group size rules).
    """
    qx = np.asarray(qx, dtype=np.int8)
    M, K = qx.shape
    g = effective_group(group, K)
    w = unpack_gptq(qweight).astype(np.float64) - 8.0          # [K, N]
    a = qx.astype(np.float64)
    G = K // g
    out = np.empty((M, G, w.shape[1]), dtype=np.int64)
    for gi in range(G):
        sl = slice(gi * g, (gi + 1) * g)
        out[:, gi, :] = _exact_int_matmul(a[:, sl], w[sl, :]).astype(np.int64)
    return out


def w4a8_linear(qx, x_scale, qweight, w_scale_f16, group, bias_bits=None) -> np.ndarray:
    """W4A8 layer output before the bf16 cast, float32 ``[M, N]``:
    ``r = fp32( s_x[m] * sum_g s_w[g,n] * P[m,g,n] + bias[n] )`` in float64.

    [INC] ``apply_weights``: ``int4_gemm_w4a8(quant_x, x_scale, ..., qweight,
    scales_fp16, ..., group_size, ..., bias)``; both scale tensors fp16 per
    the class docstring (here the activation scale stays fp32).
    """
    P = w4a8_group_partials(qx, qweight, group).astype(np.float64)  # [M,G,N]
    sw = np.asarray(w_scale_f16, dtype=np.float16).astype(np.float64)  # [G,N]
    assert sw.shape == P.shape[1:], (sw.shape, P.shape)
    acc = np.einsum("mgn,gn->mn", P, sw)
    r = np.asarray(x_scale, dtype=np.float32).astype(np.float64)[:, None] * acc
    if bias_bits is not None:
        r = r + bf16_to_f64(bias_bits)[None, :]
    return r.astype(np.float32)


def w4a16_linear(x_bits, qweight, w_scale, group, zeros_bits=None, bias_bits=None,
                 scale_dtype: str = "f16") -> np.ndarray:
    """W4A16 layer output before the bf16 cast, float32 ``[M, N]``:
    ``r = fp32( sum_k x[m,k] * ((code[k,n] - 8) * s[g,n] + z[g,n]) + bias[n] )``.

    [INC] class docstring (the W4A16 fallback reads the same GPTQ qweight) and
    [OMNI] module docstring (``w = (q - 8) * scale + zero``). The dequantized
    weight is exact in float64; the contraction is a float64 matmul.
    """
    x = bf16_to_f64(x_bits)
    M, K = x.shape
    g = effective_group(group, K)
    codes = unpack_gptq(qweight).astype(np.float64) - 8.0       # [K, N]
    if scale_dtype == "f16":
        s = np.asarray(w_scale, dtype=np.float16).astype(np.float64)
    elif scale_dtype == "bf16":
        s = bf16_to_f64(w_scale)
    else:
        raise ValueError(scale_dtype)
    s_full = np.repeat(s, g, axis=0)                              # [K, N]
    w = codes * s_full
    if zeros_bits is not None:
        w = w + np.repeat(bf16_to_f64(zeros_bits), g, axis=0)
    r = x @ w
    if bias_bits is not None:
        r = r + bf16_to_f64(bias_bits)[None, :]
    return r.astype(np.float32)


def moe_grouped_linear(qx8, x_scale, offsets, qweight, w_scale_f16, group, rows=None) -> np.ndarray:
    """W4AFP8 grouped expert layer, float32 ``[R, N]`` (or ``[len(rows), N]``).

    [FP8] ``W4AFP8Config``: int4 group-128 routed experts (symmetric), fp8
    per-token dynamic activations; ``get_checkpoint_weight_mapper``: expert
    weights in the compressed-tensors layout ``[E, N, K/8]`` with
    ``weight_scale`` ``[E, N, K/g]`` used as a multiplier. Row r belongs to the
    expert e with ``offsets[e] <= r < offsets[e+1]``:
    ``r = fp32( s_x[r] * sum_g s_w[e,n,g] * sum_{k in g} x8[r,k] * (code[e,n,k] - 8) )``.
    Each product is a multiple of 2^-9 below 2^12 in magnitude, so the float64
    group sums are exact.
    """
    qx8 = np.asarray(qx8, dtype=np.uint8)
    R, K = qx8.shape
    g = effective_group(group, K)
    offsets = np.asarray(offsets, dtype=np.int64)
    E = len(offsets) - 1
    if rows is None:
        rows = np.arange(R)
    rows = np.asarray(rows, dtype=np.int64)
    expert = np.searchsorted(offsets, rows, side="right") - 1
    N = qweight.shape[1]
    out = np.zeros((len(rows), N), dtype=np.float32)
    G = K // g
    for e in range(E):
        sel = np.nonzero(expert == e)[0]
        if len(sel) == 0:
            continue
        xe = e4m3_decode(qx8[rows[sel]])                          # [r, K]
        we = unpack_ct(qweight[e]).astype(np.float64) - 8.0        # [N, K]
        se = np.asarray(w_scale_f16[e], dtype=np.float16).astype(np.float64)  # [N, G]
        acc = np.zeros((len(sel), N))
        for gi in range(G):
            sl = slice(gi * g, (gi + 1) * g)
            acc += (xe[:, sl] @ we[:, sl].T) * se[None, :, gi]
        sx = np.asarray(x_scale, dtype=np.float32)[rows[sel]].astype(np.float64)
        out[sel] = (sx[:, None] * acc).astype(np.float32)
    return out


# ---------------------------------------------------------------------------
# weight-side tools ([OMNI])
# ---------------------------------------------------------------------------

def quantize_groupwise(w: np.ndarray, group: int):
    """[OMNI] ``quantize_groupwise``: asymmetric min/max 4-bit grid on groups
    of ``group`` consecutive input columns of ``w [N, K]``.

    ``scale = max(max - min, 1e-9) / 15``, ``zero = min + 8 * scale``,
    ``q = clamp(round(min-relative / scale), 0, 15)``, in float32 as the page
    does. Returns ``(codes uint8 [N,K], scale f32 [N,G], zero f32 [N,G])``.
    """
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    if k % group:
        raise ValueError(f"input dim {k} is not a multiple of group size {group}")
    wf = w.reshape(n, k // group, group)
    wmin, wmax = wf.min(axis=-1), wf.max(axis=-1)
    scale = (np.maximum(wmax - wmin, np.float32(1e-9)) / np.float32(15.0)).astype(np.float32)
    zero = (wmin + np.float32(8.0) * scale).astype(np.float32)
    q = np.clip(np.rint((wf - wmin[..., None]) / scale[..., None]), 0, 15)
    return q.reshape(n, k).astype(np.uint8), scale, zero


def dequant_rows(codes: np.ndarray, scale: np.ndarray, zero: np.ndarray, group: int) -> np.ndarray:
    """[OMNI] dequantization ``w = (q - 8) * scale + zero`` of rows ``[N, K]``
    (``CPUInt4EmbeddingMethod.embedding`` does this per gathered row), float64."""
    c = np.asarray(codes, dtype=np.float64)
    n, k = c.shape
    s = np.repeat(np.asarray(scale, dtype=np.float64), group, axis=1)
    z = np.repeat(np.asarray(zero, dtype=np.float64), group, axis=1)
    return (c - 8.0) * s + z


def embedding_rows(packed: np.ndarray, scale: np.ndarray, zero: np.ndarray, group: int, ids) -> np.ndarray:
    """[OMNI] ``CPUInt4EmbeddingMethod.embedding``: the rows ``ids`` of the
    packed table ``[V, D/2]`` dequantized in float32, step by step as the page
    does (codes as float32, minus 8, times the row's group scale, plus its
    zero), then rounded to bf16. Returns bf16 bits ``[T, D]``."""
    ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    codes = unpack_nibbles(np.asarray(packed)[ids]).astype(np.float32)
    n, k = codes.shape
    sc = np.asarray(scale, dtype=np.float32)[ids][:, :, None]
    ze = np.asarray(zero, dtype=np.float32)[ids][:, :, None]
    deq = (codes.reshape(n, k // group, group) - np.float32(8.0)) * sc + ze
    return f32_to_bf16_bits(deq.reshape(n, k).astype(np.float32))


def lm_head_logits(h_bits: np.ndarray, packed: np.ndarray, scale: np.ndarray, zero: np.ndarray,
                   group: int) -> np.ndarray:
    """[OMNI] ``CPUInt4EmbeddingMethod.tie_weights``: the output head reads the
    same quantized table, ``logits = h . W^T`` with
    ``W[v, d] = (q - 8) * scale + zero``. Float64 sums of exact float64
    products (a library matmul: the float64 result is the stated precision);
    returns the float32 result ``r`` ``[M, V]``."""
    w = dequant_rows(unpack_nibbles(np.asarray(packed)), scale, zero, group)     # [V, D] float64
    return (bf16_to_f64(h_bits) @ w.T).astype(np.float32)


# ---------------------------------------------------------------------------
# the MoE layer around the grouped GEMM ([FP8] routed experts; readings in the
# module docstring)
# ---------------------------------------------------------------------------

def moe_route(logits: np.ndarray, top_k: int, renormalize: bool):
    """Top-k routing and the expert-sorted row order.

    ``logits`` ``[T, E]`` (float32 values). Per token the k experts are taken
    by a plain selection on the logits themselves (the softmax is monotone, so
    this is its top-k), largest first, equal logits in ascending expert order.
    The weight of a chosen expert is its softmax probability in float64
    (``exp(l - max) / sum exp(l - max)``); with ``renormalize`` the k weights
    are divided by their sum. Rows are the pairs (t, j) listed by expert, then
    by token.

    Returns ``(ids int32 [T,k], weights float32 [T,k], offsets int32 [E+1],
    row_token int32 [T*k], row_of int32 [T,k])``: expert e owns rows
    ``offsets[e] .. offsets[e+1]-1``, ``row_token[r]`` is the token of row r
    and ``row_of[t, j]`` the row of token t's j-th choice.
    """
    lg = np.asarray(logits, dtype=np.float32).astype(np.float64)
    T, E = lg.shape
    ids = np.zeros((T, top_k), dtype=np.int32)
    wts = np.zeros((T, top_k), dtype=np.float32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-lg[t, e], e))[:top_k]
        ex = np.exp(lg[t] - lg[t].max())
        p = ex[order] / ex.sum()
        if renormalize:
            p = p / p.sum()
        ids[t] = order
        wts[t] = p
    counts = np.bincount(ids.reshape(-1), minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    # every (expert, token, choice) triple, listed by expert, then token
    pairs = sorted((int(ids[t, j]), t, j) for t in range(T) for j in range(top_k))
    row_token = np.zeros(T * top_k, dtype=np.int32)
    row_of = np.zeros((T, top_k), dtype=np.int32)
    for r, (_, t, j) in enumerate(pairs):
        row_token[r] = t
        row_of[t, j] = r
    return ids, wts, offsets, row_token, row_of


def moe_gather_quant_fp8(x_bits: np.ndarray, row_token: np.ndarray):
    """The first GEMM's input: row r is token ``row_token[r]`` of ``x`` [T, K],
    quantized per row to e4m3 (``quant_fp8_per_token``)."""
    rows = np.asarray(x_bits)[np.asarray(row_token, dtype=np.int64)]
    return quant_fp8_per_token(rows)


def silu_mul_bf16(h_bits: np.ndarray) -> np.ndarray:
    """``act = silu(gate) * up`` for a gate_up output ``[R, 2I]`` (bf16 bits):
    gate = columns ``[0, I)``, up = ``[I, 2I)``, ``silu(g) = g / (1 + e^-g)``.
    Evaluated in float64, rounded to float32, then to bf16 bits ``[R, I]``."""
    h = bf16_to_f64(h_bits)
    i = h.shape[1] // 2
    g, u = h[:, :i], h[:, i:]
    act = g / (1.0 + np.exp(-g)) * u
    return f32_to_bf16_bits(act.astype(np.float32))


def silu_mul_quant_fp8(h_bits: np.ndarray):
    """The second GEMM's input: ``silu_mul_bf16`` then the per-row e4m3
    quantization. Returns ``(q uint8 [R, I], s float32 [R], act bf16 bits)``."""
    act = silu_mul_bf16(h_bits)
    q, sc = quant_fp8_per_token(act)
    return q, sc, act


def moe_combine(y_bits: np.ndarray, weights: np.ndarray, row_of: np.ndarray) -> np.ndarray:
    """Token outputs ``out[t] = sum_j w[t, j] * y[row_of[t, j]]`` from the
    second GEMM's bf16 rows ``[R, H]``; float64 sums, returned as float32
    ``[T, H]``."""
    y = bf16_to_f64(y_bits)
    w = np.asarray(weights, dtype=np.float32).astype(np.float64)
    ro = np.asarray(row_of, dtype=np.int64)
    T, k = ro.shape
    out = np.zeros((T, y.shape[1]))
    for j in range(k):
        out += w[:, j:j + 1] * y[ro[:, j]]
    return out.astype(np.float32)
