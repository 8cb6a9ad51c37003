"""Per-token activation quantization on the GPU against the oracle, bit-exact
(codes and fp32 scales), through the C ABI."""
import numpy as np
import pytest
import torch

import int4_weight_quantized_w4_gb300 as w4
import oracle as O
import synthetic as S
from _gpu import bf16, requires_cuda

pytestmark = [pytest.mark.gpu, requires_cuda]


def _run(xb, kind):
    q, s = w4.w4_quant_act_per_token(bf16(xb), kind)
    torch.cuda.synchronize()
    q = q.cpu()
    q = q.view(torch.uint8).numpy() if kind == "fp8" else q.numpy()
    return q, s.cpu().numpy()


def _check(xb, kind):
    q, s = _run(xb, kind)
    qr, sr = (O.quant_fp8_per_token if kind == "fp8" else O.quant_int8_per_token)(xb)
    np.testing.assert_array_equal(s.view(np.uint32), sr.view(np.uint32))
    np.testing.assert_array_equal(q, qr)


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("M,K", [(1, 8), (3, 256), (16, 256), (9, 512), (5, 768), (6, 1000), (7, 1408), (33, 2048),
                                 (64, 3072), (5, 4096), (3, 5000), (2, 8192), (9, 8200), (4, 16384), (2, 24)])
def test_quant_parity(kind, M, K):
    """Row lengths for each chunk count of the warp-per-row form (K <= 4096)
    and of the CTA-per-row form (3 and 4 chunks a thread, and longer rows read
    twice), with row counts that leave part of a CTA empty."""
    _check(S.activations_bf16(M, K, seed=M * 7 + K, outlier_frac=0.01), kind)


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("M,K", [(16384, 256), (8200, 512), (5462, 768), (4100, 1024), (2981, 1408), (2049, 2048),
                                 (1366, 3072)])
def test_quant_warp_form(kind, M, K):
    """Many short rows (M x K >= 2^22, K <= 3072) take one warp per row: each
    chunk count of that form, row counts that leave part of a CTA empty."""
    _check(S.activations_bf16(M, K, seed=M + K, outlier_frac=0.01), kind)


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("M,K", [(1300, 5000), (1300, 6144), (1300, 8192), (1300, 4096)])
def test_quant_many_long_rows(kind, M, K):
    """At least 8 rows per SM with rows longer than 3072: one CTA of up to 128
    threads per row, 5 (rounded up to 6), 6, 8 and 4 chunks a thread."""
    _check(S.activations_bf16(M, K, seed=M + K, outlier_frac=0.01), kind)


@pytest.mark.parametrize("kind", ["int8", "fp8"])
def test_quant_special_rows(kind):
    """Zero rows (s = 1), rows whose amax is the code maximum (s = 1, ties at
    x.5), tiny and huge magnitudes, rows whose scale is subnormal, and sign
    mixtures."""
    K = 64
    rows = []
    rows.append(np.zeros(K))
    t = np.zeros(K); t[:8] = [127, 2.5, 3.5, -2.5, 126.5, -127, 0.5, 1.5]; rows.append(t)
    t = np.zeros(K); t[:6] = [448, 17, 19, -17, 0.0625, -448]; rows.append(t)
    rows.append(np.full(K, -3.0e-30))
    rows.append(np.linspace(-1e30, 1e30, K))
    t = np.zeros(K); t[K - 1] = 1e-3; rows.append(t)
    # rows so small that s is subnormal and fl(1 / s) may overflow: the codes
    # are still those of the IEEE quotient x / s
    rng = np.random.default_rng(7)
    rows.append(rng.uniform(-3e-39, 3e-39, K))
    rows.append(rng.uniform(-1e-37, 1e-37, K))
    t = np.zeros(K); t[:4] = [9.2e-41, -4e-40, 1e-39, -1e-39]; rows.append(t)
    t = rng.uniform(-1e-36, 1e-36, K); t[0] = 2e-36; rows.append(t)
    xb = S.to_bf16_bits(np.stack(rows))
    _check(xb, kind)


@pytest.mark.parametrize("kind", ["int8", "fp8"])
def test_quant_full_size_prefill(kind):
    """The prefill activations at full size: 4096 tokens x 4096, 1% outlier channels x20."""
    _check(S.activations_bf16(4096, 4096, seed=0, outlier_frac=0.01), kind)


def test_quant_moe_rows_full_size():
    """The expert down-projection input at full size: 32768 rows x 1408, e4m3."""
    _check(S.activations_bf16(32768, 1408, seed=3), "fp8")


def test_quant_empty():
    q, s = w4.w4_quant_act_per_token(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"), "int8")
    assert q.shape == (0, 64) and s.shape == (0,)


def _check_f16(xh, kind):
    q, s = w4.w4_quant_act_per_token(torch.from_numpy(xh).cuda(), kind)
    torch.cuda.synchronize()
    q = q.cpu()
    q = q.view(torch.uint8).numpy() if kind == "fp8" else q.numpy()
    qr, sr = (O.quant_fp8_per_token if kind == "fp8" else O.quant_int8_per_token)(xh)
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), sr.view(np.uint32))
    np.testing.assert_array_equal(q, qr)


@pytest.mark.parametrize("kind", ["int8", "fp8"])
@pytest.mark.parametrize("M,K", [(3, 256), (33, 2048), (5, 4096), (9, 8200), (2049, 2048)])
def test_quant_fp16_activations(kind, M, K):
    """fp16 activations ([INC] class docstring: bf16 or fp16), with the fp16
    extremes in one row: 65504, subnormals, and zeros."""
    x = S.bf16_bits_to_f32(S.activations_bf16(M, K, seed=M + K, outlier_frac=0.01)).astype(np.float16)
    x[0, :4] = [65504.0, -65504.0, 2.0 ** -24, -(2.0 ** -20)]
    if M > 1:
        x[1] = 0
    _check_f16(x, kind)


def _near_boundaries(kind, rows=64, K=4096, seed=3):
    """Rows whose values sit on or next to the quantizer's rounding
    boundaries: the bf16 values nearest to (k + 1/2) s for int8, or to the
    midpoints between neighbouring e4m3 values times s for e4m3, with a row
    maximum that makes s a non-power-of-two (so x / s is not exact)."""
    rng = np.random.default_rng(seed)
    Q = 127.0 if kind == "int8" else 448.0
    out = np.empty((rows, K), np.float32)
    for i in range(rows):
        amax = np.float32(rng.uniform(0.3, 40.0))
        s = np.float32(amax / np.float32(Q))
        if kind == "int8":
            mids = (rng.integers(-127, 127, K) + 0.5) * np.float64(s)
        else:
            vals = np.sort(np.unique(np.abs(O.e4m3_decode(np.arange(256, dtype=np.uint8)))))
            vals = vals[np.isfinite(vals) & (vals <= 448)]
            j = rng.integers(0, len(vals) - 1, K)
            mids = (vals[j] + vals[j + 1]) / 2 * np.sign(rng.standard_normal(K)) * np.float64(s)
        # nudge some by one bf16 step either way so both sides of each boundary occur
        b = S.to_bf16_bits(mids.astype(np.float32))
        nudge = rng.integers(-1, 2, K).astype(np.int32)
        b = (b.astype(np.int32) + nudge * (b != 0)).astype(np.uint16)
        row = S.bf16_bits_to_f32(b)
        row[0] = amax
        out[i] = np.clip(row, -amax, amax)
    return S.to_bf16_bits(out)


@pytest.mark.parametrize("kind", ["int8", "fp8"])
def test_quant_near_rounding_boundaries_bit_exact(kind):
    """The codes come from x * fl(1/s) with the IEEE divide taking over near a
    rounding boundary; on values packed around the boundaries every code and
    scale must still equal the IEEE-quotient codes of the oracle."""
    xb = _near_boundaries(kind)
    q, s = w4.w4_quant_act_per_token(bf16(xb), kind)
    torch.cuda.synchronize()
    if kind == "int8":
        rq, rs = O.quant_int8_per_token(xb)
        np.testing.assert_array_equal(q.cpu().numpy(), rq)
    else:
        rq, rs = O.quant_fp8_per_token(xb)
        np.testing.assert_array_equal(q.view(torch.uint8).cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
