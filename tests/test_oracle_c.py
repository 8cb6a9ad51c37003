"""The plain C statement of the W4A16 layer (oracle/w4_oracle_c.c, the timed
CPU baseline), pinned on the host: against the numpy oracle across shapes,
groups, zeros, bias and scale types; its fp16 scale decoding exhaustively
against numpy's float16; and the all-codes-8 closed form."""
import numpy as np
import pytest

import oracle as O
import synthetic as S
from oracle import c_oracle as C


@pytest.mark.parametrize("M,K,N,group,zeros,bias,sdt", [
    (1, 256, 64, 64, False, False, "f16"), (3, 1024, 200, 128, True, True, "f16"), (8, 512, 136, -1, True, False, "bf16"),
    (2, 2048, 96, 256, False, True, "bf16"), (5, 4096, 40, 128, True, True, "f16")])
def test_c_oracle_matches_numpy_oracle(M, K, N, group, zeros, bias, sdt):
    g = K if group == -1 else group
    x = S.activations_bf16(M, K, seed=M + K)
    qw = S.random_words((K // 8, N), seed=1)
    sw = S.scales_f16((K // g, N), seed=2) if sdt == "f16" else S.scales_bf16((K // g, N), seed=2)
    zb = S.zeros_bf16((K // g, N), seed=3) if zeros else None
    bb = S.bias_bf16(N, seed=4) if bias else None
    a = C.w4a16_linear(x, qw, sw, group, zb, bb, scale_dtype=sdt, nthreads=3)
    b = O.w4a16_linear(x, qw, sw, group, zb, bb, scale_dtype=sdt)
    # both sum in float64 (in different orders) and round once to float32
    np.testing.assert_allclose(a, b, rtol=2.0 ** -22, atol=1e-30)


def test_c_oracle_fp16_scales_exhaustive():
    """x = e_0 and codes 9 at k = 0 (8 elsewhere): r[n] = s[0, n] for every
    finite fp16 bit pattern."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = bits[np.isfinite(bits.view(np.float16))]
    N, K = len(finite), 8
    x = np.zeros((1, K), np.uint16)
    x[0, 0] = 0x3F80                                      # bf16 1.0
    qw = np.full((1, N), 0x88888889, dtype=np.uint32).view(np.int32)   # nibble 0 = 9
    r = C.w4a16_linear(x, qw, finite.view(np.float16).reshape(1, N), 8, nthreads=4)
    np.testing.assert_array_equal(r[0], finite.view(np.float16).astype(np.float32))


def test_c_oracle_codes8_closed_form():
    """All codes 8: r = sum_g z[g] * (sum of x over the group) + bias."""
    M, K, N, g = 2, 512, 48, 128
    x = S.activations_bf16(M, K, seed=9)
    qw = np.full((K // 8, N), 0x88888888, dtype=np.uint32).view(np.int32)
    zb = S.zeros_bf16((K // g, N), seed=3)
    bb = S.bias_bf16(N, seed=4)
    r = C.w4a16_linear(x, qw, S.scales_f16((K // g, N)), g, zb, bb)
    xs = O.bf16_to_f64(x).reshape(M, K // g, g).sum(axis=2)
    want = (xs @ O.bf16_to_f64(zb) + O.bf16_to_f64(bb)).astype(np.float32)
    np.testing.assert_allclose(r, want, rtol=2.0 ** -22)
