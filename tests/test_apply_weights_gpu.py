"""The per-call path choice of the INC W4A8 linear method (below 512 tokens
the W4A16 GEMM, from 512 up the per-token int8 W4A8 GEMM), through the Python
binding's ``apply_weights`` and the C ABI, against the oracle."""
import numpy as np
import pytest
import torch

import int4_weight_quantized_w4_gb300 as w4
import oracle as O
import synthetic as S
from _compare import check_bf16_output
from _gpu import bf16, bits, requires_cuda, to_dev

pytestmark = [pytest.mark.gpu, requires_cuda]

K, N, G = 512, 384, 128


def _weights():
    qw = S.random_words((K // 8, N), seed=1)
    sw = S.scales_f16((K // G, N), seed=2)
    return qw, sw


@pytest.mark.parametrize("shape", [(16,), (2, 8), (600,), (3, 200)])
def test_apply_weights_bf16_paths(shape):
    """16 tokens (W4A16) and 600 tokens (W4A8), as 1-D and 2-D token shapes."""
    M = int(np.prod(shape))
    xb = S.activations_bf16(M, K, seed=M)
    qw, sw = _weights()
    y = w4.apply_weights(bf16(xb).reshape(*shape, K), to_dev(qw), to_dev(sw), G)
    torch.cuda.synchronize()
    assert tuple(y.shape) == (*shape, N)
    if M >= w4.MIN_TOKENS_FOR_INT8:
        q, s = O.quant_int8_per_token(xb)
        r = O.w4a8_linear(q, s, qw, sw, G)
    else:
        r = O.w4a16_linear(xb, qw, sw, G)
    check_bf16_output(bits(y.reshape(M, N)), r, f"apply_weights {shape}")


def test_apply_weights_fp16_and_zeros():
    """fp16 activations take the int8 path at any token count; zeros keep even
    600 tokens on the W4A16 path."""
    qw, sw = _weights()
    xh = S.bf16_bits_to_f32(S.activations_bf16(20, K, seed=5)).astype(np.float16)
    y = w4.apply_weights(torch.from_numpy(xh).cuda(), to_dev(qw), to_dev(sw), G)
    xb = S.activations_bf16(600, K, seed=6)
    zb = S.to_bf16_bits(0.01 * S.normal(3, 1, (K // G) * N).reshape(K // G, N))
    yz = w4.apply_weights(bf16(xb), to_dev(qw), to_dev(sw), G, zeros=bf16(zb))
    torch.cuda.synchronize()
    q, s = O.quant_int8_per_token(xh)
    check_bf16_output(bits(y), O.w4a8_linear(q, s, qw, sw, G), "fp16 activations")
    check_bf16_output(bits(yz), O.w4a16_linear(xb, qw, sw, G, zeros_bits=zb), "zeros at 600 tokens")
