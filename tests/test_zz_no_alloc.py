"""The allocation-free W4A8 entry point, through the C ABI.

w4a8_gemm_noalloc serves callers that cannot allocate device memory (code
running inside a framework that owns all device memory, or a plugin that is
handed only its input and output tensors): instead of a caller-provided
workspace it uses one built into the library. Its results must equal those of
w4a8_gemm on the same inputs, call after call, even though every call reuses
(and overwrites) the same built-in workspace.

This file is collected last, so a run that stops at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import int4_weight_quantized_w4_gb300 as w4
import oracle as O
import synthetic as S
from _compare import check_bf16_output
from _gpu import bf16, bits, requires_cuda, to_dev

pytestmark = [pytest.mark.gpu, requires_cuda]


def _inputs(M, N, K, group, seed):
    g = K if group == -1 else group
    xb = S.activations_bf16(M, K, seed=seed, outlier_frac=0.01)
    qx, sx = O.quant_int8_per_token(xb)
    return (xb, to_dev(qx), to_dev(sx), to_dev(S.random_words((K // 8, N), seed=seed + 1)),
            to_dev(S.scales_f16((K // g, N), seed=seed + 2)), bf16(S.bias_bf16(N, seed=seed + 3)))


def _call_noalloc(lib, qx, sx, qw, sw, group, bias, y):
    M, K = qx.shape
    N = qw.shape[1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.w4a8_gemm_noalloc(ctypes.c_void_p(qx.data_ptr()), ctypes.c_void_p(sx.data_ptr()),
                                 ctypes.c_void_p(qw.data_ptr()), ctypes.c_void_p(sw.data_ptr()), w4.W4_FP16, group,
                                 ctypes.c_void_p(bias.data_ptr()), ctypes.c_void_p(y.data_ptr()), M, N, K, stream)


def test_noalloc_matches_w4a8_gemm_twice_in_a_row():
    lib = w4.load()
    # two different problems back to back: the second reuses the workspace the
    # first one filled, so stale contents would show up as a mismatch. Both
    # entry points run the same kernels on the same inputs, so their outputs
    # must agree bit for bit; both are also held to the oracle's bar.
    for (M, N, K, group, seed) in [(300, 264, 1024, 128, 1), (517, 392, 3072, -1, 2)]:
        xb, qx, sx, qw, sw, bias = _inputs(M, N, K, group, seed)
        y = torch.full((M, N), -7.0, dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(lib, qx, sx, qw, sw, group, bias, y) == w4.W4_OK, lib.w4_last_error()
        ref = w4.w4a8_gemm(qx, sx, qw, sw, group, bias=bias)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bits(y), bits(ref), err_msg=f"noalloc vs w4a8_gemm M={M} K={K}")
        r = O.w4a8_linear(qx.cpu().numpy(), sx.cpu().numpy(), qw.cpu().numpy(), sw.cpu().numpy(), group,
                          bits(bias))
        check_bf16_output(bits(y), r, f"noalloc vs oracle M={M} K={K}")
    assert w4.w4_device_status() == w4.W4_OK


def test_noalloc_rejects_problems_beyond_its_workspace():
    lib = w4.load()
    M, N, K = 4097, 128, 4096          # M * K just above 16,777,216
    qx = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    sx = torch.ones((M,), device="cuda")
    qw = torch.zeros((K // 8, N), dtype=torch.int32, device="cuda")
    sw = torch.ones((K // 128, N), dtype=torch.float16, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = lib.w4a8_gemm_noalloc(ctypes.c_void_p(qx.data_ptr()), ctypes.c_void_p(sx.data_ptr()),
                               ctypes.c_void_p(qw.data_ptr()), ctypes.c_void_p(sw.data_ptr()), w4.W4_FP16, 128,
                               None, ctypes.c_void_p(y.data_ptr()), M, N, K, None)
    assert st == w4.W4_ERR_UNSUPPORTED
    assert b"at most 16777216" in lib.w4_last_error()
