"""W4AFP8 grouped expert GEMM on the GPU against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import int4_weight_quantized_w4_gb300 as w4
import oracle as O
import synthetic as S
from _compare import check_bf16_output
from _gpu import bf16, bits, requires_cuda, to_dev

pytestmark = [pytest.mark.gpu, requires_cuda]


def _run(qx8, sx, off, qw, sw, group):
    y = w4.w4afp8_moe_grouped_gemm(to_dev(qx8), to_dev(sx), to_dev(off), to_dev(qw), to_dev(sw), group)
    torch.cuda.synchronize()
    return bits(y)


def _case(counts, N, K, group, seed):
    E = len(counts)
    R = int(sum(counts))
    g = K if group == -1 else group
    xb = S.activations_bf16(R, K, seed=seed)
    qx8, sx = O.quant_fp8_per_token(xb)
    qw = S.random_words((E, N, K // 8), seed=seed + 1)
    sw = S.scales_f16((E, N, K // g), seed=seed + 2)
    return qx8, sx, S.offsets_from_counts(counts), qw, sw


@pytest.mark.parametrize("counts,N,K,group", [([3, 0, 130, 17], 136, 256, 128), ([1], 128, 64, 32),
                                              ([300, 5, 0, 0, 129], 256, 512, -1), ([64] * 8, 192, 1408, 128)])
def test_moe_small(counts, N, K, group):
    qx8, sx, off, qw, sw = _case(counts, N, K, group, seed=len(counts) + N)
    y = _run(qx8, sx, off, qw, sw, group)
    check_bf16_output(y, O.moe_grouped_linear(qx8, sx, off, qw, sw, group), f"moe {counts}")


@pytest.mark.parametrize("counts,N,K,group", [([5, 0, 40], 128, 32, 32), ([5, 0, 40], 128, 32, -1),
                                              ([17, 3], 136, 96, 32), ([64] * 8, 192, 384, 128),
                                              ([33, 100], 128, 384, 48), ([9, 250], 256, 1024, 16),
                                              ([70, 260], 136, 1280, 256)])
def test_moe_stage_edges(counts, N, K, group):
    """Expert tiles against the 128-k stages: K shorter than one stage (32,
    96: most of the stage's MMAs skipped, a packed-word copy narrower than a
    slot), an odd stage count whose last copy is half used (384), groups
    that close inside a stage (48, 16), and groups of exactly one 256-k e4m3
    stage (K = 1280, five stages)."""
    qx8, sx, off, qw, sw = _case(counts, N, K, group, seed=len(counts) + K)
    y = _run(qx8, sx, off, qw, sw, group)
    check_bf16_output(y, O.moe_grouped_linear(qx8, sx, off, qw, sw, group), f"moe edges {counts} K={K} g={group}")


def test_moe_routed_layer_from_bf16():
    """Seeded top-8 routing of 64 tokens over 16 experts; fp8 quantization on
    the GPU, then the grouped GEMM, against the oracle's quantizer and GEMM."""
    T, E, top, N, K, g = 64, 16, 8, 256, 512, 128
    _, _, off, tok, _ = O.moe_route(S.router_logits(T, E, seed=5), top, False)
    x_tok = S.activations_bf16(T, K, seed=0)
    xb = x_tok[tok]
    qw = S.random_words((E, N, K // 8), seed=1)
    sw = S.scales_f16((E, N, K // g), seed=2)
    q, s = w4.w4_quant_act_per_token(bf16(xb), "fp8")
    y = w4.w4afp8_moe_grouped_gemm(q, s, to_dev(off), to_dev(qw), to_dev(sw), g)
    torch.cuda.synchronize()
    qr, sr = O.quant_fp8_per_token(xb)
    check_bf16_output(bits(y), O.moe_grouped_linear(qr, sr, off, qw, sw, g), "routed layer")


def test_moe_rows_outside_segments_untouched():
    """Rows past offsets[E] are never written."""
    counts, N, K = [5, 9], 128, 256
    qx8, sx, off, qw, sw = _case(counts, N, K, 128, seed=3)
    R = 20                                   # 6 extra rows that belong to no expert
    qx_pad = np.zeros((R, K), np.uint8); qx_pad[:14] = qx8
    sx_pad = np.ones(R, np.float32); sx_pad[:14] = sx
    y = torch.full((R, N), -7.0, dtype=torch.bfloat16, device="cuda")
    w4.w4afp8_moe_grouped_gemm(to_dev(qx_pad), to_dev(sx_pad), to_dev(off), to_dev(qw), to_dev(sw), 128, y=y)
    torch.cuda.synchronize()
    assert torch.all(y[14:] == -7.0)
    check_bf16_output(bits(y[:14]), O.moe_grouped_linear(qx8, sx, off, qw, sw, 128), "padded")


@pytest.mark.parametrize("N,K", [(2816, 2048), (2048, 1408)])
def test_moe_full_size(N, K):
    """4096 tokens, 64 experts, top-8 (32768 rows): the gate_up (K=2048,
    N=2816) and down (K=1408, N=2048) projections; sampled rows."""
    T, E, top, g = 4096, 64, 8, 128
    _, _, off, _, _ = O.moe_route(S.router_logits(T, E, seed=5), top, False)
    R = T * top
    xb = S.activations_bf16(R, K, seed=11 + K)
    qx8, sx = O.quant_fp8_per_token(xb)
    qw = S.random_words((E, N, K // 8), seed=1)
    sw = S.scales_f16((E, N, K // g), seed=2)
    y = _run(qx8, sx, off, qw, sw, g)
    rows = np.unique(np.concatenate([np.arange(0, R, 97), off[1:-1] - 1, off[1:-1], [R - 1]]))
    check_bf16_output(y[rows], O.moe_grouped_linear(qx8, sx, off, qw, sw, g, rows=rows), f"moe full {N}x{K}")
