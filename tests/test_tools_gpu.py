"""Weight-side tools on the GPU (group quantizer, XOR 0x88 repack) against
the oracle, through the C ABI; bit-exact."""
import numpy as np
import pytest
import torch

import int4_weight_quantized_w4_gb300 as w4
import oracle as O
import synthetic as S
from _compare import check_bf16_output
from _gpu import bf16, bits, requires_cuda, to_dev

pytestmark = [pytest.mark.gpu, requires_cuda]


def _weights(N, K, seed, spread=False):
    w = S.normal(seed, 90, N * K).reshape(N, K) * 0.05
    if spread:   # groups of very different magnitudes, and constant groups
        w *= 10.0 ** S.normal(seed, 91, N).reshape(N, 1)
        w[:, :32] = 0.125
    return w


def _quant_and_check(wbits_or_half, N, K, group, fp16, label):
    if fp16:
        wt = torch.from_numpy(wbits_or_half).to("cuda")
        wf = wbits_or_half.astype(np.float32)
    else:
        wt = bf16(wbits_or_half)
        wf = S.bf16_bits_to_f32(wbits_or_half)
    packed, scale, zero = w4.w4_quantize_groupwise(wt, group)
    torch.cuda.synchronize()
    q_ref, s_ref, z_ref = O.quantize_groupwise(wf, K if group == -1 else group)
    assert np.array_equal(packed.cpu().numpy(), O.pack_nibbles(q_ref)), f"{label}: codes"
    assert np.array_equal(scale.cpu().numpy().view(np.uint32), s_ref.view(np.uint32)), f"{label}: scales"
    assert np.array_equal(zero.cpu().numpy().view(np.uint32), z_ref.view(np.uint32)), f"{label}: zeros"
    return packed, scale, zero


@pytest.mark.parametrize("group", [2, 8, 16, 32, 64, 128, 256, 512, -1])
def test_quantize_groupwise_bf16(group):
    N, K = 96, 512
    _quant_and_check(S.to_bf16_bits(_weights(N, K, seed=group % 7)), N, K, group, False, f"bf16 g={group}")


def test_quantize_groupwise_fp16_and_spread():
    N, K = 40, 256
    w = _weights(N, K, seed=3, spread=True).astype(np.float16)
    _quant_and_check(w, N, K, 64, True, "fp16 spread")
    _quant_and_check(S.to_bf16_bits(_weights(N, K, seed=4, spread=True)), N, K, 32, False, "bf16 spread")


@pytest.mark.parametrize("N,K,group", [(7, 200, 8), (5, 48, 16), (3, 776, 8), (9, 264, 24)])
def test_quantize_groupwise_ragged(N, K, group):
    """Chunk counts that leave the last block partly empty, and a group of 24
    (not a power of two: one warp per group)."""
    _quant_and_check(S.to_bf16_bits(_weights(N, K, seed=K)), N, K, group, False, f"ragged {N}x{K} g={group}")


def test_quantize_groupwise_ties():
    """Quotients on and next to half-integers: groups with min 0 and max 15
    (scale exactly 1) holding k + 0.5 (ties to even) and k + 0.5 +- 1/16, and
    groups with max 1 (scale fl(1/15)) holding bf16 values next to
    (k + 0.5) / 15, where the fast reciprocal product must hand over to the
    IEEE quotient."""
    N, K, g = 8, 256, 32
    w = np.zeros((N, K), np.float32)
    for n in range(N):
        for j in range(K // g):
            blk = np.zeros(g, np.float32)
            blk[1] = 15.0 if n % 2 == 0 else 1.0
            for i in range(2, g):
                k = (i + j + n) % 15
                if n % 2 == 0:
                    blk[i] = k + 0.5 + ((i % 3) - 1) / 16.0
                else:
                    blk[i] = (k + 0.5) / 15.0
            w[n, j * g:(j + 1) * g] = blk
    _quant_and_check(S.to_bf16_bits(w), N, K, g, False, "ties")


def test_quantize_groupwise_edges():
    _quant_and_check(S.to_bf16_bits(np.array([[0.5, -0.25]])), 1, 2, -1, False, "1x2")
    _quant_and_check(S.to_bf16_bits(np.zeros((3, 64))), 3, 64, 64, False, "all zeros")


def test_quantize_groupwise_full_size():
    N, K = 14336, 4096
    _quant_and_check(S.to_bf16_bits(_weights(N, K, seed=11)), N, K, 128, False, "full size")


@pytest.mark.parametrize("nbytes", [1, 15, 16, 1000, 4096 * 37 + 5])
def test_repack_s4_to_uint4b8(nbytes):
    src = (S.raw_u64(8, 80, nbytes) >> np.uint64(56)).astype(np.uint8)
    out = w4.w4_repack_s4_to_uint4b8(to_dev(src))
    torch.cuda.synchronize()
    ref = O.repack_signed_int4_to_uint4b8(np.concatenate([src, np.zeros((-nbytes) % 4, np.uint8)])).view(np.uint8)
    assert np.array_equal(out.cpu().numpy(), ref[:nbytes])


def test_repack_in_place_expert_layout():
    """[E, N, K/2] signed pairs -> [E, N, K/8] int32 uint4b8, in place."""
    E, N, K = 4, 64, 256
    s4 = (S.raw_u64(9, 81, E * N * K // 2) >> np.uint64(56)).astype(np.uint8).reshape(E, N, K // 2)
    t = to_dev(s4)
    w4.w4_repack_s4_to_uint4b8(t, dst=t)
    torch.cuda.synchronize()
    assert np.array_equal(t.cpu().numpy().view(np.int32), O.repack_signed_int4_to_uint4b8(s4))


def test_quantized_weights_drive_w4a16():
    """bf16 W [N, K] -> GPU group quantizer -> GPTQ qweight + bf16 scales and
    zeros (layout glue on the host) -> w4a16_gemm, against the oracle on the
    same packed weights: the quantizer's (q - 8) * scale + zero grid is the
    GEMM's asymmetric rule."""
    N, K, g, M = 512, 1024, 128, 3
    wb = S.to_bf16_bits(_weights(N, K, seed=21))
    packed, scale, zero = w4.w4_quantize_groupwise(bf16(wb), g)
    torch.cuda.synchronize()
    codes = O.unpack_nibbles(packed.cpu().numpy()).astype(np.uint32)           # [N, K]
    qw = np.zeros((K // 8, N), dtype=np.uint32)
    for j in range(8):
        qw |= codes[:, j::8].T << np.uint32(4 * j)
    sw = S.to_bf16_bits(scale.cpu().numpy().T)                                   # [G, N] bf16
    zb = S.to_bf16_bits(zero.cpu().numpy().T)
    xb = S.activations_bf16(M, K, seed=5)
    y = w4.w4a16_gemm(bf16(xb), to_dev(qw.view(np.int32)), bf16(sw), g, zeros=bf16(zb))
    torch.cuda.synchronize()
    check_bf16_output(bits(y), O.w4a16_linear(xb, qw.view(np.int32), sw, g, zeros_bits=zb, scale_dtype="bf16"),
                      "quantized weights through w4a16")
