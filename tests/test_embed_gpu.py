"""Quantized embedding gather and the tied output head on the GPU against the
oracle, through the C ABI, on one shared table."""
import numpy as np
import pytest
import torch

import int4_weight_quantized_w4_gb300 as w4
import oracle as O
import synthetic as S
from _compare import check_bf16_output
from _gpu import bf16, bits, requires_cuda, to_dev

pytestmark = [pytest.mark.gpu, requires_cuda]


def _table(V, D, g, seed):
    w = S.normal(seed, 95, V * D).reshape(V, D) * 0.02
    q, sc, z = O.quantize_groupwise(w.astype(np.float32), g)
    return O.pack_nibbles(q), sc, z


@pytest.mark.parametrize("V,D,g", [(1000, 512, 128), (77, 64, 8), (300, 256, -1)])
def test_embedding_gather_bit_exact(V, D, g):
    gg = D if g == -1 else g
    packed, sc, z = _table(V, D, gg, seed=V)
    ids = np.array([0, V - 1, 3, 3, V // 2, 1], dtype=np.int32)
    out = w4.w4_embedding_gather(to_dev(ids), to_dev(packed), to_dev(sc), to_dev(z), g)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), O.embedding_rows(packed, sc, z, gg, ids))


def test_embedding_gather_bad_id_gives_zeros_and_status():
    V, D, g = 64, 64, 32
    packed, sc, z = _table(V, D, g, seed=1)
    assert w4.w4_device_status() == w4.W4_OK
    out = w4.w4_embedding_gather(to_dev(np.array([2, V, -1], np.int32)), to_dev(packed), to_dev(sc), to_dev(z), g)
    assert w4.w4_device_status() == w4.W4_ERR_SHAPE
    b = bits(out)
    assert np.array_equal(b[0], O.embedding_rows(packed, sc, z, g, [2])[0])
    assert not b[1:].any()


@pytest.mark.parametrize("M", [1, 3, 8, 11])
def test_lm_head_small(M):
    V, D, g = 1000, 512, 128
    packed, sc, z = _table(V, D, g, seed=M + 2)
    h = S.activations_bf16(M, D, seed=M)
    y = w4.w4_lm_head_gemv(bf16(h), to_dev(packed), to_dev(sc), to_dev(z), g)
    torch.cuda.synchronize()
    check_bf16_output(bits(y), O.lm_head_logits(h, packed, sc, z, g), f"lm_head M={M}")


@pytest.mark.parametrize("V,D,g,M", [(77, 64, 8, 2), (333, 96, 16, 5), (250, 5792, 32, 8), (129, 2048, -1, 1),
                                     (4099, 1024, 64, 4)])
def test_lm_head_shapes(V, D, g, M):
    """Groups of 8 and 16 codes (several groups per 16-byte chunk), a whole
    row as one group, the longest row the head takes, and vocabularies that
    do not fill the last warp's stride."""
    gg = D if g == -1 else g
    packed, sc, z = _table(V, D, gg, seed=V + D)
    h = S.activations_bf16(M, D, seed=V)
    y = w4.w4_lm_head_gemv(bf16(h), to_dev(packed), to_dev(sc), to_dev(z), g)
    torch.cuda.synchronize()
    check_bf16_output(bits(y), O.lm_head_logits(h, packed, sc, z, gg), f"lm_head V={V} D={D} g={g} M={M}")


@pytest.mark.parametrize("V,D,g,M", [(37, 8192, 256, 9), (48, 1024, 512, 8), (17, 256, -1, 2)])
def test_lm_head_tensor_core_shapes(V, D, g, M):
    """The tensor-core form: a group spanning several 128-code segments, the
    longest row it takes, two passes of tokens (9 = 8 + 1), a row as one
    group, and whole vs. partial 16-row tiles."""
    gg = D if g == -1 else g
    packed, sc, z = _table(V, D, gg, seed=V * 3 + D)
    h = S.activations_bf16(M, D, seed=V + 1)
    y = w4.w4_lm_head_gemv(bf16(h), to_dev(packed), to_dev(sc), to_dev(z), g)
    torch.cuda.synchronize()
    check_bf16_output(bits(y), O.lm_head_logits(h, packed, sc, z, gg), f"lm_head tc V={V} D={D} g={g} M={M}")


@pytest.mark.parametrize("V,D,g,M", [(4099, 1152, 128, 1), (37, 8192, 256, 1), (48, 1024, 512, 1), (17, 256, 256, 1),
                                     (161, 640, 128, 1), (3000, 768, 384, 1), (2500, 2048, 128, 1),
                                     (1, 128, 128, 1), (15, 8192, -1, 1), (2433, 1920, 128, 2), (4099, 1280, 256, 5)])
def test_lm_head_tensor_core_split_tiles(V, D, g, M):
    """Tiles shared by several warps of a CTA (every CTA's run of tiles is
    cut into equal runs of segments), for one token (eight segments to a
    window of MMA columns: 9, 5, 15 and 6 segments leave a partial window;
    scale groups of 2, 3 and 4 segments; 64 segments cut mid-window by 24
    warps; a one-row table of one segment; a row as one scale group) and for
    several tokens."""
    gg = D if g == -1 else g
    packed, sc, z = _table(V, D, gg, seed=V + D)
    h = S.activations_bf16(M, D, seed=V * 7 + M)
    y = w4.w4_lm_head_gemv(bf16(h), to_dev(packed), to_dev(sc), to_dev(z), g)
    torch.cuda.synchronize()
    check_bf16_output(bits(y), O.lm_head_logits(h, packed, sc, z, gg), f"lm_head split V={V} D={D} g={g} M={M}")


def test_lm_head_one_token_wide_range_h():
    """One token whose segments differ by up to 2^40 in magnitude, with an
    all-zero segment: each segment keeps its own power of two in its MMA
    column."""
    V, D, g = 2000, 1024, 128
    packed, sc, z = _table(V, D, g, seed=79)
    hf = S.bf16_bits_to_f32(S.activations_bf16(1, D, seed=80)).astype(np.float64).reshape(1, D // 128, 128)
    hf *= 2.0 ** np.array([-20, 0, 20, 7, -13, 0, 3, -1])[None, :, None]
    hf[0, 5] = 0.0
    h = S.to_bf16_bits(hf.reshape(1, D).astype(np.float32))
    y = w4.w4_lm_head_gemv(bf16(h), to_dev(packed), to_dev(sc), to_dev(z), g)
    torch.cuda.synchronize()
    check_bf16_output(bits(y), O.lm_head_logits(h, packed, sc, z, g), "lm_head one token wide-range h")


def test_lm_head_wide_range_h():
    """h whose 128-code segments differ by up to 2^40 in magnitude (and one
    all-zero segment): the per-segment power-of-two staging keeps every
    segment exact."""
    V, D, g, M = 300, 1024, 128, 3
    packed, sc, z = _table(V, D, g, seed=77)
    hf = S.bf16_bits_to_f32(S.activations_bf16(M, D, seed=78)).astype(np.float64).reshape(M, D // 128, 128)
    hf *= 2.0 ** np.array([-20, 0, 20, 7, -13, 0, 3, -1])[None, :, None]
    hf[1, 5] = 0.0
    h = S.to_bf16_bits(hf.reshape(M, D).astype(np.float32))
    y = w4.w4_lm_head_gemv(bf16(h), to_dev(packed), to_dev(sc), to_dev(z), g)
    torch.cuda.synchronize()
    check_bf16_output(bits(y), O.lm_head_logits(h, packed, sc, z, g), "lm_head wide-range h")


def test_tied_table_full_size():
    """131072 x 2048 group 128: the head for one token, checked on every 7th
    vocabulary row, and a gather of 8 ids from the same tensors."""
    V, D, g = 131072, 2048, 128
    blk = _table(4096, D, g, seed=31)
    packed = np.tile(blk[0], (V // 4096, 1))
    sc, z = np.tile(blk[1], (V // 4096, 1)), np.tile(blk[2], (V // 4096, 1))
    pk_d, sc_d, z_d = to_dev(packed), to_dev(sc), to_dev(z)
    h = S.activations_bf16(1, D, seed=3)
    y = w4.w4_lm_head_gemv(bf16(h), pk_d, sc_d, z_d, g)
    ids = np.array([0, 1, 4095, 4096, 70000, 131071, 5, 5], np.int32)
    e = w4.w4_embedding_gather(to_dev(ids), pk_d, sc_d, z_d, g)
    torch.cuda.synchronize()
    rows = np.arange(0, V, 7)
    check_bf16_output(bits(y)[:, rows], O.lm_head_logits(h, packed[rows], sc[rows], z[rows], g), "lm_head full")
    assert np.array_equal(bits(e), O.embedding_rows(packed, sc, z, g, ids))
