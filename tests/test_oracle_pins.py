"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong rounding mode) fails it.
None of these tests needs a GPU.
"""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle as O
import synthetic as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [p.strip() for p in line.split(";")]


# ---------------------------------------------------------------------------
# layouts
# ---------------------------------------------------------------------------

def test_nibble_golden():
    for codes, packed in _golden_rows("nibble_layout.txt"):
        c = np.array([int(v) for v in codes.split()], dtype=np.uint8)[None, :]
        b = np.array([int(v, 16) for v in packed.split()], dtype=np.uint8)[None, :]
        np.testing.assert_array_equal(O.pack_nibbles(c), b)
        np.testing.assert_array_equal(O.unpack_nibbles(b), c)


def test_nibble_pack_exhaustive():
    """Every (lo, hi) pair: byte = lo | hi << 4, and unpack inverts pack."""
    lo, hi = np.meshgrid(np.arange(16), np.arange(16), indexing="ij")
    codes = np.stack([lo.ravel(), hi.ravel()], axis=1).astype(np.uint8)   # [256, 2]
    packed = O.pack_nibbles(codes)
    np.testing.assert_array_equal(packed[:, 0], (lo.ravel() + 16 * hi.ravel()).astype(np.uint8))
    np.testing.assert_array_equal(O.unpack_nibbles(packed), codes)
    allbytes = np.arange(256, dtype=np.uint8)[:, None]
    np.testing.assert_array_equal(O.pack_nibbles(O.unpack_nibbles(allbytes)), allbytes)


def test_int32_packing_is_the_little_endian_nibble_stream():
    """[ZEN] DA8W4 repack: eight int4 per int32 on little-endian is the same
    byte stream as s4 [N, K/2]. unpack_ct (bit arithmetic on words) must agree
    with unpack_nibbles (bytes, low nibble first) on the byte view."""
    words = S.random_words((5, 6), seed=11)                  # CT [N=5, K/8=6]
    via_words = O.unpack_ct(words)                          # [5, 48]
    via_bytes = O.unpack_nibbles(words.view(np.uint8).reshape(5, 24))
    np.testing.assert_array_equal(via_words, via_bytes)
    # and the word-level bit positions, written out for one word
    w = np.array([[0x76543210]], dtype=np.uint32).view(np.int32)
    np.testing.assert_array_equal(O.unpack_ct(w)[0], np.arange(8, dtype=np.uint8))
    np.testing.assert_array_equal(O.unpack_gptq(w)[:, 0], np.arange(8, dtype=np.uint8))


def test_gptq_and_ct_are_transposes():
    """GPTQ packs along K with K/8 as the row index ([K/8, N]); the
    compressed-tensors layout packs along K inside each output row ([N, K/8]).
    The same codes packed both ways (by a plain loop) must unpack to W and W^T."""
    K, N = 32, 12
    codes = (S.random_words((K, N), seed=12).view(np.uint32) & 0xF).astype(np.uint8)
    gptq = np.zeros((K // 8, N), dtype=np.uint32)
    ct = np.zeros((N, K // 8), dtype=np.uint32)
    for k in range(K):
        for n in range(N):
            gptq[k // 8, n] |= np.uint32(int(codes[k, n]) << (4 * (k % 8)))
            ct[n, k // 8] |= np.uint32(int(codes[k, n]) << (4 * (k % 8)))
    np.testing.assert_array_equal(O.unpack_gptq(gptq.view(np.int32)), codes)
    np.testing.assert_array_equal(O.unpack_ct(ct.view(np.int32)), codes.T)


def test_xor88_golden():
    for signed, s4, u4b8, codes in _golden_rows("xor88_repack.txt"):
        lo, hi = (int(v) for v in signed.split())
        b = np.array([int(s4, 16)] * 4, dtype=np.uint8)
        assert int(b[0]) == ((lo & 0xF) | ((hi & 0xF) << 4))
        out = O.repack_signed_int4_to_uint4b8(b.view(np.int8))
        assert out.dtype == np.int32 and out.shape == (1,)
        assert int(out.view(np.uint8)[0]) == int(u4b8, 16)
        c = O.unpack_ct(out.reshape(1, 1))[0]
        assert [int(c[0]), int(c[1])] == [int(v) for v in codes.split()]
        assert int(c[0]) - 8 == lo and int(c[1]) - 8 == hi


def test_xor88_exhaustive():
    """For every byte: code(b ^ 0x88) - 8 equals the two's-complement int4
    value of each nibble of b (XOR 0x88 is +8 mod 16 on both nibbles)."""
    b = np.arange(256, dtype=np.uint8)
    rep = O.repack_signed_int4_to_uint4b8(np.tile(b, 4).reshape(4, 256).T.copy().view(np.int8))
    codes = O.unpack_nibbles(rep.view(np.uint8).reshape(256, 4))[:, :2].astype(np.int64)
    s_lo = ((b & 0xF).astype(np.int64) ^ 8) - 8
    s_hi = ((b >> 4).astype(np.int64) ^ 8) - 8
    np.testing.assert_array_equal(codes[:, 0] - 8, s_lo)
    np.testing.assert_array_equal(codes[:, 1] - 8, s_hi)


def test_effective_group():
    assert O.effective_group(-1, 4096) == 4096
    assert O.effective_group(128, 4096) == 128
    for bad in (0, -2, 96, 5000):
        with pytest.raises(ValueError):
            O.effective_group(bad, 4096)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def test_bf16_rounding_ties_to_even():
    vals = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 1.0 + 2 ** -8 + 2 ** -20,
                     3.0, 0.0], dtype=np.float32)
    want = np.array([1.0, 1.0 + 2 ** -6, -1.0, 1.0 + 2 ** -7, 3.0, 0.0])
    got = O.bf16_to_f64(O.f32_to_bf16_bits(vals))
    np.testing.assert_array_equal(got, want)


def test_bf16_rounding_matches_torch():
    x = S.normal(7, 1, 100000).astype(np.float32) * np.float32(3.7)
    mine = O.f32_to_bf16_bits(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(mine, theirs)


def test_e4m3_decode_known_values():
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x30: 0.5, 0x50: 8.0, 0x51: 9.0, 0x58: 16.0, 0x59: 18.0, 0x7E: 448.0, 0xFE: -448.0, 0xB8: -1.0}
    for c, v in table.items():
        assert O.e4m3_decode(np.array([c]))[0] == v, hex(c)
    assert np.isnan(O.e4m3_decode(np.array([0x7F, 0xFF]))).all()


def _finite_e4m3_table():
    codes = np.array([c for c in range(128) if c != 0x7F], dtype=np.uint8)
    return codes, O.e4m3_decode(codes)


def test_e4m3_encoder_exhaustive_over_bf16():
    """Every finite bf16 value: the encoder returns the nearest e4m3 value
    (ties to the even code), saturating to 448, with the input's sign."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = O.bf16_to_f64(bits)
    keep = np.isfinite(v)
    bits, v = bits[keep], v[keep]
    got = O.e4m3_encode(v.astype(np.float32))
    codes, vals = _finite_e4m3_table()
    a = np.minimum(np.abs(v), 448.0)
    d = np.abs(a[:, None] - vals[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = np.where(d == best, codes[None, :].astype(np.int64), 1 << 20)
    even = np.where((cand & 1) == 0, cand, 1 << 20).min(axis=1)
    nearest = np.where(even < (1 << 20), even, cand.min(axis=1))
    want = (nearest | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)
    np.testing.assert_array_equal(got, want)


def test_e4m3_encoder_matches_torch_in_range():
    x = np.concatenate([S.normal(3, 2, 50000) * 40.0, S.normal(3, 3, 50000) * 0.01]).astype(np.float32)
    x = x[np.abs(x) <= 448.0]
    mine = O.e4m3_encode(x)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(mine, theirs)


# ---------------------------------------------------------------------------
# per-token quantization
# ---------------------------------------------------------------------------

def _parse_x(xs):
    return O.f32_to_bf16_bits(np.array([float(v) for v in xs.split()], dtype=np.float32))


def test_quant_golden_ties():
    for kind, xs, scale, q in _golden_rows("quant_ties.txt"):
        x = _parse_x(xs)[None, :]
        assert np.array_equal(O.bf16_to_f64(x)[0], [float(v) for v in xs.split()]), "fixture not bf16-exact"
        if kind == "int8":
            got_q, got_s = O.quant_int8_per_token(x)
            np.testing.assert_array_equal(got_q[0], [int(v) for v in q.split()])
        else:
            got_q, got_s = O.quant_fp8_per_token(x)
            np.testing.assert_array_equal(got_q[0], [int(v, 16) for v in q.split()])
        assert got_s[0] == np.float32(float(scale))


def test_quant_int8_invariants():
    x = S.activations_bf16(64, 300, seed=21, outlier_frac=0.02)
    q, s = O.quant_int8_per_token(x)
    xf = O.bf16_to_f64(x)
    amax = np.abs(xf).max(axis=1)
    assert np.all(np.abs(q.astype(np.int64)).max(axis=1) == 127)
    assert np.all(s == (amax.astype(np.float32) / np.float32(127)))
    err = np.abs(xf - q.astype(np.float64) * s[:, None].astype(np.float64))
    assert np.all(err <= s[:, None] * 0.5 * (1 + 2.0 ** -20))


def test_quant_int8_uses_division_not_reciprocal():
    """x / s and x * (1/s) differ on some inputs; the reading is the IEEE
    divide. Find a case where they differ after rounding and check the
    oracle follows the divide."""
    x = S.activations_bf16(256, 512, seed=22)
    q, s = O.quant_int8_per_token(x)
    xf = O.bf16_bits_to_f32(x)
    by_div = np.clip(np.rint((xf / s[:, None]).astype(np.float32)), -127, 127)
    by_mul = np.clip(np.rint((xf * (np.float32(1) / s)[:, None]).astype(np.float32)), -127, 127)
    np.testing.assert_array_equal(q, by_div.astype(np.int8))
    assert np.any(by_div != by_mul), "fixture has no divide/multiply disagreement"


def test_quant_fp8_invariants():
    x = S.activations_bf16(32, 256, seed=23)
    q, s = O.quant_fp8_per_token(x)
    xf = O.bf16_to_f64(x)
    dq = O.e4m3_decode(q) * s[:, None]
    assert np.all(np.abs(O.e4m3_decode(q)).max(axis=1) == 448.0)
    # e4m3 relative spacing is 2^-3: round-to-nearest error <= 2^-4 relative (normals)
    big = np.abs(xf) >= s[:, None] * 2.0 ** -6
    assert np.all(np.abs(dq - xf)[big] <= np.abs(xf)[big] * 2.0 ** -4 * (1 + 1e-6))


def test_quant_fp16_activations():
    """fp16 activations ([INC] class docstring: bf16 or fp16): values that both
    formats hold exactly quantize identically either way; the fp16 extremes
    (65504, the smallest subnormal) quantize by the same rules, 65504 giving
    the row's +-127 / +-448 codes."""
    vals = np.array([[0.5, -3.25, 7.0, 0.0, 1.5, -0.125, 2.0, 96.0]], np.float32)
    for fn in (O.quant_int8_per_token, O.quant_fp8_per_token):
        qa, sa = fn(S.to_bf16_bits(vals))
        qb, sb = fn(vals.astype(np.float16))
        np.testing.assert_array_equal(qa, qb)
        np.testing.assert_array_equal(sa, sb)
    x = np.array([[65504.0, -65504.0, 2.0 ** -24, 1.0, 0, 0, 0, 0]], np.float16)
    q, s = O.quant_int8_per_token(x)
    assert s[0] == np.float32(65504.0) / np.float32(127.0)
    np.testing.assert_array_equal(q[0, :4], [127, -127, 0, 0])
    q8, s8 = O.quant_fp8_per_token(x)
    assert s8[0] == np.float32(65504.0) / np.float32(448.0)
    assert O.e4m3_decode(q8[:, :2]).tolist() == [[448.0, -448.0]]


# ---------------------------------------------------------------------------
# W4A8 layer
# ---------------------------------------------------------------------------

def _gptq_from_codes(codes):
    """[K, N] codes -> GPTQ int32 [K/8, N] by a plain loop (independent of the oracle)."""
    K, N = codes.shape
    out = np.zeros((K // 8, N), dtype=np.uint32)
    for j in range(8):
        out |= codes[j::8, :].astype(np.uint32) << np.uint32(4 * j)
    return out.view(np.int32)


def test_w4a8_codes8_gives_bias():
    M, K, N = 3, 64, 16
    qx = np.random.default_rng(0).integers(-127, 128, (M, K)).astype(np.int8)
    qw = _gptq_from_codes(np.full((K, N), 8, np.uint8))
    sw = S.scales_f16((K // 32, N))
    bias = S.bias_bf16(N)
    r = O.w4a8_linear(qx, np.full(M, 0.5, np.float32), qw, sw, 32, bias)
    np.testing.assert_array_equal(r, np.broadcast_to(O.bf16_to_f64(bias).astype(np.float32), (M, N)))


def test_w4a8_codes9_closed_form():
    M, K, N, g = 4, 128, 8, 32
    rng = np.random.default_rng(1)
    qx = rng.integers(-127, 128, (M, K)).astype(np.int8)
    sx = rng.uniform(0.01, 0.1, M).astype(np.float32)
    qw = _gptq_from_codes(np.full((K, N), 9, np.uint8))
    sw = S.scales_f16((K // g, N))
    r = O.w4a8_linear(qx, sx, qw, sw, g)
    gs = qx.astype(np.int64).reshape(M, K // g, g).sum(axis=2)      # [M, G]
    want = sx.astype(np.float64)[:, None] * (gs.astype(np.float64) @ sw.astype(np.float64))
    np.testing.assert_array_equal(r, want.astype(np.float32))


def test_w4a8_extreme_partial():
    M, K, N = 2, 256, 8
    qx = np.full((M, K), 127, np.int8)
    qx[1] = -127
    qw = _gptq_from_codes(np.zeros((K, N), np.uint8))
    P = O.w4a8_group_partials(qx, qw, 128)
    assert P.shape == (M, 2, N)
    assert np.all(P[0] == -130048) and np.all(P[1] == 130048)


def test_w4a8_group_minus1_equals_K():
    M, K, N = 5, 96, 16
    qx = np.random.default_rng(2).integers(-127, 128, (M, K)).astype(np.int8)
    qw = S.random_words((K // 8, N), seed=3)
    sw = S.scales_f16((1, N))
    sx = np.random.default_rng(3).uniform(0.01, 0.1, M).astype(np.float32)
    a = O.w4a8_linear(qx, sx, qw, sw, -1)
    b = O.w4a8_linear(qx, sx, qw, sw, K)
    np.testing.assert_array_equal(a, b)


def test_w4a8_partials_bruteforce():
    """Group partials against plain Python integer loops on a tiny shape."""
    M, K, N, g = 3, 32, 5, 8
    rng = np.random.default_rng(4)
    qx = rng.integers(-127, 128, (M, K)).astype(np.int8)
    codes = rng.integers(0, 16, (K, N)).astype(np.uint8)
    P = O.w4a8_group_partials(qx, _gptq_from_codes(codes), g)
    for m, gi, n in itertools.product(range(M), range(K // g), range(N)):
        want = sum(int(qx[m, k]) * (int(codes[k, n]) - 8) for k in range(gi * g, gi * g + g))
        assert P[m, gi, n] == want


@pytest.mark.parametrize("group", [8, 16, 32, -1])
def test_w4a8_vs_dequantize_then_matmul(group):
    """The integer-group form equals dequantize-then-multiply
    (sum_k (qx*s_x) * ((q-8)*s_w)), written as Python loops, to 1e-12."""
    M, K, N = 3, 32, 6
    rng = np.random.default_rng(5)
    qx = rng.integers(-127, 128, (M, K)).astype(np.int8)
    codes = rng.integers(0, 16, (K, N)).astype(np.uint8)
    g = K if group == -1 else group
    sw = S.scales_f16((K // g, N), seed=8)
    sx = rng.uniform(0.001, 0.1, M).astype(np.float32)
    bias = S.bias_bf16(N, seed=9)
    r = O.w4a8_linear(qx, sx, _gptq_from_codes(codes), sw, group, bias)
    bf = O.bf16_to_f64(bias)
    for m, n in itertools.product(range(M), range(N)):
        acc = 0.0
        for k in range(K):
            acc += (float(qx[m, k]) * float(sx[m])) * ((int(codes[k, n]) - 8) * float(sw[k // g, n]))
        want = acc + bf[n]
        assert abs(float(r[m, n]) - want) <= 1e-12 * max(1.0, abs(want)) + abs(want) * 2.0 ** -24


# ---------------------------------------------------------------------------
# W4A16 layer
# ---------------------------------------------------------------------------

def test_w4a16_closed_forms():
    M, K, N, g = 2, 64, 8, 32
    x = S.activations_bf16(M, K, seed=30)
    xf = O.bf16_to_f64(x)
    sw = S.scales_f16((K // g, N))
    z = S.zeros_bf16((K // g, N))
    # codes 8: only the zeros act: r = sum_g z[g,n] * sum_{k in g} x
    r8 = O.w4a16_linear(x, _gptq_from_codes(np.full((K, N), 8, np.uint8)), sw, g, zeros_bits=z)
    xs = xf.reshape(M, K // g, g).sum(axis=2)
    np.testing.assert_allclose(r8, xs @ O.bf16_to_f64(z), rtol=1e-6, atol=1e-9)
    # codes 9, no zeros: r = sum_g s[g,n] * sum_{k in g} x
    r9 = O.w4a16_linear(x, _gptq_from_codes(np.full((K, N), 9, np.uint8)), sw, g)
    np.testing.assert_allclose(r9, xs @ sw.astype(np.float64), rtol=1e-6, atol=1e-9)


@pytest.mark.parametrize("scale_dtype", ["f16", "bf16"])
def test_w4a16_bruteforce(scale_dtype):
    M, K, N, g = 2, 32, 4, 16
    rng = np.random.default_rng(6)
    x = S.activations_bf16(M, K, seed=31)
    codes = rng.integers(0, 16, (K, N)).astype(np.uint8)
    if scale_dtype == "f16":
        sw = S.scales_f16((K // g, N))
        sv = sw.astype(np.float64)
    else:
        sw = S.scales_bf16((K // g, N))
        sv = O.bf16_to_f64(sw)
    z = S.zeros_bf16((K // g, N))
    bias = S.bias_bf16(N)
    r = O.w4a16_linear(x, _gptq_from_codes(codes), sw, g, zeros_bits=z, bias_bits=bias,
                       scale_dtype=scale_dtype)
    xf, zf, bf = O.bf16_to_f64(x), O.bf16_to_f64(z), O.bf16_to_f64(bias)
    for m, n in itertools.product(range(M), range(N)):
        want = sum(xf[m, k] * ((int(codes[k, n]) - 8) * sv[k // g, n] + zf[k // g, n]) for k in range(K)) + bf[n]
        assert abs(float(r[m, n]) - want) <= abs(want) * 2.0 ** -23 + 1e-12


def test_bf16_scale_bits_misread_as_fp16():
    """[INC] class docstring: the W4A8 kernel reads scales as fp16, so bf16
    scales are silently misinterpreted. The same 16 bits decode to a
    different value in the other format."""
    sw_bf16 = S.scales_bf16((4, 8))
    as_f16 = sw_bf16.view(np.float16).astype(np.float64)
    as_bf16 = O.bf16_to_f64(sw_bf16)
    assert np.all(as_f16 != as_bf16)


# ---------------------------------------------------------------------------
# W4AFP8 grouped experts
# ---------------------------------------------------------------------------

def _moe_case(E, counts, K, N, g, seed):
    R = int(sum(counts))
    qx8 = S.fp8_codes((R, K), seed=seed)
    sx = np.random.default_rng(seed).uniform(0.001, 0.05, R).astype(np.float32)
    qw = S.random_words((E, N, K // 8), seed=seed + 1)
    sw = S.scales_f16((E, N, K // g), seed=seed + 2)
    return qx8, sx, S.offsets_from_counts(counts), qw, sw


def test_moe_single_expert_bruteforce():
    K, N, g = 32, 4, 16
    qx8, sx, off, qw, sw = _moe_case(1, [3], K, N, g, 40)
    r = O.moe_grouped_linear(qx8, sx, off, qw, sw, g)
    xv = O.e4m3_decode(qx8)
    codes = O.unpack_nibbles(qw[0].view(np.uint8).reshape(N, K // 2))      # [N, K]
    for row, n in itertools.product(range(3), range(N)):
        acc = sum(xv[row, k] * (int(codes[n, k]) - 8) * float(sw[0, n, k // g]) for k in range(K))
        want = float(sx[row]) * acc
        assert abs(float(r[row, n]) - want) <= abs(want) * 2.0 ** -23 + 1e-30


def test_moe_empty_experts_and_permutation():
    K, N, g = 64, 8, 32
    counts = [3, 0, 5, 0, 2]
    qx8, sx, off, qw, sw = _moe_case(5, counts, K, N, g, 50)
    r = O.moe_grouped_linear(qx8, sx, off, qw, sw, g)
    assert r.shape == (10, N)
    # reorder experts: segments move with their expert's weights, results follow
    perm = [2, 4, 0, 3, 1]
    segs = [np.arange(off[e], off[e + 1]) for e in range(5)]
    rows = np.concatenate([segs[e] for e in perm])
    off2 = S.offsets_from_counts([counts[e] for e in perm])
    r2 = O.moe_grouped_linear(qx8[rows], sx[rows], off2, qw[perm], sw[perm], g)
    np.testing.assert_array_equal(r2, r[rows])
    # sampled rows equal the full computation
    sub = np.array([9, 0, 4])
    np.testing.assert_array_equal(O.moe_grouped_linear(qx8, sx, off, qw, sw, g, rows=sub), r[sub])


def test_moe_route_worked_example():
    """tests/golden/moe_route_worked.txt, worked by hand: selection order, the
    tie to the lower expert index, renormalized weights, the expert-then-token
    row order and its inverse."""
    g = {k: v for k, v in _golden_rows("moe_route_worked.txt")}
    lg = np.array([[1, 3, 2, 0], [0, 0, 0, 0], [5, -1, 5, 2]], np.float32)
    ids, w, off, rt, ro = O.moe_route(lg, 2, True)
    np.testing.assert_array_equal(ids.reshape(-1), [int(v) for v in g["ids"].split()])
    np.testing.assert_allclose(w.reshape(-1), [float(v) for v in g["weights"].split()], rtol=1e-7)
    np.testing.assert_array_equal(off, [int(v) for v in g["offsets"].split()])
    np.testing.assert_array_equal(rt, [int(v) for v in g["row_token"].split()])
    np.testing.assert_array_equal(ro.reshape(-1), [int(v) for v in g["row_of"].split()])


@pytest.mark.parametrize("renorm", [False, True])
def test_moe_route_properties(renorm):
    """For random logits: no unchosen expert beats a chosen one; the chosen are
    listed by falling logit; 1 / w equals sum_e exp(l_e - l_chosen) (softmax
    written the other way round), or the k weights sum to 1 with ratios
    exp(l_i - l_j) when renormalized; the rows form a bijection with the
    (token, choice) pairs, sorted by expert, then token."""
    T, E, k = 37, 11, 3
    lg = S.router_logits(T, E, seed=12)
    lg[5, :] = lg[5, 0]                              # a fully tied token
    ids, w, off, rt, ro = O.moe_route(lg, k, renorm)
    l64 = lg.astype(np.float64)
    for t in range(T):
        ch = list(ids[t])
        rest = [e for e in range(E) if e not in ch]
        assert min(lg[t, ch]) >= max(lg[t, rest])
        for a, b in zip(ch, ch[1:]):
            assert lg[t, a] > lg[t, b] or (lg[t, a] == lg[t, b] and a < b)
        if renorm:
            assert abs(w[t].astype(np.float64).sum() - 1.0) < 1e-6
            assert np.allclose(w[t][0] / w[t][1:], np.exp(l64[t, ch[0]] - l64[t, ch[1:]]), rtol=1e-6)
        else:
            inv = np.exp(l64[t][None, :] - l64[t, ch][:, None]).sum(axis=1)
            assert np.allclose(w[t] * inv, 1.0, rtol=1e-6)
    np.testing.assert_array_equal(ids[5], np.arange(k))
    assert off[0] == 0 and off[-1] == T * k
    np.testing.assert_array_equal(np.diff(off), np.bincount(ids.reshape(-1), minlength=E))
    assert sorted(ro.reshape(-1).tolist()) == list(range(T * k))
    for t in range(T):
        for j in range(k):
            r = ro[t, j]
            assert rt[r] == t
            assert off[ids[t, j]] <= r < off[ids[t, j] + 1]
    for e in range(E):
        assert np.all(np.diff(rt[off[e]:off[e + 1]]) > 0)


def test_silu_mul_values_and_halves():
    """silu(g) * u with g from the first half: g = 1, u = 2 gives
    2 / (1 + e^-1) = 1.46211716 (swapped halves would give silu(2) = 1.76);
    silu(0) = 0; silu(20) rounds to 20; and silu(x) - silu(-x) = x."""
    def h(g, u):
        return S.to_bf16_bits(np.array([list(g) + list(u)], np.float32))
    a = S.bf16_bits_to_f32(O.silu_mul_bf16(h([1.0, 0.0, 20.0], [2.0, 5.0, 1.0])))[0]
    assert a[0] == S.bf16_bits_to_f32(S.to_bf16_bits(np.array([1.4621171572600098], np.float32)))[0]
    assert a[1] == 0.0 and a[2] == 20.0
    x = S.bf16_bits_to_f32(S.activations_bf16(1, 64, seed=13))[0]
    pos = S.bf16_bits_to_f32(O.silu_mul_bf16(h(x, np.ones(64))))[0].astype(np.float64)
    neg = S.bf16_bits_to_f32(O.silu_mul_bf16(h(-x, np.ones(64))))[0].astype(np.float64)
    bound = (np.abs(pos) + np.abs(neg)) * 2.0 ** -8
    assert np.all(np.abs(pos - neg - x) <= bound + 1e-30)


def test_silu_mul_quant_round_trip():
    """The requantized activations decode to within half an e4m3 step of the
    bf16 activations, and the row maximum maps to 448."""
    hb = S.activations_bf16(6, 2 * 96, seed=14)
    q, sc, act = O.silu_mul_quant_fp8(hb)
    a = S.bf16_bits_to_f32(act).astype(np.float64)
    d = O.e4m3_decode(q) * sc[:, None].astype(np.float64)
    assert np.all(np.abs(d - a) <= np.abs(a) * 2.0 ** -4 + sc[:, None] * 2.0 ** -9 + 1e-30)
    am = np.abs(a).max(axis=1)
    np.testing.assert_array_equal(np.abs(O.e4m3_decode(q)).max(axis=1), 448.0)
    np.testing.assert_array_equal(sc, (am / 448.0).astype(np.float32))


def test_moe_gather_quant_follows_row_token():
    """Row r is token row_token[r], quantized on its own: repeated tokens give
    identical rows, every nonzero row's largest code is +-448, codes decode to
    within half an e4m3 step of the token, and a token doubled (exact in
    bf16) keeps its codes with twice the scale. A gather along the wrong axis,
    by the wrong index or with a shared scale fails one of these."""
    T, K = 6, 48
    x = S.activations_bf16(T, K, seed=17)
    xf = S.bf16_bits_to_f32(x).astype(np.float64)
    rt = np.array([4, 0, 4, 5, 2, 0, 1], dtype=np.int32)
    q, sc = O.moe_gather_quant_fp8(x, rt)
    assert q.shape == (len(rt), K) and sc.shape == (len(rt),)
    np.testing.assert_array_equal(q[0], q[2])
    np.testing.assert_array_equal(q[1], q[5])
    assert sc[0] == sc[2] and sc[1] == sc[5]
    d = O.e4m3_decode(q)
    np.testing.assert_array_equal(np.abs(d).max(axis=1), 448.0)
    xr = xf[rt]
    assert np.all(np.abs(d * sc[:, None].astype(np.float64) - xr)
                  <= np.abs(xr) * 2.0 ** -4 + sc[:, None] * 2.0 ** -9 + 1e-30)
    x2 = x.copy()
    x2[4] = S.to_bf16_bits((xf[4] * 2.0).astype(np.float32))
    q2, sc2 = O.moe_gather_quant_fp8(x2, rt)
    np.testing.assert_array_equal(q2, q)
    np.testing.assert_array_equal(sc2[[0, 2]], sc[[0, 2]] * np.float32(2.0))
    np.testing.assert_array_equal(np.delete(sc2, [0, 2]), np.delete(sc, [0, 2]))


def test_moe_combine_bruteforce():
    """k = 1 with weight 1 copies y's rows; in general each output element is
    the k-term weighted sum, computed here one element at a time."""
    T, k, H, R = 5, 3, 7, 15
    y = S.activations_bf16(R, H, seed=15)
    ro = np.arange(R, dtype=np.int32)[::-1].reshape(T, k).copy()
    w = S.uniform(16, 1, T * k).reshape(T, k).astype(np.float32)
    out = O.moe_combine(y, w, ro)
    yf = S.bf16_bits_to_f32(y).astype(np.float64)
    for t in range(T):
        for hh in range(H):
            ref = sum(float(w[t, j]) * yf[ro[t, j], hh] for j in range(k))
            assert out[t, hh] == np.float32(ref)
    one = O.moe_combine(y, np.ones((R, 1), np.float32), np.arange(R, dtype=np.int32)[:, None])
    np.testing.assert_array_equal(one, S.bf16_bits_to_f32(y))


# ---------------------------------------------------------------------------
# weight-side tools
# ---------------------------------------------------------------------------

def test_quantize_groupwise_reproduces_extremes():
    """[OMNI] quantize_groupwise: (q-8)*scale+zero reproduces each group's
    min and max (exactly in real arithmetic; to fp32 rounding here)."""
    w = S.normal(8, 1, 16 * 64).reshape(16, 64).astype(np.float32)
    codes, scale, zero = O.quantize_groupwise(w, 32)
    deq = O.dequant_rows(codes, scale, zero, 32)
    g = w.reshape(16, 2, 32)
    d = deq.reshape(16, 2, 32)
    assert np.all(codes.reshape(16, 2, 32).min(axis=2) == 0)
    assert np.all(codes.reshape(16, 2, 32).max(axis=2) == 15)
    np.testing.assert_allclose(d.min(axis=2), g.min(axis=2), rtol=0, atol=4e-6)
    np.testing.assert_allclose(d.max(axis=2), g.max(axis=2), rtol=0, atol=4e-6)
    assert np.all(np.abs(deq - w) <= np.repeat(scale, 32, axis=1) * 0.5 + 1e-6)


def test_embedding_rows_within_the_quantization_error():
    """[OMNI] embedding: a gathered row dequantizes to within half a scale step
    (plus bf16 rounding) of the weights quantize_groupwise was given, and
    each group's extremes come back to within bf16 rounding."""
    V, D, g = 12, 128, 32
    w = (S.normal(3, 4, V * D).reshape(V, D) * 0.2).astype(np.float32)
    q, sc, z = O.quantize_groupwise(w, g)
    ids = [5, 0, 11, 5]
    e = S.bf16_bits_to_f32(O.embedding_rows(O.pack_nibbles(q), sc, z, g, ids)).astype(np.float64)
    ref = w[ids].astype(np.float64)
    step = np.repeat(sc[ids], g, axis=1).astype(np.float64)
    assert np.all(np.abs(e - ref) <= 0.5 * step * (1 + 1e-6) + np.abs(ref) * 2.0 ** -8 + 1e-12)
    for t, v in enumerate(ids):
        for gi in range(D // g):
            blk = slice(gi * g, (gi + 1) * g)
            i_max, i_min = np.argmax(w[v, blk]), np.argmin(w[v, blk])
            assert abs(e[t, blk][i_max] - w[v, blk][i_max]) <= abs(w[v, blk][i_max]) * 2.0 ** -8 + 1e-7
            assert abs(e[t, blk][i_min] - w[v, blk][i_min]) <= abs(w[v, blk][i_min]) * 2.0 ** -8 + 1e-7


def test_lm_head_one_hot_reads_a_table_column():
    """A one-hot h at column d gives logits equal to column d of the
    dequantized table, for every vocabulary row (pins the transposition and
    the group indexing); a constant code 8 table gives logits = sum_d h * zero."""
    V, D, g = 9, 64, 16
    codes = (S.raw_u64(5, 6, V * D) >> np.uint64(60)).astype(np.uint8).reshape(V, D)
    sc = (0.01 + 0.01 * S.uniform(5, 7, V * (D // g))).astype(np.float32).reshape(V, D // g)
    z = (0.1 * S.normal(5, 8, V * (D // g))).astype(np.float32).reshape(V, D // g)
    packed = O.pack_nibbles(codes)
    for d in (0, 17, 63):
        h = np.zeros((1, D), np.float32)
        h[0, d] = 1.0
        r = O.lm_head_logits(S.to_bf16_bits(h), packed, sc, z, g)
        col = (codes[:, d].astype(np.float64) - 8.0) * sc[:, d // g] + z[:, d // g]
        assert np.allclose(r[0], col.astype(np.float32), rtol=0, atol=0)
    h = S.activations_bf16(2, D, seed=9)
    r = O.lm_head_logits(h, O.pack_nibbles(np.full((V, D), 8, np.uint8)), sc, z, g)
    hz = S.bf16_bits_to_f32(h).astype(np.float64).reshape(2, D // g, g).sum(-1)      # [2, G]
    assert np.allclose(r, (hz @ z.astype(np.float64).T).astype(np.float32), rtol=1e-6, atol=1e-7)
