"""The routed MoE layer around the grouped GEMM on the GPU against the oracle,
through the C ABI: routing and the row order, the gathered fp8 input, the
fused gather + GEMM, SiLU(gate)*up with fp8 requantization, the combine, and
a whole layer end to end."""
import numpy as np
import pytest
import torch

import int4_weight_quantized_w4_gb300 as w4
import oracle as O
import synthetic as S
from _compare import check_bf16_output
from _gpu import bf16, bits, requires_cuda, to_dev

pytestmark = [pytest.mark.gpu, requires_cuda]


def _logits(T, E, seed, dtype):
    lg = S.router_logits(T, E, seed=seed)
    if dtype == "bf16":
        b = S.to_bf16_bits(lg)
        return bf16(b), S.bf16_bits_to_f32(b)
    return to_dev(lg), lg


def _route_check(T, E, k, renorm, dtype, seed, tie_rows=()):
    lg_d, lg = _logits(T, E, seed, dtype)
    for t in tie_rows:                         # fully tied tokens: lowest indices win
        lg[t, :] = lg[t, 0]
    if tie_rows:
        lg_d = bf16(S.to_bf16_bits(lg)) if dtype == "bf16" else to_dev(lg)
    ids, wts, off, rt, ro = w4.w4_moe_route(lg_d, k, renorm)
    torch.cuda.synchronize()
    r_ids, r_w, r_off, r_rt, r_ro = O.moe_route(lg, k, renorm)
    np.testing.assert_array_equal(ids.cpu().numpy(), r_ids)
    np.testing.assert_array_equal(off.cpu().numpy(), r_off)
    np.testing.assert_array_equal(rt.cpu().numpy(), r_rt)
    np.testing.assert_array_equal(ro.cpu().numpy(), r_ro)
    np.testing.assert_allclose(wts.cpu().numpy(), r_w, rtol=2e-5, atol=1e-9)


@pytest.mark.parametrize("T,E,k,renorm,dtype", [
    (100, 64, 8, False, "f32"), (1000, 60, 6, True, "f32"), (37, 1, 1, False, "f32"), (300, 256, 8, True, "bf16"),
    (513, 1024, 64, False, "f32"), (257, 33, 33, True, "bf16"), (1, 8, 2, True, "f32")])
def test_route_matches_oracle(T, E, k, renorm, dtype):
    """ids, offsets, row order and its inverse bit-exact; weights to fp32
    rounding. bf16 logits tie often, so the lower-index rule is exercised."""
    _route_check(T, E, k, renorm, dtype, seed=T + E, tie_rows=(0,) if T > 1 else ())


def test_route_full_size():
    """4096 tokens, 64 experts, top-8: the MoE workload's routing."""
    _route_check(4096, 64, 8, False, "f32", seed=5)


def test_gather_quant_bit_exact_and_bad_row():
    T, K = 50, 264
    x = S.activations_bf16(T, K, seed=21)
    x[7] = 0                                   # a zero row: scale 1, all codes 0
    rows = np.array([3, 3, 49, 0, 7, 12, 12, 12], np.int32)
    q, s = w4.w4_moe_gather_quant_fp8(bf16(x), to_dev(rows))
    torch.cuda.synchronize()
    rq, rs = O.moe_gather_quant_fp8(x, rows)
    np.testing.assert_array_equal(q.view(torch.uint8).cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy(), rs)
    assert w4.w4_device_status() == w4.W4_OK
    q, s = w4.w4_moe_gather_quant_fp8(bf16(x), to_dev(np.array([1, T, -2], np.int32)))
    assert w4.w4_device_status() == w4.W4_ERR_SHAPE
    qb = q.view(torch.uint8).cpu().numpy()
    np.testing.assert_array_equal(qb[0], O.moe_gather_quant_fp8(x, [1])[0][0])
    assert not qb[1:].any() and np.all(s.cpu().numpy()[1:] == 1.0)


def test_gather_quant_many_rows_and_bad_rows():
    """Enough gathered rows for the warp-per-row form (R x K >= 2^22), with
    repeated tokens and two ids outside [0, T) among them."""
    T, K, R = 1000, 2048, 2100
    x = S.activations_bf16(T, K, seed=22)
    rows = (S.raw_u64(23, 5, R) % T).astype(np.int32)
    rows[5], rows[R - 1] = T, -1
    q, s = w4.w4_moe_gather_quant_fp8(bf16(x), to_dev(rows))
    torch.cuda.synchronize()
    assert w4.w4_device_status() == w4.W4_ERR_SHAPE
    qb, sb = q.view(torch.uint8).cpu().numpy(), s.cpu().numpy()
    good = np.ones(R, bool)
    good[[5, R - 1]] = False
    rq, rs = O.moe_gather_quant_fp8(x, rows[good])
    np.testing.assert_array_equal(qb[good], rq)
    np.testing.assert_array_equal(sb[good], rs)
    assert not qb[~good].any() and np.all(sb[~good] == 1.0)


@pytest.mark.parametrize("T,E,k,N,K,g", [(64, 8, 2, 256, 256, 128), (200, 16, 4, 384, 512, -1)])
def test_moe_gemm_bf16in_equals_gather_then_gemm(T, E, k, N, K, g):
    """The fused gather + quant + GEMM is bit-identical to the two-step path,
    and matches the oracle."""
    x = S.activations_bf16(T, K, seed=T)
    _, _, off, rt, _ = w4.w4_moe_route(to_dev(S.router_logits(T, E, seed=E)), k)
    qw = S.random_words((E, N, K // 8), seed=1)
    sw = S.scales_f16((E, N, K // (K if g == -1 else g)), seed=2)
    y, sx = w4.w4afp8_moe_gemm_bf16in(bf16(x), rt, off, to_dev(qw), to_dev(sw), g)
    q2, s2 = w4.w4_moe_gather_quant_fp8(bf16(x), rt)
    y2 = w4.w4afp8_moe_grouped_gemm(q2, s2, off, to_dev(qw), to_dev(sw), g)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(y), bits(y2))
    np.testing.assert_array_equal(sx.cpu().numpy(), s2.cpu().numpy())
    _, _, r_off, r_rt, _ = O.moe_route(S.router_logits(T, E, seed=E), k, False)
    rq, rs = O.moe_gather_quant_fp8(x, r_rt)
    r = O.moe_grouped_linear(rq, rs, r_off, qw, sw, g)
    check_bf16_output(bits(y), r, "moe_gemm_bf16in")


def test_moe_gemm_bf16in_without_gather():
    T, E, N, K, g = 96, 3, 128, 256, 128
    x = S.activations_bf16(T, K, seed=8)
    off = S.offsets_from_counts([40, 0, 56])
    qw = S.random_words((E, N, K // 8), seed=1)
    sw = S.scales_f16((E, N, K // g), seed=2)
    y, _ = w4.w4afp8_moe_gemm_bf16in(bf16(x), None, to_dev(off), to_dev(qw), to_dev(sw), g)
    torch.cuda.synchronize()
    rq, rs = O.quant_fp8_per_token(x)
    check_bf16_output(bits(y), O.moe_grouped_linear(rq, rs, off, qw, sw, g), "moe_gemm_bf16in rows as tokens")


def _act_check(h, what):
    """SiLU(gate)*up then the per-row e4m3 requantization, against the oracle.

    The activations come from a fast fp32 exponential and divide on the GPU
    and from fp64 in the oracle, so they are held to >= 99.9% bit-equal and
    every one within one bf16 step. The requantization is a pure function of
    the GPU's own bf16 activations, so its codes and row scales are held
    bit-exact: the oracle's per-token e4m3 quantizer applied to the GPU's act
    must give the GPU's (q, scale) on every element. Returns the GPU's
    (q, scale, act) as numpy arrays."""
    R, I2 = h.shape
    I = I2 // 2
    act = torch.empty((R, I), dtype=torch.bfloat16, device="cuda")
    q, s = w4.w4_moe_silu_mul_quant_fp8(bf16(h), act=act)
    torch.cuda.synchronize()
    _, _, ract = O.silu_mul_quant_fp8(h)
    a = bits(act)
    av, rav = S.bf16_bits_to_f32(a).astype(np.float64), S.bf16_bits_to_f32(ract).astype(np.float64)
    same = a == ract
    assert same.mean() >= 0.999, f"{what}: only {same.mean():.5f} of activations bit-equal"
    assert np.all(np.abs(av - rav) <= np.abs(rav) * 2.0 ** -7 + 1e-38), f"{what}: activation off by > 1 bf16 ulp"
    sg, qg = s.cpu().numpy(), q.view(torch.uint8).cpu().numpy()
    oq, osc = O.quant_fp8_per_token(a)
    np.testing.assert_array_equal(sg.view(np.uint32), osc.view(np.uint32), err_msg=f"{what}: row scales")
    np.testing.assert_array_equal(qg, oq, err_msg=f"{what}: e4m3 codes")
    return qg, sg, a


@pytest.mark.parametrize("R,I", [(300, 1408), (5, 8), (9, 512), (6, 768), (5, 1024), (7, 2048), (17, 2056),
                                 (3, 5000), (2, 8192), (3, 8200), (65536, 64), (8200, 512), (6000, 704),
                                 (4097, 1024), (2979, 1408), (2049, 2048)])
def test_silu_mul_quant(R, I):
    """Row lengths for each chunk count of the CTA-per-row form and, with many
    rows (R x I >= 2^22, I <= 2048), of the warp-per-row form; row counts that
    leave part of a CTA empty; the long-row path."""
    h = S.activations_bf16(R, 2 * I, seed=R + I)
    _act_check(h, f"silu R={R} I={I}")


def test_silu_mul_quant_edge_values():
    """Gates far below zero (silu -> -0), a zero row (scale 1, codes 0), large
    gates (silu(g) = g), and gates from -100 to -60 (tiny activations, down
    into the fp32 subnormals)."""
    R, I = 4, 64
    h = S.activations_bf16(R, 2 * I, seed=3)
    gf = S.bf16_bits_to_f32(h).copy()
    gf[0, :I] = -200.0
    gf[1, :] = 0.0
    gf[2, :I] = 90.0
    gf[3, :I] = np.linspace(-100.0, -60.0, I)
    _act_check(S.to_bf16_bits(gf), "silu edges")


@pytest.mark.parametrize("T,k,H", [(100, 8, 2048), (7, 1, 64), (33, 3, 136)])
def test_combine(T, k, H):
    R = T * k
    y = S.activations_bf16(R, H, seed=T)
    ro = np.argsort(S.raw_u64(T, 9, R), kind="stable").astype(np.int32).reshape(T, k)   # a seeded permutation
    w = S.uniform(T, 3, T * k).reshape(T, k).astype(np.float32)
    out = w4.w4_moe_combine(bf16(y), to_dev(w), to_dev(ro))
    torch.cuda.synchronize()
    check_bf16_output(bits(out), O.moe_combine(y, w, ro), f"combine T={T} k={k}")


def test_combine_bad_row_sets_status():
    y = S.activations_bf16(4, 16, seed=1)
    ro = np.array([[0, 9], [3, 1]], np.int32)
    w = np.array([[0.5, 0.5], [0.25, 0.75]], np.float32)
    assert w4.w4_device_status() == w4.W4_OK
    out = w4.w4_moe_combine(bf16(y), to_dev(w), to_dev(ro))
    assert w4.w4_device_status() == w4.W4_ERR_SHAPE
    r = O.moe_combine(y, np.array([[0.5, 0.0], [0.25, 0.75]], np.float32), np.array([[0, 0], [3, 1]], np.int32))
    check_bf16_output(bits(out), r, "combine with a bad row")


def test_moe_layer_end_to_end():
    """route -> gather + gate_up GEMM -> SiLU*up + requant -> down GEMM ->
    combine, every stage held to its full bar against the oracle run on the
    previous stage's GPU output (each stage's inputs are identical on both
    sides): routing and the gathered fp8 input bit-exact, both GEMM outputs and
    the combine at the bf16 parity bar, the requantized activations through
    _act_check (codes and scales bit-exact)."""
    T, E, k, Hd, I, g = 128, 8, 2, 256, 128, 128
    lg = S.router_logits(T, E, seed=31)
    x = S.activations_bf16(T, Hd, seed=32)
    w1 = S.random_words((E, 2 * I, Hd // 8), seed=1, tag=40)
    s1 = S.scales_f16((E, 2 * I, Hd // g), seed=2, tag=41)
    w2 = S.random_words((E, Hd, I // 8), seed=1, tag=42)
    s2 = S.scales_f16((E, Hd, I // g), seed=2, tag=43)
    ids, wts, off, rt, ro = w4.w4_moe_route(to_dev(lg), k, True)
    h1, sx1 = w4.w4afp8_moe_gemm_bf16in(bf16(x), rt, off, to_dev(w1), to_dev(s1), g)
    torch.cuda.synchronize()

    r_ids, r_w, r_off, r_rt, r_ro = O.moe_route(lg, k, True)
    for got, ref, nm in ((ids, r_ids, "ids"), (off, r_off, "offsets"), (rt, r_rt, "row_token"), (ro, r_ro, "row_of")):
        np.testing.assert_array_equal(got.cpu().numpy(), ref, err_msg=f"layer routing: {nm}")
    np.testing.assert_allclose(wts.cpu().numpy(), r_w, rtol=2e-5, atol=1e-9)
    rq, rs = O.moe_gather_quant_fp8(x, r_rt)
    np.testing.assert_array_equal(sx1.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    check_bf16_output(bits(h1), O.moe_grouped_linear(rq, rs, r_off, w1, s1, g), "layer gate_up")

    # the second GEMM's input from the GPU's own gate_up output
    qa, sa, _ = _act_check(bits(h1), "layer act")
    qa_d = to_dev(qa).view(torch.float8_e4m3fn)
    y2 = w4.w4afp8_moe_grouped_gemm(qa_d, to_dev(sa), off, to_dev(w2), to_dev(s2), g)
    torch.cuda.synchronize()
    check_bf16_output(bits(y2), O.moe_grouped_linear(qa, sa, r_off, w2, s2, g), "layer down")

    # the combine from the GPU's own down output and routing weights
    out = w4.w4_moe_combine(y2, wts, ro)
    torch.cuda.synchronize()
    check_bf16_output(bits(out), O.moe_combine(bits(y2), wts.cpu().numpy(), r_ro), "layer combine")


def test_moe_gemm_bf16in_full_size():
    """The fused gather + fp8 quant + gate_up GEMM as the MoE layer times it:
    4096 tokens, 64 experts, top-8 (32768 rows), K=2048, N=2816, group 128.
    Row scales bit-exact on every row; outputs on sampled rows (every column,
    including each expert segment's first and last row) at the parity bar."""
    T, E, top, N, K, g = 4096, 64, 8, 2816, 2048, 128
    lg = S.router_logits(T, E, seed=5)
    x = S.activations_bf16(T, K, seed=0)
    qw = S.random_words((E, N, K // 8), seed=1)
    sw = S.scales_f16((E, N, K // g), seed=2)
    _, _, off, rt, _ = w4.w4_moe_route(to_dev(lg), top, True)
    y, sx = w4.w4afp8_moe_gemm_bf16in(bf16(x), rt, off, to_dev(qw), to_dev(sw), g)
    torch.cuda.synchronize()
    _, _, r_off, r_rt, _ = O.moe_route(lg, top, True)
    np.testing.assert_array_equal(off.cpu().numpy(), r_off)
    np.testing.assert_array_equal(rt.cpu().numpy(), r_rt)
    rq, rs = O.moe_gather_quant_fp8(x, r_rt)
    np.testing.assert_array_equal(sx.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    R = T * top
    rows = np.unique(np.concatenate([np.arange(0, R, 101), r_off[1:-1] - 1, r_off[1:-1], [R - 1]]))
    rows = rows[(rows >= 0) & (rows < R)]
    check_bf16_output(bits(y)[rows], O.moe_grouped_linear(rq, rs, r_off, qw, sw, g, rows=rows),
                      "moe gate_up bf16in full size")
