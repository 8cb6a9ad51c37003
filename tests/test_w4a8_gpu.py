"""W4A8 GEMM on the GPU (tcgen05 path) against the oracle, through the C ABI:
integer group partials bit-exact, bf16 outputs within tolerance."""
import numpy as np
import pytest
import torch

import int4_weight_quantized_w4_gb300 as w4
import oracle as O
import synthetic as S
from _compare import check_bf16_output
from _gpu import bf16, bits, requires_cuda, to_dev

pytestmark = [pytest.mark.gpu, requires_cuda]


def _inputs(M, N, K, group, seed, outliers=0.0):
    g = K if group == -1 else group
    xb = S.activations_bf16(M, K, seed=seed, outlier_frac=outliers)
    qx, sx = O.quant_int8_per_token(xb)
    qw = S.random_words((K // 8, N), seed=seed + 1)
    sw = S.scales_f16((K // g, N), seed=seed + 2)
    return xb, qx, sx, qw, sw


@pytest.mark.parametrize("M,N,K,group", [(16, 256, 256, 128), (1, 128, 64, 16), (130, 200, 512, 64),
                                         (7, 136, 1024, 16), (33, 128, 2048, -1), (129, 384, 4096, 128),
                                         (200, 264, 1408, 128), (5, 72, 48, 48)])
def test_w4a8_partials_bit_exact(M, N, K, group):
    _, qx, _, qw, _ = _inputs(M, N, K, group, seed=M + N)
    P = w4.w4a8_group_partials(to_dev(qx), to_dev(qw), group)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(P.cpu().numpy(), O.w4a8_group_partials(qx, qw, group))


def test_w4a8_partials_more_tiles_than_sms():
    """2176 x 2600 at K = 384: 9 x 21 = 189 tiles of 256 x 128 for 152 SMs, so
    some persistent CTAs take two tiles (both ragged in M and N); bit-exact."""
    M, N, K, group = 2176, 2600, 384, 128
    _, qx, _, qw, _ = _inputs(M, N, K, group, seed=77)
    P = w4.w4a8_group_partials(to_dev(qx), to_dev(qw), group)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(P.cpu().numpy(), O.w4a8_group_partials(qx, qw, group))


def test_w4a8_partials_extremes():
    """|P| = 127 * 8 * group at the extreme codes: 130048 at group 128, and the
    largest exact case, group 16384."""
    for K, group in ((256, 128), (16384, -1)):
        M, N = 3, 128
        qx = np.full((M, K), 127, np.int8)
        qx[1] = -127
        qx[2, ::2] = -127
        qw = np.zeros((K // 8, N), np.int32)
        P = w4.w4a8_group_partials(to_dev(qx), to_dev(qw), group)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(P.cpu().numpy(), O.w4a8_group_partials(qx, qw, group))


@pytest.mark.parametrize("M,N,K,group,bias", [(16, 256, 256, 128, False), (16, 256, 256, 128, True),
                                              (130, 200, 512, 64, True), (7, 136, 1024, 16, False),
                                              (33, 128, 2048, -1, True), (257, 392, 3072, -1, False),
                                              (300, 520, 4096, 128, True)])
def test_w4a8_outputs(M, N, K, group, bias):
    _, qx, sx, qw, sw = _inputs(M, N, K, group, seed=3 * M + K, outliers=0.01)
    bb = S.bias_bf16(N, seed=7) if bias else None
    y = w4.w4a8_gemm(to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw), group, bias=None if bb is None else bf16(bb))
    torch.cuda.synchronize()
    check_bf16_output(bits(y), O.w4a8_linear(qx, sx, qw, sw, group, bb), f"w4a8 M={M} N={N} K={K} g={group}")


@pytest.mark.parametrize("M,N,K,group", [(70, 264, 1088, 64), (300, 520, 4160, 64), (40, 136, 2048, 512),
                                         (260, 392, 1280, 256)])
def test_w4a8_stage_paths(M, N, K, group):
    """Whole k-stages whose accumulations change only at the stage's start or
    middle run without per-MMA checks; a tile's ragged last stage and other
    groups take the checked loop. Groups of 64 (two per stage) with a half
    stage left over at the end (K = 1088, 4160), and groups spanning several
    stages (512 over four, 256 over two with a K of ten stages)."""
    _, qx, sx, qw, sw = _inputs(M, N, K, group, seed=M + K, outliers=0.01)
    y = w4.w4a8_gemm(to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw), group)
    torch.cuda.synchronize()
    check_bf16_output(bits(y), O.w4a8_linear(qx, sx, qw, sw, group), f"w4a8 stages M={M} N={N} K={K} g={group}")


def test_w4a8_layer_from_bf16():
    """The whole W4A8 layer: per-token int8 quantization then the GEMM, both on
    the GPU, against the oracle's quantizer and GEMM (16 tokens, K=N=256, g128)."""
    M, N, K, g = 16, 256, 256, 128
    xb = S.activations_bf16(M, K, seed=0)
    qw = S.random_words((K // 8, N), seed=1)
    sw = S.scales_f16((K // g, N), seed=2)
    q, s = w4.w4_quant_act_per_token(bf16(xb), "int8")
    y = w4.w4a8_gemm(q, s, to_dev(qw), to_dev(sw), g)
    torch.cuda.synchronize()
    qr, sr = O.quant_int8_per_token(xb)
    check_bf16_output(bits(y), O.w4a8_linear(qr, sr, qw, sw, g), "w4a8 layer")


def test_w4a8_codes8_gives_bias():
    M, N, K = 64, 128, 256
    qx = np.random.default_rng(0).integers(-127, 128, (M, K)).astype(np.int8)
    qw = np.full((K // 8, N), 0x88888888, dtype=np.uint32).view(np.int32)
    bb = S.bias_bf16(N)
    y = w4.w4a8_gemm(to_dev(qx), to_dev(np.ones(M, np.float32)), to_dev(qw), to_dev(S.scales_f16((2, N))), 128,
                     bias=bf16(bb))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(y), np.broadcast_to(bb, (M, N)))


def test_w4a8_group_minus1_equals_group_K():
    M, N, K = 40, 128, 512
    _, qx, sx, qw, sw = _inputs(M, N, K, -1, seed=9)
    a = w4.w4a8_gemm(to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw), -1)
    b = w4.w4a8_gemm(to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw), K)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_w4a8_output_guard_and_empty():
    M, N, K = 20, 136, 256
    _, qx, sx, qw, sw = _inputs(M, N, K, 128, seed=4)
    buf = torch.full((M * N + 512,), -7.0, dtype=torch.bfloat16, device="cuda")
    y = buf[256:256 + M * N].view(M, N)
    w4.w4a8_gemm(to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw), 128, y=y)
    torch.cuda.synchronize()
    assert torch.all(buf[:256] == -7.0) and torch.all(buf[256 + M * N:] == -7.0)
    e = w4.w4a8_gemm(torch.empty((0, K), dtype=torch.int8, device="cuda"), torch.empty((0,), device="cuda"),
                     to_dev(qw), to_dev(sw), 128)
    assert e.shape == (0, N)
    assert w4.w4_device_status() == w4.W4_OK


@pytest.mark.parametrize("M,N", [(4096, 11008), (512, 4096)])
def test_w4a8_full_size_prefill(M, N):
    """K=4096, group 128, 1% outlier channels x20; sampled rows against the oracle."""
    K, g = 4096, 128
    xb, qx, sx, qw, sw = _inputs(M, N, K, g, seed=0, outliers=0.01)
    y = w4.w4a8_gemm(to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw), g)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // 48)), [M - 1]]))
    check_bf16_output(bits(y)[rows], O.w4a8_linear(qx[rows], sx[rows], qw, sw, g), f"prefill {M}x{N}")


def test_w4a8_full_size_diffusion():
    """M=16384, K=N=3072, per-channel scales (group -1); sampled rows."""
    M, N, K = 16384, 3072, 3072
    xb, qx, sx, qw, sw = _inputs(M, N, K, -1, seed=1)
    y = w4.w4a8_gemm(to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw), -1)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, M, 331), [M - 1]]))
    check_bf16_output(bits(y)[rows], O.w4a8_linear(qx[rows], sx[rows], qw, sw, -1), "diffusion")


def test_bounded_wait_selftest():
    """A wait that nothing completes runs out, records W4_ERR_TIMEOUT and the
    context stays usable."""
    assert w4.w4_device_status() == w4.W4_OK
    w4.w4_selftest_bounded_wait(1 << 12)
    assert w4.w4_device_status() == w4.W4_ERR_TIMEOUT
    assert w4.w4_device_status() == w4.W4_OK
    x = torch.ones(4, 4, device="cuda")
    assert float((x + x).sum()) == 32.0


@pytest.mark.parametrize("M,N,K,group,outliers", [(16, 256, 256, 128, 0.0), (300, 384, 1024, 128, 0.01),
                                                  (77, 136, 512, -1, 0.0), (1, 128, 4096, 64, 0.01)])
def test_w4a8_bf16in_equals_quant_then_gemm(M, N, K, group, outliers):
    """Quantization fused into the GEMM's activation pass: same scales and the
    same output bits as w4_quant_act_per_token followed by w4a8_gemm, and the
    oracle's result within tolerance."""
    g = K if group == -1 else group
    xb = S.activations_bf16(M, K, seed=M + K, outlier_frac=outliers)
    qw = S.random_words((K // 8, N), seed=M + 1)
    sw = S.scales_f16((K // g, N), seed=M + 2)
    bb = S.bias_bf16(N, seed=M + 3)
    x, qw_d, sw_d, b_d = bf16(xb), to_dev(qw), to_dev(sw), bf16(bb)
    y_f, s_f = w4.w4a8_gemm_bf16in(x, qw_d, sw_d, group, bias=b_d)
    q, s = w4.w4_quant_act_per_token(x, "int8")
    y_u = w4.w4a8_gemm(q, s, qw_d, sw_d, group, bias=b_d)
    torch.cuda.synchronize()
    assert np.array_equal(s_f.cpu().numpy().view(np.uint32), s.cpu().numpy().view(np.uint32))
    assert np.array_equal(bits(y_f), bits(y_u))
    qr, sr = O.quant_int8_per_token(xb)
    check_bf16_output(bits(y_f), O.w4a8_linear(qr, sr, qw, sw, group, bias_bits=bb), f"bf16in M={M}")


@pytest.mark.parametrize("M,N,K,group,outliers", [(4096, 11008, 4096, 128, 0.01), (16384, 3072, 3072, -1, 0.0)])
def test_w4a8_bf16in_full_size(M, N, K, group, outliers):
    """The fused quantize + GEMM entry point at the sizes the bench times: the
    prefill shape (K=4096, group 128, 1% outlier channels x20) and the
    diffusion shape (per-channel scales). Per-token scales bit-exact on every
    row; outputs on sampled rows (every column) against the oracle's quantizer
    and GEMM at the parity bar."""
    g = K if group == -1 else group
    xb = S.activations_bf16(M, K, seed=0, outlier_frac=outliers)
    qw = S.random_words((K // 8, N), seed=1)
    sw = S.scales_f16((K // g, N), seed=2)
    y, sx = w4.w4a8_gemm_bf16in(bf16(xb), to_dev(qw), to_dev(sw), group)
    torch.cuda.synchronize()
    qr, sr = O.quant_int8_per_token(xb)
    np.testing.assert_array_equal(sx.cpu().numpy().view(np.uint32), sr.view(np.uint32))
    rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // 40)), [1, M - 2, M - 1]]))
    check_bf16_output(bits(y)[rows], O.w4a8_linear(qr[rows], sr[rows], qw, sw, group),
                      f"bf16in full size {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,group,bias", [(300, 10240, 2048, 128, True), (700, 6656, 2048, 64, False),
                                              (1000, 5120, 2048, -1, True)])
def test_w4a8_last_wave_split(M, N, K, group, bias):
    """Shapes whose last wave of tiles would leave most SMs idle (160, 156 and
    160 tiles on 152 SMs): the whole waves run as tiles, the last wave's 8, 4
    and 8 tiles in 8 K parts each, whose fp32 sums a reduce pass adds. The
    split tiles are the last ones, in the last, ragged row tile. Outputs on
    every row of that tile and on rows of the whole tiles, against the oracle;
    the same call with only the minimal workspace (unsplit) likewise."""
    _, qx, sx, qw, sw = _inputs(M, N, K, group, seed=M + K, outliers=0.01)
    bb = S.bias_bf16(N, seed=5) if bias else None
    args = (to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw), group)
    kw = {} if bb is None else {"bias": bf16(bb)}
    assert w4.w4_workspace_bytes(w4.W4_OP_W4A8, M, N, K, group) > M * K * 2, "this shape should be split"
    y_split = w4.w4a8_gemm(*args, **kw)
    ws_min = torch.empty((M * K * 2,), dtype=torch.uint8, device="cuda")
    y_one = w4.w4a8_gemm(*args, workspace=ws_min, **kw)
    torch.cuda.synchronize()
    last = (M - 1) // 256 * 256
    rows = np.unique(np.concatenate([np.arange(0, last, 37), np.arange(last, M)]))
    r = O.w4a8_linear(qx[rows], sx[rows], qw, sw, group, bb)
    check_bf16_output(bits(y_split)[rows], r, f"last-wave split M={M} N={N} K={K} g={group}")
    check_bf16_output(bits(y_one)[rows], r, f"unsplit M={M} N={N} K={K} g={group}")
    assert w4.w4_device_status() == w4.W4_OK


@pytest.mark.parametrize("M,N,K,group,bias", [(300, 264, 2048, 128, True), (100, 136, 3072, -1, False),
                                              (33, 128, 1536, 48, True), (512, 4096, 4096, 128, False)])
def test_w4a8_split_k(M, N, K, group, bias):
    """Shapes whose output tiles fill the SMs poorly run split along K (the
    workspace w4_workspace_bytes asks for holds the parts' fp32 sums): 4 parts
    for the first two, 2 for the last two (the group of 48 cuts on 384-k
    boundaries). The same call with only the minimal workspace runs unsplit.
    Both against the oracle."""
    _, qx, sx, qw, sw = _inputs(M, N, K, group, seed=M + K, outliers=0.01)
    bb = S.bias_bf16(N, seed=5) if bias else None
    args = (to_dev(qx), to_dev(sx), to_dev(qw), to_dev(sw), group)
    kw = {} if bb is None else {"bias": bf16(bb)}
    full = w4.w4_workspace_bytes(w4.W4_OP_W4A8, M, N, K, group)
    assert full > M * K * 2, "this shape should be split"
    y_split = w4.w4a8_gemm(*args, **kw)
    ws_min = torch.empty((M * K * 2,), dtype=torch.uint8, device="cuda")
    y_one = w4.w4a8_gemm(*args, workspace=ws_min, **kw)
    torch.cuda.synchronize()
    r = O.w4a8_linear(qx, sx, qw, sw, group, bb)
    check_bf16_output(bits(y_split), r, f"split M={M} N={N} K={K} g={group}")
    check_bf16_output(bits(y_one), r, f"unsplit M={M} N={N} K={K} g={group}")
    assert w4.w4_device_status() == w4.W4_OK
