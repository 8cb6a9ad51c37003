"""W4A16 decode GEMM on the GPU against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import int4_weight_quantized_w4_gb300 as w4
import oracle as O
import synthetic as S
from _compare import check_bf16_output
from _gpu import bf16, bits, requires_cuda, to_dev

pytestmark = [pytest.mark.gpu, requires_cuda]


def _case(M, N, K, group, scale_dtype="f16", zeros=False, bias=False, seed=0, cols=None):
    g = K if group == -1 else group
    xb = S.activations_bf16(M, K, seed=seed)
    qw = S.random_words((K // 8, N), seed=seed + 1)
    sw = S.scales_f16((K // g, N), seed=seed + 2) if scale_dtype == "f16" else S.scales_bf16((K // g, N), seed=seed + 2)
    zb = S.zeros_bf16((K // g, N), seed=seed + 3) if zeros else None
    bb = S.bias_bf16(N, seed=seed + 4) if bias else None
    sw_t = to_dev(sw) if scale_dtype == "f16" else bf16(sw)
    y = w4.w4a16_gemm(bf16(xb), to_dev(qw), sw_t, group, zeros=None if zb is None else bf16(zb),
                      bias=None if bb is None else bf16(bb))
    torch.cuda.synchronize()
    yb = bits(y)
    if cols is None:
        cols = np.arange(N)
    parts = []
    for c0 in range(0, len(cols), 2048):
        cc = cols[c0:c0 + 2048]
        parts.append(O.w4a16_linear(xb, qw[:, cc], sw[:, cc], group, zeros_bits=None if zb is None else zb[:, cc],
                                    bias_bits=None if bb is None else bb[cc], scale_dtype=scale_dtype))
    r = np.concatenate(parts, axis=1)
    check_bf16_output(yb[:, cols], r, f"w4a16 M={M} N={N} K={K} g={group}")
    return yb


@pytest.mark.parametrize("M", [1, 2, 3, 8])
@pytest.mark.parametrize("group", [64, 128, 256, -1])
def test_w4a16_small(M, group):
    _case(M, 200, 256, group, seed=M)


@pytest.mark.parametrize("K,group", [(576, 192), (1536, 768), (2560, -1), (8192, 128), (4096, 1024)])
def test_w4a16_groups_and_stages(K, group):
    """Groups that straddle the 1024-wide stages, K not a multiple of 1024, and
    more stages per strip than consumer warp groups."""
    _case(3, 136, K, group, zeros=True, seed=K)


@pytest.mark.parametrize("scale_dtype", ["f16", "bf16"])
@pytest.mark.parametrize("zeros", [False, True])
@pytest.mark.parametrize("bias", [False, True])
def test_w4a16_variants(scale_dtype, zeros, bias):
    _case(4, 328, 1024, 128, scale_dtype=scale_dtype, zeros=zeros, bias=bias, seed=11)


@pytest.mark.parametrize("M,N,K,group,zeros,bias", [(8, 6400, 4096, 128, False, True), (5, 5120, 8192, 128, False, False),
                                                    (7, 20000, 2048, 64, False, True), (6, 20000, 3072, -1, True, True)])
def test_w4a16_partials_in_tensor_memory(M, N, K, group, zeros, bias):
    """Token blocks whose strip partials in shared memory would leave room for
    only a 4-deep ring: the partials go to tensor memory. 16, 32, 8 and 12
    units of 256 k a strip (8 and 12: some warps add nothing to a strip, whose
    columns stay zero), 2 to 5 strips a CTA; every output column."""
    _case(M, N, K, group, zeros=zeros, bias=bias, seed=M + K)


@pytest.mark.parametrize("M,N,K,group,zeros", [(1, 20000, 2048, 128, False), (1, 4096, 8192, 64, True),
                                               (1, 6400, 3072, -1, False), (2, 14336, 4096, 128, False),
                                               (1, 9728, 5120, 128, True)])
def test_w4a16_resident_stages(M, N, K, group, zeros):
    """Shares of a CTA (strips x 1024-k stages) that take a slot per stage:
    five strips of 2 stages and two strips of 5 (10, on 16-slot indexing),
    one strip of 8, two strips of 3; and three strips of 4 at M = 2, whose
    shared memory does not fit them (the refilled ring)."""
    _case(M, N, K, group, zeros=zeros, seed=N + K)


@pytest.mark.parametrize("M,N,K,zeros", [(1, 1024, 1152, False), (4, 520, 640, True), (2, 4096, 4224, False),
                                         (3, 136, 128, True)])
def test_w4a16_group_columns_ragged_units(M, N, K, zeros):
    """Groups of 128 at up to four tokens fold a 256-k unit's two groups at
    once: K an odd number of groups leaves the last unit half past K (nine,
    five and 33 groups), and K = 128 is a single half unit."""
    _case(M, N, K, 128, zeros=zeros, seed=M * 100 + K)


@pytest.mark.parametrize("M", [9, 17, 40])
def test_w4a16_more_than_8_tokens(M):
    _case(M, 136, 512, 64, zeros=True, bias=True, seed=M)


@pytest.mark.parametrize("M", [1, 4, 8])
@pytest.mark.parametrize("zeros", [False, True])
def test_w4a16_full_size_decode(M, zeros):
    """K=4096, N=14336, group 128 (the decode GEMV): every output column
    (the oracle runs in column chunks)."""
    _case(M, 14336, 4096, 128, zeros=zeros, seed=100 + M, cols=np.arange(14336))


def test_w4a16_bf16_scales_full_size():
    _case(1, 14336, 4096, 128, scale_dtype="bf16", seed=7)


def test_w4a16_codes8_closed_form():
    """All codes 8 and zeros z: y = sum_g z[g,n] * sum_{k in g} x + bias."""
    M, N, K, g = 3, 64, 256, 64
    xb = S.activations_bf16(M, K, seed=5)
    qw = np.full((K // 8, N), 0x88888888, dtype=np.uint32).view(np.int32)
    sw = S.scales_f16((K // g, N))
    zb = S.zeros_bf16((K // g, N))
    bb = S.bias_bf16(N)
    y = w4.w4a16_gemm(bf16(xb), to_dev(qw), to_dev(sw), g, zeros=bf16(zb), bias=bf16(bb))
    xs = O.bf16_to_f64(xb).reshape(M, K // g, g).sum(axis=2)
    want = (xs @ O.bf16_to_f64(zb) + O.bf16_to_f64(bb)).astype(np.float32)
    check_bf16_output(bits(y), want, "codes 8")


def test_w4a16_shares_weights_with_w4a8_layout():
    """The same qweight buffer is a valid input to both paths (bit-identical layout)."""
    K, N = 256, 64
    qw = to_dev(S.random_words((K // 8, N), seed=9))
    before = qw.clone()
    w4.w4a16_gemm(bf16(S.activations_bf16(1, K)), qw, to_dev(S.scales_f16((2, N))), 128)
    torch.cuda.synchronize()
    assert torch.equal(qw, before)


def test_w4a16_output_guard():
    """Writes stay inside y: a sentinel band around the output is untouched."""
    M, N, K = 3, 72, 256
    buf = torch.full((M * N + 256,), -7.0, dtype=torch.bfloat16, device="cuda")
    y = buf[128:128 + M * N].view(M, N)
    xb = S.activations_bf16(M, K)
    w4.w4a16_gemm(bf16(xb), to_dev(S.random_words((K // 8, N))), to_dev(S.scales_f16((2, N))), 128, y=y)
    torch.cuda.synchronize()
    assert torch.all(buf[:128] == -7.0) and torch.all(buf[128 + M * N:] == -7.0)


def test_w4a16_back_to_back_chain_reads_previous_output():
    """Back-to-back calls on one stream where each call's x is the previous
    call's y (K == N): every call must read the finished output of the call
    before it, although the calls overlap through programmatic dependent
    launch. Each y_i is checked against the oracle applied to the GPU's
    y_{i-1}; the output buffers start out holding a constant, so a call that
    read its input early would disagree."""
    M, K, g, steps = 2, 4096, 128, 6
    N = K
    x0 = S.activations_bf16(M, K, seed=21)
    qws = [S.random_words((K // 8, N), seed=40 + i) for i in range(steps)]
    # scales chosen so the activations keep a similar magnitude from call to call
    sws = [S.scales_f16((K // g, N), lo=0.003, hi=0.004, seed=60 + i) for i in range(steps)]
    ys = [torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda") for _ in range(steps)]
    qws_d = [to_dev(q) for q in qws]
    sws_d = [to_dev(s_) for s_ in sws]
    x_d = bf16(x0)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        inp = x_d
        for i in range(steps):
            w4.w4a16_gemm(inp, qws_d[i], sws_d[i], g, y=ys[i], stream=s)
            inp = ys[i]
    s.synchronize()
    prev = x0
    for i in range(steps):
        yb = bits(ys[i])
        r = np.concatenate([O.w4a16_linear(prev, qws[i][:, c:c + 1024], sws[i][:, c:c + 1024], g)
                            for c in range(0, N, 1024)], axis=1)
        check_bf16_output(yb, r, f"chain step {i}")
        prev = yb


@pytest.mark.parametrize("x_pinned,y_pinned,M", [(True, True, 3), (True, False, 3), (False, True, 3),
                                                  (False, False, 3), (True, True, 17)])
def test_w4a16_host_entry_matches_device_entry(x_pinned, y_pinned, M):
    """w4a16_gemm_host gives the bytes of w4a16_gemm on device buffers and
    matches the oracle, and x_dev and y_dev hold x and y afterwards. With both
    host buffers page-locked, the call's L2-prefetch grid copies x in and the
    GEMV writes y out (17 tokens: three GEMV launches of up to 8 tokens, one
    copy of x); otherwise the copies are copy-engine jobs."""
    K, N, g = 1024, 512, 128
    xb = S.activations_bf16(M, K, seed=41)
    qw_np, sw_np = S.random_words((K // 8, N), seed=1), S.scales_f16((K // g, N), seed=2)
    qw, sw = to_dev(qw_np), to_dev(sw_np)
    x_host = torch.from_numpy(xb.view(np.int16).copy()).view(torch.bfloat16)
    y_host = torch.empty((M, N), dtype=torch.bfloat16)
    if x_pinned:
        x_host = x_host.pin_memory()
    if y_pinned:
        y_host = y_host.pin_memory()
    x_dev = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    y_dev = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    w4.w4a16_gemm_host(x_host, x_dev, qw, sw, g, y_dev, y_host)
    y_ref = w4.w4a16_gemm(bf16(xb), qw, sw, g)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y_host.view(torch.int16).numpy().view(np.uint16), bits(y_ref))
    np.testing.assert_array_equal(bits(y_dev), bits(y_ref))
    np.testing.assert_array_equal(bits(x_dev), xb)
    check_bf16_output(bits(y_ref), O.w4a16_linear(xb, qw_np, sw_np, g), "host entry")


def test_w4a16_host_entry_chain():
    """Eight host-entry calls queued back to back on one stream, each with its
    own x and y host buffers but the same x_dev and y_dev: every call's copy
    into x_dev waits for the GEMV before it, and every y_host gets its own
    call's result."""
    M, K, N, g, calls = 1, 4096, 2048, 128, 8
    qw_np, sw_np = S.random_words((K // 8, N), seed=3), S.scales_f16((K // g, N), seed=4)
    qw, sw = to_dev(qw_np), to_dev(sw_np)
    xs = [S.activations_bf16(M, K, seed=100 + i) for i in range(calls)]
    x_hosts = [torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).pin_memory() for x in xs]
    y_hosts = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(calls)]
    x_dev = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    y_dev = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    for i in range(calls):
        w4.w4a16_gemm_host(x_hosts[i], x_dev, qw, sw, g, y_dev, y_hosts[i])
    torch.cuda.synchronize()
    for i in range(calls):
        y_ref = w4.w4a16_gemm(bf16(xs[i]), qw, sw, g)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(y_hosts[i].view(torch.int16).numpy().view(np.uint16), bits(y_ref),
                                      err_msg=f"call {i}")
