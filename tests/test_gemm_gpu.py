"""Parity of the CUDA W4A16 GEMM with the CPU oracle, through the C ABI.

Each case draws x and W from the seeded generators, quantises W twice - on
the device with w4a16_quantize and on the host with the oracle's quantiser -
checks the two packings are bit-identical, then compares every output of
the device GEMM with the oracle's fp64 product:
  fp32 activations: |y - y_ref| <= 1e-5 * sum_k |x * W_hat|
  bf16 activations: |y - y_ref| <= 4e-3 * sum_k |x * W_hat| (oracle fed the
  same bf16 values).
Workload shapes: the tiny GEMM (1x256 -> 512), the decode GEMV (1x7168 ->
4096), the tree-verify pair (64x7168 -> 4096 and 64x2048 -> 7168, 1 % of
activations x20), the prefill GEMM (2048x7168 -> 18432, checked on sampled
rows) and ragged edge cases.
"""

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 4e-3}


@pytest.fixture(scope="module")
def w4():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import int4_w4a16_group_gemm_gb300 as w4
    return w4


def quantize_both(w4, w, group=32):
    """Device quantiser and oracle quantiser on the same W; must agree bit-exactly."""
    wd = torch.from_numpy(w).cuda()
    qw_d, sc_d = w4.w4a16_quantize(wd, group=group)
    qw_h, sc_h = oracle.quantize_w4a16(w, group)
    np.testing.assert_array_equal(qw_d.cpu().numpy(), qw_h)
    np.testing.assert_array_equal(sc_d.cpu().numpy().view(np.uint32), sc_h.view(np.uint32))
    return qw_d, sc_d, qw_h, sc_h


def run_case(w4, M, N, K, dt, seed=0, outlier=0.0, algo="auto", rows=None, group=32):
    x = synth.activations(seed, M, K, outlier_frac=outlier)
    w = synth.weights(seed, N, K)
    qw_d, sc_d, qw_h, sc_h = quantize_both(w4, w, group)
    xt = torch.from_numpy(x)
    if dt == "bf16":
        xt = xt.to(torch.bfloat16)
    y = w4.w4a16_gemm(xt.cuda(), qw_d, sc_d, group=group, algo=algo)
    torch.cuda.synchronize()
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    yh = y.cpu().numpy().astype(np.float64)
    xo = xt.float().numpy()
    if rows is not None:
        xo = xo[rows]
        yh = yh[rows]
    ref, bound = oracle.gemm_ref(xo, qw_h, sc_h, group)
    err = np.abs(yh - ref)
    ratio = np.max(err / np.maximum(bound, 1e-300))
    assert np.all(err <= TOL[dt] * bound), f"max err/bound = {ratio:.3e}"
    return y, ratio


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_tiny_gemm(w4, dt):
    run_case(w4, 1, 512, 256, dt)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_decode_gemv(w4, dt):
    run_case(w4, 1, 4096, 7168, dt, seed=1)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(4096, 7168), (7168, 2048)])
def test_tree_verify_pair(w4, dt, shape):
    N, K = shape
    run_case(w4, 64, N, K, dt, seed=2, outlier=0.01)


@pytest.mark.parametrize("algo", ["simt"])
def test_tree_verify_forced_simt(w4, algo):
    run_case(w4, 64, 4096, 7168, "bf16", seed=3, outlier=0.01, algo=algo)


def test_prefill_gemm_sampled_rows(w4):
    M, N, K = 2048, 18432, 7168
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(M, size=48, replace=False))
    rows[0], rows[-1] = 0, M - 1
    run_case(w4, M, N, K, "bf16", seed=4, rows=rows)


@pytest.mark.parametrize("M,N,K", [
    (1, 1, 32), (2, 13, 96), (3, 1000, 160), (5, 37, 4128), (7, 8, 1024),
    (4, 100, 8192), (3, 24, 8224), (2, 9, 16384), (1, 5, 16384), (9, 33, 256),
])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_ragged_shapes(w4, M, N, K, dt):
    run_case(w4, M, N, K, dt, seed=M * 1000 + N)


def test_degenerate_weights_and_activations(w4):
    M, N, K = 3, 16, 256
    # all nibbles 0 (q = -8), unit scales: y = -8 * sum_k x exactly representable
    nib = np.zeros((N, K), np.int64)
    qw = oracle.pack_nibbles(nib)
    sc = np.ones((N, K // 32), np.float32)
    x = np.ones((M, K), np.float32)
    y = w4.w4a16_gemm(torch.from_numpy(x).cuda(), torch.from_numpy(qw).cuda(),
                      torch.from_numpy(sc).cuda())
    assert (y.cpu().numpy() == -8.0 * K).all()
    # zero activations give exact zeros; zero scales too
    x0 = np.zeros((M, K), np.float32)
    w = synth.weights(9, N, K)
    qw2, sc2 = oracle.quantize_w4a16(w)
    y0 = w4.w4a16_gemm(torch.from_numpy(x0).cuda(), torch.from_numpy(qw2).cuda(),
                       torch.from_numpy(sc2).cuda())
    assert (y0.cpu().numpy() == 0).all()
    y1 = w4.w4a16_gemm(torch.from_numpy(synth.activations(9, M, K)).cuda(),
                       torch.from_numpy(qw2).cuda(), torch.zeros_like(torch.from_numpy(sc2)).cuda())
    assert (y1.cpu().numpy() == 0).all()


def test_deterministic_bits(w4):
    M, N, K = 5, 777, 7168
    x = torch.from_numpy(synth.activations(5, M, K)).cuda()
    qw, sc = w4.w4a16_quantize(torch.from_numpy(synth.weights(5, N, K)).cuda())
    a = w4.w4a16_gemm(x, qw, sc)
    b = w4.w4a16_gemm(x, qw, sc)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_gemm_on_side_stream(w4):
    M, N, K = 2, 300, 2048
    x = torch.from_numpy(synth.activations(6, M, K)).cuda()
    qw, sc = w4.w4a16_quantize(torch.from_numpy(synth.weights(6, N, K)).cuda())
    ref = w4.w4a16_gemm(x, qw, sc)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = w4.w4a16_gemm(x, qw, sc, stream=s)
    s.synchronize()
    assert torch.equal(y, ref)


@pytest.mark.parametrize("M,N,K", [
    (256, 256, 64), (1, 256, 96), (300, 300, 7168), (257, 513, 160), (64, 4096, 7168),
    (512, 1000, 2048), (31, 40, 4128),
    # beyond 64 tokens with the split-K tiles in one wave
    (128, 4096, 7168), (100, 1000, 4224), (200, 300, 1024), (512, 2048, 2048),
    # the persistent 256 x 256 kernel (split tiles would exceed one wave), ragged
    (600, 2100, 160), (1100, 1500, 2080),
])
def test_tensor_core_path(w4, M, N, K):
    """The tcgen05 kernels on one-tile, ragged (M, N not multiples of the
    tile; K % 64 == 32) and multi-tile shapes: the split-K kernel up to one
    wave of 64 x 128 tiles, the persistent kernel beyond."""
    run_case(w4, M, N, K, "bf16", seed=M + N + K, algo="tc")


def test_tensor_core_path_rejects_fp32_beyond_64_tokens(w4):
    x = torch.zeros((65, 64), dtype=torch.float32, device="cuda")
    qw = torch.zeros((8, 8), dtype=torch.int32, device="cuda")
    sc = torch.zeros((8, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(w4.W4A16Error) as ei:
        w4.w4a16_gemm(x, qw, sc, algo="tc")
    assert ei.value.code == w4.W4A16_ERR_UNSUPPORTED


@pytest.mark.parametrize("M,N,K,outlier", [
    (64, 4096, 7168, 0.01), (64, 7168, 2048, 0.01), (33, 300, 160, 0.0), (17, 1000, 4128, 0.0),
    (64, 13, 96, 0.0), (1, 256, 64, 0.0), (5, 129, 2080, 0.0), (64, 128, 32, 0.0),
    (40, 520, 16384, 0.01),
])
def test_fp32_tensor_core_path(w4, M, N, K, outlier):
    """The fp32-exact tensor-core kernel (activations split into three bf16
    pieces, group scales applied in fp32) against the fp32 tolerance 1e-5 of
    sum|x * W_hat|: tree-verify shapes with outliers, ragged N and K (a
    single group, a last stage holding one group), M = 1 and the largest K."""
    _, ratio = run_case(w4, M, N, K, "f32", seed=M * 7 + N + K, outlier=outlier, algo="tc")
    assert ratio < 0.1  # far inside the bound, as fp32 accumulation should be


def test_fp32_tensor_core_deterministic_and_auto_choice(w4):
    M, N, K = 64, 700, 3072
    x = torch.from_numpy(synth.activations(16, M, K)).cuda()
    qw, sc = w4.w4a16_quantize(torch.from_numpy(synth.weights(16, N, K)).cuda())
    a = w4.w4a16_gemm(x, qw, sc, algo="tc")
    b = w4.w4a16_gemm(x, qw, sc)  # M = 64 fp32: the automatic choice is the same kernel
    assert w4.w4a16_gemm_launches(M, N, K, "f32", "auto") == 1
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_tensor_core_deterministic(w4):
    M, N, K = 700, 900, 1024
    x = torch.from_numpy(synth.activations(8, M, K)).to(torch.bfloat16).cuda()
    qw, sc = w4.w4a16_quantize(torch.from_numpy(synth.weights(8, N, K)).cuda())
    a = w4.w4a16_gemm(x, qw, sc, algo="tc")
    b = w4.w4a16_gemm(x, qw, sc, algo="tc")
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_overlap_flag_keeps_the_chain_ordered(w4, dt):
    """With W4A16_FLAG_OVERLAP a call may start streaming weights while the
    previous kernel runs, but must read x only after it. Chain four GEMMs,
    each consuming the previous output, into buffers poisoned with NaN: the
    overlapped chain must give the same bits as the plain one (a read of x
    before the previous call finished would see NaN or stale values). The
    first link is also checked against the oracle."""
    K = 2048
    x = synth.activations(12, 1, K)
    ws = [synth.weights(12, K, K, sub=i) for i in range(4)]
    dev = [w4.w4a16_quantize(torch.from_numpy(w).cuda()) for w in ws]
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32

    def chain(overlap):
        bufs = [torch.full((1, K), float("nan"), device="cuda") for _ in dev]
        ins = [torch.full((1, K), float("nan"), device="cuda", dtype=dtype) for _ in dev]
        torch.cuda.synchronize()
        ins[0].copy_(torch.from_numpy(x).to(dtype))
        for i, (qw, sc) in enumerate(dev):
            w4.w4a16_gemm(ins[i], qw, sc, y=bufs[i], overlap=overlap)
            if i + 1 < len(dev):
                ins[i + 1].copy_(bufs[i].to(dtype))
        torch.cuda.synchronize()
        return bufs

    plain = chain(False)
    over = chain(True)
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    for a, b in zip(plain, over):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
        assert torch.isfinite(a).all()
    xo = torch.from_numpy(x).to(dtype).float().numpy()
    q0, c0 = oracle.quantize_w4a16(ws[0])
    ref, bound = oracle.gemm_ref(xo, q0, c0)
    assert np.all(np.abs(plain[0].cpu().numpy().astype(np.float64) - ref) <= TOL[dt] * bound)


def test_overlap_back_to_back_same_output(w4):
    """Back-to-back overlapped calls writing the same y (a write-after-write
    chain) leave the last call's result."""
    M, N, K = 1, 4096, 7168
    x = torch.from_numpy(synth.activations(13, M, K)).cuda()
    qa, sa = w4.w4a16_quantize(torch.from_numpy(synth.weights(13, N, K, sub=0)).cuda())
    qb, sb = w4.w4a16_quantize(torch.from_numpy(synth.weights(13, N, K, sub=1)).cuda())
    ref_b = w4.w4a16_gemm(x, qb, sb)
    y = torch.empty((M, N), device="cuda")
    for _ in range(5):
        w4.w4a16_gemm(x, qa, sa, y=y, overlap=True)
        w4.w4a16_gemm(x, qb, sb, y=y, overlap=True)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int32), ref_b.view(torch.int32))


def test_cuda_core_path_rejects_k_beyond_its_limit(w4):
    K = 16416
    x = torch.zeros((1, K), dtype=torch.float32, device="cuda")
    qw = torch.zeros((4, K // 8), dtype=torch.int32, device="cuda")
    sc = torch.zeros((4, K // 32), dtype=torch.float32, device="cuda")
    with pytest.raises(w4.W4A16Error) as ei:
        w4.w4a16_gemm(x, qw, sc)
    assert ei.value.code == w4.W4A16_ERR_UNSUPPORTED


@pytest.mark.parametrize("M", [64, 300])
def test_tensor_core_overlap_chain(w4, M):
    """The tensor-core kernel under W4A16_FLAG_OVERLAP (split-K at M = 64,
    persistent tiles at M = 300): a chain of bf16 GEMMs, each consuming the
    previous output, into NaN-poisoned buffers gives the same bits as the
    plain chain; the first link is checked against the oracle."""
    K = 2048
    x = synth.activations(14, M, K)
    ws = [synth.weights(14, K, K, sub=i) for i in range(3)]
    dev = [w4.w4a16_quantize(torch.from_numpy(w).cuda()) for w in ws]

    def chain(overlap):
        ins = [torch.full((M, K), float("nan"), device="cuda", dtype=torch.bfloat16) for _ in dev]
        outs = [torch.full((M, K), float("nan"), device="cuda") for _ in dev]
        torch.cuda.synchronize()
        ins[0].copy_(torch.from_numpy(x).to(torch.bfloat16))
        for i, (qw, sc) in enumerate(dev):
            w4.w4a16_gemm(ins[i], qw, sc, y=outs[i], algo="tc", overlap=overlap)
            if i + 1 < len(dev):
                ins[i + 1].copy_(outs[i].to(torch.bfloat16))
        torch.cuda.synchronize()
        return outs

    plain = chain(False)
    over = chain(True)
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    for a, b in zip(plain, over):
        assert torch.isfinite(a).all()
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    xo = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    q0, c0 = oracle.quantize_w4a16(ws[0])
    ref, bound = oracle.gemm_ref(xo, q0, c0)
    assert np.all(np.abs(plain[0].cpu().numpy().astype(np.float64) - ref) <= TOL["bf16"] * bound)


@pytest.mark.parametrize("M", [64, 300])
def test_tensor_core_overlap_back_to_back_same_output(w4, M):
    """Back-to-back overlapped tensor-core calls writing the same y (a
    write-after-write chain with no other kernel between them) leave the
    last call's result."""
    N, K = 4096, 2048
    x = torch.from_numpy(synth.activations(15, M, K)).to(torch.bfloat16).cuda()
    qa, sa = w4.w4a16_quantize(torch.from_numpy(synth.weights(15, N, K, sub=0)).cuda())
    qb, sb = w4.w4a16_quantize(torch.from_numpy(synth.weights(15, N, K, sub=1)).cuda())
    ref_b = w4.w4a16_gemm(x, qb, sb, algo="tc")
    y = torch.empty((M, N), device="cuda")
    for _ in range(5):
        w4.w4a16_gemm(x, qa, sa, y=y, algo="tc", overlap=True)
        w4.w4a16_gemm(x, qb, sb, y=y, algo="tc", overlap=True)
    torch.cuda.synchronize()
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    assert torch.equal(y.view(torch.int32), ref_b.view(torch.int32))


# Group sizes 64 and 128 on every kernel: the streaming kernel with scale
# rows staged by bulk copy (K / group a multiple of 4) and loaded per lane
# (K = 4224: 66 or 33 groups), the bf16 tensor-core kernel (whole and
# split-K) and the fp32-exact tensor-core kernel.
GROUP_CASES = [
    # M, N, K, dtype, algo, outlier
    (1, 4096, 7168, "f32", "simt", 0.0),
    (1, 4096, 7168, "bf16", "simt", 0.0),
    (3, 513, 4224, "f32", "simt", 0.0),
    (2, 1000, 2048, "bf16", "simt", 0.0),
    (64, 700, 1024, "f32", "simt", 0.01),
    (300, 300, 7168, "bf16", "tc", 0.0),
    (64, 4096, 7168, "bf16", "tc", 0.01),
    (31, 40, 4224, "bf16", "tc", 0.0),
    (64, 4096, 7168, "f32", "tc", 0.01),
    (17, 1000, 4224, "f32", "tc", 0.0),
    (33, 300, 384, "f32", "tc", 0.0),
]


@pytest.mark.parametrize("group", [64, 128])
@pytest.mark.parametrize("M,N,K,dt,algo,outlier", GROUP_CASES)
def test_group_sizes_64_and_128(w4, group, M, N, K, dt, algo, outlier):
    _, ratio = run_case(w4, M, N, K, dt, seed=M + N + K + group, outlier=outlier, algo=algo,
                        group=group)
    if dt == "f32":
        assert ratio < 0.1


def test_group_size_mismatch_is_rejected(w4):
    x = torch.zeros((1, 192), dtype=torch.float32, device="cuda")
    qw = torch.zeros((8, 24), dtype=torch.int32, device="cuda")
    sc = torch.zeros((8, 3), dtype=torch.float32, device="cuda")
    for group, code in ((128, w4.W4A16_ERR_INVALID_ARG), (16, w4.W4A16_ERR_UNSUPPORTED)):
        with pytest.raises(w4.W4A16Error) as ei:
            w4.w4a16_gemm(x, qw, sc, group=group)
        assert ei.value.code == code


# bf16 output (W4A16_FLAG_OUT_BF16) on every kernel: each element is the
# fp32 result of the same call rounded to nearest even, and within the
# tolerance plus one bf16 rounding (2^-8 |y|) of the oracle.
OUT_BF16_CASES = [
    # M, N, K, x dtype, algo, group
    (1, 4096, 7168, "f32", "simt", 32),
    (3, 513, 4224, "bf16", "simt", 64),
    (7, 300, 1024, "f32", "simt", 128),
    (300, 300, 7168, "bf16", "tc", 32),
    (64, 4096, 7168, "bf16", "tc", 128),
    (64, 4096, 7168, "f32", "tc", 32),
    (17, 1000, 4224, "f32", "tc", 64),
]


@pytest.mark.parametrize("M,N,K,dt,algo,group", OUT_BF16_CASES)
def test_bf16_output(w4, M, N, K, dt, algo, group):
    seed = 3 * M + N + K
    x = synth.activations(seed, M, K)
    w = synth.weights(seed, N, K)
    qw_d, sc_d, qw_h, sc_h = quantize_both(w4, w, group)
    xt = torch.from_numpy(x)
    if dt == "bf16":
        xt = xt.to(torch.bfloat16)
    xd = xt.cuda()
    y32 = w4.w4a16_gemm(xd, qw_d, sc_d, group=group, algo=algo)
    y16 = w4.w4a16_gemm(xd, qw_d, sc_d, group=group, algo=algo, out_dtype="bf16")
    torch.cuda.synchronize()
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    assert y16.dtype == torch.bfloat16 and y16.shape == (M, N)
    # same fp32 sums, then one round-to-nearest-even (torch's conversion)
    assert torch.equal(y16.view(torch.int16), y32.to(torch.bfloat16).view(torch.int16))
    ref, bound = oracle.gemm_ref(xt.float().numpy(), qw_h, sc_h, group)
    err = np.abs(y16.float().cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= TOL[dt] * bound * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(ref))


def test_bf16_output_needs_a_bf16_buffer(w4):
    x = torch.zeros((1, 64), dtype=torch.float32, device="cuda")
    qw = torch.zeros((8, 8), dtype=torch.int32, device="cuda")
    sc = torch.zeros((8, 2), dtype=torch.float32, device="cuda")
    with pytest.raises(TypeError):
        w4.w4a16_gemm(x, qw, sc, y=torch.zeros((1, 8), device="cuda"), out_dtype="bf16")


# The bench's launch configuration: programmatic launch (overlap) inside one
# CUDA graph replayed on a side stream, back-to-back calls on rotating weight
# copies. Every call's output must match the oracle as in eager mode.
@pytest.mark.parametrize("M,N,K,dt", [
    (1, 4096, 7168, "f32"),      # decode GEMV: streaming kernel
    (64, 4096, 7168, "bf16"),    # tree-verify gate/up: small-M tensor-core kernel
    (64, 7168, 2048, "f32"),     # tree-verify down: fp32-exact tensor-core kernel
])
def test_graph_replay_with_overlap_matches_oracle(w4, M, N, K, dt):
    ncopies = 3
    x = synth.activations(40 + M, M, K, outlier_frac=0.01 if M > 1 else 0.0)
    xt = torch.from_numpy(x)
    if dt == "bf16":
        xt = xt.to(torch.bfloat16)
    xd = xt.cuda()
    host, dev = [], []
    for c in range(ncopies):
        w = synth.weights(40 + M, N, K, sub=c)
        qw_d, sc_d, qw_h, sc_h = quantize_both(w4, w)
        host.append((qw_h, sc_h))
        dev.append((qw_d, sc_d))
    ys = [torch.full((M, N), float("nan"), device="cuda") for _ in range(2 * ncopies)]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(2):  # warm-up outside the graph
            w4.w4a16_gemm(xd, *dev[i % ncopies], y=ys[i], overlap=True, stream=stream)
    stream.synchronize()
    for y in ys:
        y.fill_(float("nan"))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(2 * ncopies):
            w4.w4a16_gemm(xd, *dev[i % ncopies], y=ys[i], overlap=True,
                          stream=torch.cuda.current_stream())
    graph.replay()
    torch.cuda.synchronize()
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    xo = xt.float().numpy()
    for c in range(ncopies):
        ref, bound = oracle.gemm_ref(xo, *host[c])
        for y in (ys[c], ys[c + ncopies]):
            err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
            assert np.all(err <= TOL[dt] * bound), f"copy {c}: max err/bound {np.max(err / bound):.3e}"
        assert torch.equal(ys[c].view(torch.int32), ys[c + ncopies].view(torch.int32))


# The decode GEMV kernel (one token, one CTA per SM, weights prefetched
# across calls) and the streaming kernel at M = 1, each forced, against the
# oracle: the decode shape, ragged N (fewer rows than SMs, rows not a
# multiple of the 4-row stage), one-word-only warps (small K), all-two-word
# warps (K = 8192), more stages than ring slots (refills), group 128.
GEMV_CASES = [
    # N, K, group
    (4096, 7168, 32), (1, 128, 32), (7, 2048, 32), (153, 8192, 32), (5000, 4096, 32),
    (9728, 7168, 32), (4096, 7168, 128), (300, 1024, 64), (2, 256, 64),
]


@pytest.mark.parametrize("algo", ["gemv", "stream"])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("N,K,group", GEMV_CASES)
def test_decode_kernels_m1(w4, algo, dt, N, K, group):
    _, ratio = run_case(w4, 1, N, K, dt, seed=N + K + group, algo=algo, group=group)
    if dt == "f32":
        assert ratio < 0.1


def test_gemv_kernel_rejects_other_shapes(w4):
    # M = 1 with K <= 8192 and whole 16-byte scale rows: one launch of it
    assert w4.w4a16_gemm_launches(1, 4096, 7168, "f32", "gemv") == 1
    for M, N, K in ((2, 64, 256), (1, 64, 8448), (1, 64, 96)):
        x = torch.zeros((M, K), dtype=torch.float32, device="cuda")
        qw = torch.zeros((N, K // 8), dtype=torch.int32, device="cuda")
        sc = torch.zeros((N, K // 32), dtype=torch.float32, device="cuda")
        with pytest.raises(w4.W4A16Error) as ei:
            w4.w4a16_gemm(x, qw, sc, algo="gemv")
        assert ei.value.code == w4.W4A16_ERR_UNSUPPORTED
    # the same call twice: identical bits (fixed reduction order)
    x = torch.from_numpy(synth.activations(50, 1, 7168)).cuda()
    qw, sc = w4.w4a16_quantize(torch.from_numpy(synth.weights(50, 4096, 7168)).cuda())
    a = w4.w4a16_gemm(x, qw, sc, algo="gemv")
    b = w4.w4a16_gemm(x, qw, sc, algo="gemv")
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_gemv_overlap_chain_long(w4, dt):
    """Twelve overlapped decode GEMVs, each consuming the previous output,
    into NaN-poisoned buffers (so the next call's CTAs prefetch beside the
    running call for the whole chain): same bits as the plain chain."""
    K, n = 4096, 12
    x = synth.activations(51, 1, K)
    dev = [w4.w4a16_quantize(torch.from_numpy(synth.weights(51, K, K, sub=i)).cuda())
           for i in range(n)]
    dtype = torch.bfloat16 if dt == "bf16" else torch.float32

    def chain(overlap):
        outs = [torch.full((1, K), float("nan"), device="cuda") for _ in dev]
        ins = [torch.full((1, K), float("nan"), device="cuda", dtype=dtype) for _ in dev]
        torch.cuda.synchronize()
        ins[0].copy_(torch.from_numpy(x).to(dtype))
        for i, (qw, sc) in enumerate(dev):
            # scale down so that the chain stays in range
            w4.w4a16_gemm(ins[i], qw, sc, y=outs[i], algo="gemv", overlap=overlap)
            if i + 1 < n:
                ins[i + 1].copy_((outs[i] * 0.5).to(dtype))
        torch.cuda.synchronize()
        return outs

    plain = chain(False)
    over = chain(True)
    assert w4.w4a16_last_device_status() == w4.W4A16_OK
    for a, b in zip(plain, over):
        assert torch.isfinite(a).all()
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
