"""GPU parity of the prefill matrix product (tcgen05 tensor cores; the
dispatcher's choice for large M) against the float64 oracle, through the C
ABI: t5 and the 1/2-bit formats.  Most cases force the product
(the kernel option set to "qmm") so that it is tested at every shape.

Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" §二.3 -- for M > 16
the t5 weights go through a fused unpack + matrix-multiply kernel; §二.1 -- the
1-bit prefill path is a separate (there: dequantise + dense) product, here the
same fused kernel with a 1/2-bit decode.
Bar: |y_gpu - y| <= 2e-3 * sum_k |x_k w_k| for every checked output.
"""
import numpy as np
import pytest

import oracle
import bit_quantized_decode_unpack_gb300 as bqd
from bit_quantized_decode_unpack_gb300 import synth
from _util import assert_within_tolerance, forced_kernel, to_dev

pytestmark = pytest.mark.gpu
T5, F1, F2 = bqd.FMT_T5, bqd.FMT_AFFINE1, bqd.FMT_AFFINE2


def run(p, kernel="qmm", m_rows=None, n_rows=None):
    import torch
    gs, fmt = p["gs"], p["fmt"]
    w = bqd.pack(to_dev(p["codes"]), fmt, gs)
    with forced_kernel(kernel):
        y = bqd.qmv(to_dev(p["x"]), w, to_dev(p["scales"]), to_dev(p["biases"]), fmt, gs)
    torch.cuda.synchronize()
    assert bqd.device_status() == 0
    packed = oracle.c_pack(p["codes"], fmt, gs)
    xs = p["x"] if m_rows is None else p["x"][m_rows]
    yr, bound = oracle.c_qmv_rows(xs, packed, p["scales"], p["biases"], fmt, gs, rows=n_rows)
    yg = y.cpu().numpy().astype(np.float64)
    if m_rows is not None:
        yg = yg[m_rows]
    if n_rows is not None:
        yg = yg[:, n_rows]
    return assert_within_tolerance(yg, yr, bound, what=p["key"])


# (M, N, K): ragged M and N tails, one to many tiles, split-K clusters when few tiles
SMALL = [(17, 128, 1024), (32, 200, 2048), (33, 384, 1024), (64, 130, 3072), (100, 256, 2048),
         (200, 129, 1024), (48, 40, 5120)]


@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("bias", [False, True])
def test_small_shapes_all_outputs(gs, bias):
    for M, N, K in SMALL:
        p = synth.problem(T5, M, N, K, gs, sym=True)
        if bias:  # general affine t5 (explicit bias tensor)
            p["biases"] = synth.biases(np.random.default_rng(M + N), F2, p["scales"])
        run(p)


def test_default_dispatch_takes_the_matrix_product_and_agrees():
    import torch
    p = synth.problem(T5, 40, 256, 2048, 128, sym=True)
    w = bqd.pack(to_dev(p["codes"]), T5, 128)
    x, s = to_dev(p["x"]), to_dev(p["scales"])
    y_default = bqd.qmv(x, w, s, None, T5, 128)
    with forced_kernel("mma"):
        y_forced = bqd.qmv(x, w, s, None, T5, 128)
    with forced_kernel("generic"):
        y_generic = bqd.qmv(x, w, s, None, T5, 128)
    torch.cuda.synchronize()
    assert torch.equal(y_default.view(torch.int16), y_forced.view(torch.int16))
    run(p, None)
    # the generic kernel is an independent implementation: same tolerance
    packed = oracle.c_pack(p["codes"], T5, 128)
    yr, bound = oracle.c_qmv_rows(p["x"], packed, p["scales"], None, T5, 128)
    assert_within_tolerance(y_generic.cpu().numpy(), yr, bound)


def test_large_scales_use_the_exact_decode():
    rng = np.random.default_rng(8)
    p = synth.problem(T5, 24, 160, 1024, 64, sym=True)
    p["scales"] = (np.abs(rng.normal(0, 200, size=p["scales"].shape)) + 1).astype(np.float16)
    p["x"] = (p["x"].astype(np.float32) * 1e-3).astype(np.float16)
    run(p)


def test_deterministic():
    import torch
    p = synth.problem(T5, 64, 512, 5120, 128, sym=True)
    w = bqd.pack(to_dev(p["codes"]), T5, 128)
    x, s = to_dev(p["x"]), to_dev(p["scales"])
    y0 = bqd.qmv(x, w, s, None, T5, 128)
    y1 = bqd.qmv(x, w, s, None, T5, 128)
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


# the prefill sizes the benchmark times: M in {32, 512, 2048}, gs=128
FULL = [(M, N, K) for M in (32, 512, 2048) for (N, K) in [(17408, 5120), (5120, 17408)]]


@pytest.mark.slow
@pytest.mark.parametrize("M,N,K", FULL)
def test_full_size_sampled(M, N, K):
    rng = np.random.default_rng(M + N)
    p = synth.problem(T5, M, N, K, 128, sym=True)
    m_rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 10)]))
    n_rows = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 12)]))
    run(p, None, m_rows=m_rows, n_rows=n_rows)


# ---- 1/2-bit formats --------------------------------------------------------------

# (M, N, K): K down to one group (gs=128: K=128 is a single K step), ragged M
# and N
AFFINE_SMALL = SMALL + [(17, 33, 128), (40, 257, 384), (300, 257, 1024), (260, 40, 128)]


@pytest.mark.parametrize("fmt", [F1, F2])
@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("sym", [False, True])
def test_affine_small_shapes_all_outputs(fmt, gs, sym):
    for M, N, K in AFFINE_SMALL:
        if K % gs:
            continue
        run(synth.problem(fmt, M, N, K, gs, sym=sym))


@pytest.mark.parametrize("fmt", [F1, F2])
@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("sym", [False, True])
def test_affine_two_column_blocks_per_cta(fmt, gs, sym):
    """M > 256 on a wide layer (N >= 8192): each CTA owns two 256-column x
    blocks (two TMEM accumulators) with 64-code K steps.  M = 300 leaves one
    block half empty, 513 adds a nearly empty CTA column; N = 8200 a ragged
    row tile.  Sampled outputs (rows of the first, a middle and the last tile)."""
    rng = np.random.default_rng(fmt * 10 + gs)
    for M, N, K in [(300, 8200, 256), (513, 8192, 384)]:
        if K % gs:
            continue
        p = synth.problem(fmt, M, N, K, gs, sym=sym)
        m_rows = np.unique(np.concatenate([[0, 255, 256, M - 1], rng.integers(0, M, 12)]))
        n_rows = np.unique(np.concatenate([[0, 127, 4096, N - 1], rng.integers(0, N, 12)]))
        run(p, m_rows=m_rows, n_rows=n_rows)


@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("bias", [False, True])
def test_t5_two_column_blocks_per_cta(gs, bias):
    """t5 takes the two-block mode too: a 64-code group splits into 32-code
    halves at bytes 0 and 6, a 128-code group into quarters that start inside
    bytes 0, 6, 12 and 18 (the product takes rows of whole 16-byte pieces, so
    K / gs is a multiple of 16 at gs=64 and of 8 at gs=128).  Sampled outputs
    as above."""
    rng = np.random.default_rng(gs + bias)
    for M, N, K in [(300, 8200, 1024), (513, 8192, 3072)]:
        p = synth.problem(T5, M, N, K, gs, sym=True)
        if bias:
            p["biases"] = synth.biases(rng, F2, p["scales"])
        m_rows = np.unique(np.concatenate([[0, 255, 256, M - 1], rng.integers(0, M, 12)]))
        n_rows = np.unique(np.concatenate([[0, 127, 4096, N - 1], rng.integers(0, N, 12)]))
        run(p, m_rows=m_rows, n_rows=n_rows)


@pytest.mark.parametrize("fmt", [F1, F2, T5])
@pytest.mark.parametrize("gs", [64, 128])
def test_forced_product_at_decode_sizes(fmt, gs):
    """The forced product runs for M <= 16 too (one x tile of 32
    columns, mostly empty): still exact to the bar."""
    for M, N, K in [(1, 129, 1024), (5, 256, 2048), (16, 40, 1024)]:
        run(synth.problem(fmt, M, N, K, gs, sym=fmt == T5), "qmm")


@pytest.mark.parametrize("fmt", [F1, F2])
def test_affine_default_dispatch_takes_the_product_and_agrees(fmt):
    """A prefill-sized M (here 70 rows of a narrow layer) goes to the product by
    default (bit-identical to the forced call); the generic CUDA-core kernel,
    an independent implementation, meets the same bar."""
    import torch
    p = synth.problem(fmt, 70, 256, 2048, 64)
    w = bqd.pack(to_dev(p["codes"]), fmt, 64)
    x, s, b = to_dev(p["x"]), to_dev(p["scales"]), to_dev(p["biases"])
    y_default = bqd.qmv(x, w, s, b, fmt, 64)
    with forced_kernel("qmm"):
        y_forced = bqd.qmv(x, w, s, b, fmt, 64)
    with forced_kernel("generic"):
        y_generic = bqd.qmv(x, w, s, b, fmt, 64)
    torch.cuda.synchronize()
    assert torch.equal(y_default.view(torch.int16), y_forced.view(torch.int16))
    run(p, None)
    packed = oracle.c_pack(p["codes"], fmt, 64)
    yr, bound = oracle.c_qmv_rows(p["x"], packed, p["scales"], p["biases"], fmt, 64)
    assert_within_tolerance(y_generic.cpu().numpy(), yr, bound)


@pytest.mark.parametrize("fmt", [F1, F2])
def test_affine_large_scales_use_the_exact_decode(fmt):
    """|s| >= 63 would overflow the fp16 constant -1024*s: those groups take the
    (magic - offset) * s form; both forms give fp16(s*q) exactly."""
    rng = np.random.default_rng(9)
    p = synth.problem(fmt, 24, 160, 1024, 64)
    p["scales"] = (np.abs(rng.normal(0, 200, size=p["scales"].shape)) + 1).astype(np.float16)
    p["biases"] = (-p["scales"].astype(np.float32) * 0.5).astype(np.float16)
    p["x"] = (p["x"].astype(np.float32) * 1e-3).astype(np.float16)
    run(p)


@pytest.mark.parametrize("fmt", [F1, F2])
def test_affine_one_hot_x_recovers_the_weights(fmt):
    """x = e_k: y[m, n] is the dequantised weight fp16(fp16(s*q) + b) exactly
    (one non-zero product, accumulated in fp32, rounded once to fp16)."""
    import torch
    M, N, K, gs = 32, 200, 512, 64
    p = synth.problem(fmt, M, N, K, gs)
    ks = np.arange(M) * 13 % K
    x = np.zeros((M, K), dtype=np.float16)
    x[np.arange(M), ks] = 1.0
    w = bqd.pack(to_dev(p["codes"]), fmt, gs)
    with forced_kernel("qmm"):  # the product materialises the fp16 weights
        y = bqd.qmv(to_dev(x), w, to_dev(p["scales"]), to_dev(p["biases"]), fmt, gs)
    torch.cuda.synchronize()
    s = p["scales"][:, ks // gs].astype(np.float32)            # [N, M]
    b = p["biases"][:, ks // gs].astype(np.float32)
    q = p["codes"][:, ks].astype(np.float32)
    want = ((s * q).astype(np.float16).astype(np.float32) + b).astype(np.float16).T
    assert np.array_equal(y.cpu().numpy().view(np.int16), want.view(np.int16))


@pytest.mark.parametrize("gs", [64, 128])
def test_t5_two_column_blocks_one_hot_x_recovers_the_weights(gs):
    """Two-block mode (M > 256, N >= 8192), x = e_k with k = m mod K: every
    code position of every half / quarter pattern comes back as the
    dequantised weight fp16(fp16(s*t) + b), bit for bit."""
    import torch
    M, N, K = 300, 8192, 1024  # k = 0 .. 299: all of the first two 128-code groups
    rng = np.random.default_rng(7 + gs)
    p = synth.problem(T5, M, N, K, gs, sym=True)
    p["biases"] = synth.biases(rng, F2, p["scales"])
    ks = np.arange(M) % K
    x = np.zeros((M, K), dtype=np.float16)
    x[np.arange(M), ks] = 1.0
    w = bqd.pack(to_dev(p["codes"]), T5, gs)
    with forced_kernel("qmm"):
        y = bqd.qmv(to_dev(x), w, to_dev(p["scales"]), to_dev(p["biases"]), T5, gs)
    torch.cuda.synchronize()
    assert bqd.device_status() == 0
    s = p["scales"][:, ks // gs].astype(np.float32)            # [N, M]
    b = p["biases"][:, ks // gs].astype(np.float32)
    t = p["codes"][:, ks].astype(np.float32)
    want = ((s * t).astype(np.float16).astype(np.float32) + b).astype(np.float16).T
    assert np.array_equal(y.cpu().numpy().view(np.int16), want.view(np.int16))


@pytest.mark.parametrize("fmt", [F1, F2])
def test_affine_zero_codes_zero_bias_give_exact_zeros(fmt):
    import torch
    M, N, K, gs = 48, 300, 1024, 128
    p = synth.problem(fmt, M, N, K, gs)
    w = bqd.pack(to_dev(np.zeros_like(p["codes"])), fmt, gs)
    b = torch.zeros((N, K // gs), dtype=torch.float16, device="cuda")
    with forced_kernel("qmm"):
        y = bqd.qmv(to_dev(p["x"]), w, to_dev(p["scales"]), b, fmt, gs)
    torch.cuda.synchronize()
    assert torch.all(y == 0)


AFFINE_FULL = [(fmt, M, N, K) for fmt in (F1, F2) for M in (32, 512, 2048)
               for (N, K) in [(17408, 5120), (5120, 17408)]]


@pytest.mark.slow
@pytest.mark.parametrize("fmt,M,N,K", AFFINE_FULL)
def test_affine_full_size_sampled(fmt, M, N, K):
    rng = np.random.default_rng(M + N + fmt)
    p = synth.problem(fmt, M, N, K, 128)
    m_rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 10)]))
    n_rows = np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 12)]))
    run(p, "qmm", m_rows=m_rows, n_rows=n_rows)
