"""GPU parity of the t5 prefill matrix product (tcgen05 tensor cores, M > 16)
against the float64 oracle, through the C ABI.

Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" §二.3 -- for M > 16
the t5 weights go through a fused unpack + matrix-multiply kernel.
Bar: |y_gpu - y| <= 2e-3 * sum_k |x_k w_k| for every checked output.
"""
import numpy as np
import pytest

import oracle
import bit_quantized_decode_unpack_gb300 as bqd
from bit_quantized_decode_unpack_gb300 import synth
from _util import assert_within_tolerance, forced_kernel, to_dev

pytestmark = pytest.mark.gpu
T5, F2 = bqd.FMT_T5, bqd.FMT_AFFINE2


def run(p, kernel="mma", m_rows=None, n_rows=None):
    import torch
    gs = p["gs"]
    w = bqd.pack(to_dev(p["codes"]), T5, gs)
    with forced_kernel(kernel):
        y = bqd.qmv(to_dev(p["x"]), w, to_dev(p["scales"]), to_dev(p["biases"]), T5, gs)
    torch.cuda.synchronize()
    assert bqd.device_status() == 0
    packed = oracle.c_pack(p["codes"], T5, gs)
    xs = p["x"] if m_rows is None else p["x"][m_rows]
    yr, bound = oracle.c_qmv_rows(xs, packed, p["scales"], p["biases"], T5, gs, rows=n_rows)
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
