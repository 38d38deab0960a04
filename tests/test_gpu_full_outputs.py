"""Every output of one full-size call per kernel family, against the NumPy
float64 oracle (the whole [M, N] product x @ W^T and its bound |x| @ |W|^T),
at the bar |y_gpu - y| <= 2e-3 * sum_k |x_k w_k|.

The sampled-row tests elsewhere cover many shapes; these three cover every
CTA of a launch at the benchmark's sizes:
  * the 1/2-bit decode ring kernel: gate projection 17408x5120, 2-bit, gs=64,
    with biases, M=5;
  * the t5 decode ring kernel: down projection 5120x17408, gs=128, M=5;
  * the t5 prefill product: gate projection, gs=128, M=512.
"""
import numpy as np
import pytest

from oracle import oracle as npo
import bit_quantized_decode_unpack_gb300 as bqd
from bit_quantized_decode_unpack_gb300 import synth
from _util import assert_within_tolerance, forced_kernel, to_dev

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
F2, T5 = bqd.FMT_AFFINE2, bqd.FMT_T5


def full_check(fmt, M, N, K, gs, sym, kernel):
    import torch
    p = synth.problem(fmt, M, N, K, gs, sym=sym)
    packed = npo.pack(p["codes"], fmt, gs)
    w = bqd.pack(to_dev(p["codes"]), fmt, gs)
    # the device packer and the oracle's agree byte for byte
    assert np.array_equal(w.cpu().numpy(), packed)
    x, s, b = to_dev(p["x"]), to_dev(p["scales"]), to_dev(p["biases"])
    with forced_kernel(kernel):
        y = bqd.qmv(x, w, s, b, fmt, gs)
    torch.cuda.synchronize()
    yr, bound = npo.qmv(p["x"], packed, p["scales"], p["biases"], fmt, gs)
    assert_within_tolerance(y.cpu().numpy(), yr, bound, what=p["key"])


def test_decode_affine2_gate_m5_every_output():
    full_check(F2, 5, 17408, 5120, 64, False, "tma")


def test_decode_t5_down_m5_every_output():
    full_check(T5, 5, 5120, 17408, 128, True, "tma")


def test_prefill_t5_gate_m512_every_output():
    full_check(T5, 512, 17408, 5120, 128, True, "qmm")
