"""Failure detection without a GPU fault: every ring kernel bounds its
pipeline waits by %globaltimer.  With the limit set to 1 ns (bqd_set_option)
the first wait for data still in flight runs out; the CTA skips its work,
lets the copies it issued land (their drain waits keep the full second),
passes its cluster barriers, and bqd_device_status reports
BQD_ERR_TIMEOUT.  The context stays usable: with the default limit back, the
next call returns BQD_OK and matches the oracle."""
import numpy as np
import pytest

import oracle
import bit_quantized_decode_unpack_gb300 as bqd
from bit_quantized_decode_unpack_gb300 import synth
from _util import assert_within_tolerance, forced_kernel, to_dev

pytestmark = pytest.mark.gpu
F2, T5 = bqd.FMT_AFFINE2, bqd.FMT_T5
BQD_ERR_TIMEOUT = 7

CASES = [
    # (kernel family, fmt, M, N, K, gs, sym): the 1/2-bit and t5 TMA-ring decode
    # kernels with split-K clusters, and the tcgen05 prefill product
    ("tma", F2, 3, 4096, 5120, 64, False),
    ("tma", F2, 5, 2100, 2560, 128, False),  # scale boxes by 4-byte copies (20 groups a row)
    ("tma", T5, 2, 2048, 5120, 64, True),
    ("qmm", T5, 64, 1024, 2048, 128, True),
    ("qmm", F2, 64, 1024, 2048, 64, False),
]


@pytest.mark.parametrize("kernel,fmt,M,N,K,gs,sym", CASES)
def test_expired_wait_is_reported_and_the_next_call_is_clean(kernel, fmt, M, N, K, gs, sym):
    import torch
    p = synth.problem(fmt, M, N, K, gs, sym=sym)
    w = bqd.pack(to_dev(p["codes"]), fmt, gs)
    x, s, b = to_dev(p["x"]), to_dev(p["scales"]), to_dev(p["biases"])
    assert bqd.device_status() == 0  # nothing pending from earlier tests
    bqd.set_option(bqd.OPT_WAIT_LIMIT_NS, 1)
    try:
        with forced_kernel(kernel):
            for _ in range(3):
                bqd.qmv(x, w, s, b, fmt, gs)
        assert bqd.device_status() == BQD_ERR_TIMEOUT
    finally:
        bqd.set_option(bqd.OPT_WAIT_LIMIT_NS, 0)
    assert bqd.get_option(bqd.OPT_WAIT_LIMIT_NS) == 1_000_000_000
    with forced_kernel(kernel):
        y = bqd.qmv(x, w, s, b, fmt, gs)
    assert bqd.device_status() == 0
    torch.cuda.synchronize()
    packed = oracle.c_pack(p["codes"], fmt, gs)
    rows = np.unique(np.concatenate([[0, N - 1], np.random.default_rng(1).integers(0, N, 64)]))
    yr, bound = oracle.c_qmv_rows(p["x"], packed, p["scales"], p["biases"], fmt, gs, rows=rows)
    assert_within_tolerance(y.cpu().numpy()[:, rows], yr, bound, what=p["key"])
