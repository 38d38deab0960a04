"""Shared helpers for the GPU parity tests."""
from __future__ import annotations

import contextlib

import numpy as np

#: per-element bound: |y_gpu - y_oracle| <= RTOL * sum_k |x_k * w_k|
#: (fp16 inputs, fp32 accumulation, fp16 output)
RTOL = 2e-3


def assert_within_tolerance(y_gpu, y_ref, bound, what=""):
    y = np.asarray(y_gpu, dtype=np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite output"
    err = np.abs(y - y_ref)
    ok = err <= RTOL * bound
    if not ok.all():
        i = np.unravel_index(np.argmax(err - RTOL * bound), err.shape)
        raise AssertionError(f"{what}: {int((~ok).sum())} elements outside tolerance; worst at {i}: "
                             f"gpu {y[i]!r} oracle {y_ref[i]!r} bound {bound[i]!r}")
    return float((err / np.maximum(bound, 1e-300)).max())


@contextlib.contextmanager
def forced_kernel(name):
    """Force one kernel family (bqd_set_option) for the duration of a block."""
    import bit_quantized_decode_unpack_gb300 as bqd
    old = bqd.get_option(bqd.OPT_KERNEL)
    bqd.force_kernel(name)
    try:
        yield
    finally:
        bqd.set_option(bqd.OPT_KERNEL, old)


def to_dev(a, dev="cuda"):
    import torch
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)
