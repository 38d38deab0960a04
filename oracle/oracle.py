"""NumPy float64 twin of the C oracle.  TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this module.  It shares no code with the CUDA library (and none with
``bqd_oracle.c`` either: the C file decodes one weight at a time with shifts
and divisions, this file decodes whole matrices with NumPy array operations,
so that the two can check each other).

Page followed: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" (oMLX Bonsai
custom kernels: the fast QMV path for the Qwen family), cnnetsun.cn/a/4328761.

* §二.1 (qmv_fast): 1-bit affine codes, 32 per uint32, unpacked by shifting,
  dotted with x without materialising float weights.  Read as LSB first.
* §二.2 (qmv_wide): same product for M = 2..5 rows of x; sym variant whose
  bias obeys identity I-B, bias = -scale * ratio, and is not read.
* §二.3 (t5): trits {0,1,2} in uint8, 13/26 bytes per 64/128-weight group.
  Read as five trits per byte, byte = sum_i t_i 3^i, first weight least
  significant, each group starting on a fresh byte.
* §四 (benchmark): bits in {1,2}, group_size in {64,128}.

The product itself is the plain definition
    y[m, n] = sum_k x[m, k] * (scale[n, k // gs] * q[n, k] + bias[n, k // gs])
evaluated with a float64 matrix product (a library primitive) on the
dequantised weight matrix.
"""
from __future__ import annotations

import numpy as np

FMT_AFFINE1 = 1
FMT_AFFINE2 = 2
FMT_T5 = 3
FORMATS = (FMT_AFFINE1, FMT_AFFINE2, FMT_T5)
GROUP_SIZES = (64, 128)

#: midpoint of each format's code range: the ratio used when no bias tensor
#: is given (1-bit: 0.5, 2-bit: 1.5, t5: 1.0, i.e. w = scale*t - scale).
DEFAULT_SYM_RATIO = {FMT_AFFINE1: 0.5, FMT_AFFINE2: 1.5, FMT_T5: 1.0}
MAX_CODE = {FMT_AFFINE1: 1, FMT_AFFINE2: 3, FMT_T5: 2}

_POW3 = np.array([1, 3, 9, 27, 81], dtype=np.int64)


def t5_bytes_per_group(gs: int) -> int:
    """ceil(gs / 5): 13 bytes for gs=64, 26 for gs=128 (§二.3)."""
    return -(-gs // 5)


def row_bytes(fmt: int, K: int, gs: int) -> int:
    """Bytes of one packed row."""
    if fmt not in FORMATS or gs not in GROUP_SIZES or K % gs:
        raise ValueError(f"invalid format/K/group_size: {fmt}, {K}, {gs}")
    if fmt == FMT_AFFINE1:
        return K // 8
    if fmt == FMT_AFFINE2:
        return K // 4
    return (K // gs) * t5_bytes_per_group(gs)


def unpack(packed: np.ndarray, N: int, K: int, fmt: int, gs: int) -> np.ndarray:
    """Packed bytes [N, row_bytes] -> codes uint8 [N, K]."""
    rb = row_bytes(fmt, K, gs)
    b = np.ascontiguousarray(packed, dtype=np.uint8).reshape(N, rb)
    if fmt == FMT_AFFINE1:
        # little-endian words, LSB first == bytes in order, bits LSB first
        return np.unpackbits(b, axis=1, count=K, bitorder="little").astype(np.uint8)
    if fmt == FMT_AFFINE2:
        shifts = np.array([0, 2, 4, 6], dtype=np.uint8)
        return ((b[:, :, None] >> shifts) & 3).reshape(N, K).astype(np.uint8)
    B = t5_bytes_per_group(gs)
    G = K // gs
    digits = (b.reshape(N, G, B).astype(np.int64)[..., None] // _POW3) % 3
    return digits.reshape(N, G, B * 5)[:, :, :gs].reshape(N, K).astype(np.uint8)


def pack(codes: np.ndarray, fmt: int, gs: int) -> np.ndarray:
    """Codes uint8 [N, K] -> packed bytes [N, row_bytes]."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    N, K = c.shape
    row_bytes(fmt, K, gs)
    if c.size and int(c.max()) > MAX_CODE[fmt]:
        raise ValueError("code out of range for the format")
    if fmt == FMT_AFFINE1:
        return np.packbits(c, axis=1, bitorder="little")
    if fmt == FMT_AFFINE2:
        q = c.reshape(N, K // 4, 4).astype(np.uint8)
        return (q[..., 0] | (q[..., 1] << 2) | (q[..., 2] << 4) | (q[..., 3] << 6)).astype(np.uint8)
    B = t5_bytes_per_group(gs)
    G = K // gs
    padded = np.zeros((N, G, B * 5), dtype=np.int64)
    padded[:, :, :gs] = c.reshape(N, G, gs)
    return (padded.reshape(N, G, B, 5) * _POW3).sum(axis=-1).reshape(N, G * B).astype(np.uint8)


def sym_bias(scales: np.ndarray, ratio: float) -> np.ndarray:
    """Identity I-B (§二.2): bias = -scale * ratio, formed in float32 and
    rounded once to fp16."""
    return (np.float32(-ratio) * np.asarray(scales, dtype=np.float16).astype(np.float32)).astype(np.float16)


def dequantize(packed, scales, biases, N: int, K: int, fmt: int, gs: int,
               ratio: float | None = None) -> np.ndarray:
    """float64 [N, K] weights w = scale*q + bias; biases None -> sym."""
    q = unpack(packed, N, K, fmt, gs).astype(np.float64)
    s = np.asarray(scales, dtype=np.float16).reshape(N, K // gs)
    if biases is None:
        b = sym_bias(s, DEFAULT_SYM_RATIO[fmt] if ratio is None else ratio)
    else:
        b = np.asarray(biases, dtype=np.float16).reshape(N, K // gs)
    s64 = np.repeat(s.astype(np.float64), gs, axis=1)
    b64 = np.repeat(b.astype(np.float64), gs, axis=1)
    return s64 * q + b64


def qmv(x, packed, scales, biases, fmt: int, gs: int, ratio: float | None = None):
    """(y, bound), both float64 [M, N]: y = x W^T, bound = |x| |W|^T."""
    x64 = np.asarray(x, dtype=np.float16).astype(np.float64)
    M, K = x64.shape
    N = np.asarray(scales).shape[0]
    W = dequantize(packed, scales, biases, N, K, fmt, gs, ratio)
    return x64 @ W.T, np.abs(x64) @ np.abs(W).T


def t5_invalid_bytes(packed, N: int, K: int, gs: int) -> int:
    """Bytes >= 243, plus group-final bytes whose padding trits are non-zero."""
    B = t5_bytes_per_group(gs)
    b = np.asarray(packed, dtype=np.uint8).reshape(N, K // gs, B).astype(np.int64)
    over = b >= 243
    live = gs - 5 * (B - 1)
    last = b[:, :, B - 1]
    pad_bad = (last // _POW3[live]) % (3 ** (5 - live)) != 0
    pad_bad &= ~over[:, :, B - 1]
    return int(over.sum() + pad_bad.sum())
