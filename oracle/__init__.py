"""Float64 CPU oracle for the low-bit quantized matrix-vector product.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import, call or link anything
here.  The CUDA library never does, and this package never imports the CUDA
library: the two share no code.

Two independent implementations of the same definitions:

* ``bqd_oracle.c`` (C99, one weight at a time; loaded through ctypes here),
* ``oracle.py`` (NumPy, whole-matrix array operations).

``spec_verify.py`` holds the oracle of the speculative-decoding verification
step (plain Python loops).

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against closed forms, exhaustive enumerations and brute force.  None of them
is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from pathlib import Path

import numpy as np

from . import oracle as np_oracle  # noqa: F401  (the NumPy twin)
from .spec_verify import spec_decode_verify  # noqa: F401  (speculative-decoding verification)
from .oracle import (DEFAULT_SYM_RATIO, FMT_AFFINE1, FMT_AFFINE2, FMT_T5,  # noqa: F401
                     FORMATS, GROUP_SIZES, MAX_CODE, t5_bytes_per_group)

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "bqd_oracle.c"
_LIB = _HERE / "_build" / "libbqd_oracle.so"
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> Path:
    """Compile the C oracle with gcc (plain -O2, no vectorisation flags)."""
    _LIB.parent.mkdir(parents=True, exist_ok=True)
    if force or not _LIB.exists() or _LIB.stat().st_mtime < max(
            _SRC.stat().st_mtime, (_HERE / "bqd_oracle.h").stat().st_mtime):
        tmp = _LIB.with_suffix(f".{os.getpid()}.tmp.so")
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared",
                               "-o", str(tmp), str(_SRC), "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _c():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(str(build()))
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            vp = ctypes.c_void_p
            lib.orc_half_to_double.argtypes = [ctypes.c_uint16]
            lib.orc_half_to_double.restype = dbl
            lib.orc_float_to_half_rne.argtypes = [ctypes.c_float]
            lib.orc_float_to_half_rne.restype = ctypes.c_uint16
            lib.orc_row_bytes.argtypes = [i32, i64, i32]
            lib.orc_row_bytes.restype = i64
            lib.orc_code_at.argtypes = [vp, i32, i32, i64]
            lib.orc_code_at.restype = i32
            lib.orc_t5_encode.argtypes = [vp]
            lib.orc_t5_encode.restype = i32
            lib.orc_t5_decode.argtypes = [i32, vp]
            lib.orc_t5_decode.restype = None
            lib.orc_pack.argtypes = [vp, i64, i64, i32, i32, vp]
            lib.orc_pack.restype = i64
            lib.orc_unpack.argtypes = [vp, i64, i64, i32, i32, vp]
            lib.orc_unpack.restype = i64
            lib.orc_t5_invalid_bytes.argtypes = [vp, i64, i64, i32]
            lib.orc_t5_invalid_bytes.restype = i64
            lib.orc_sym_bias.argtypes = [ctypes.c_uint16, dbl]
            lib.orc_sym_bias.restype = ctypes.c_uint16
            lib.orc_sym_mismatches.argtypes = [vp, vp, i64, i64, dbl]
            lib.orc_sym_mismatches.restype = i64
            lib.orc_qmv_rows.argtypes = [vp, vp, vp, vp, dbl, i64, i64, i64, i32, i32,
                                         vp, i64, vp, vp]
            lib.orc_qmv_rows.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits16(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float16)).view(np.uint16)


# ---- C oracle, Python face ------------------------------------------------

def c_half_to_double(bits: int) -> float:
    return _c().orc_half_to_double(bits)


def c_float_to_half_bits(f: float) -> int:
    return _c().orc_float_to_half_rne(f)


def c_row_bytes(fmt: int, K: int, gs: int) -> int:
    return _c().orc_row_bytes(fmt, K, gs)


def c_t5_encode(trits) -> int:
    t = np.ascontiguousarray(trits, dtype=np.uint8)
    return _c().orc_t5_encode(_ptr(t))


def c_t5_decode(byte_value: int) -> np.ndarray:
    t = np.zeros(5, dtype=np.uint8)
    _c().orc_t5_decode(int(byte_value), _ptr(t))
    return t


def c_pack(codes: np.ndarray, fmt: int, gs: int) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    N, K = c.shape
    out = np.zeros((N, c_row_bytes(fmt, K, gs)), dtype=np.uint8)
    bad = _c().orc_pack(_ptr(c), N, K, fmt, gs, _ptr(out))
    if bad != 0:
        raise ValueError(f"orc_pack: {bad}")
    return out


def c_unpack(packed: np.ndarray, N: int, K: int, fmt: int, gs: int) -> np.ndarray:
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros((N, K), dtype=np.uint8)
    if _c().orc_unpack(_ptr(p), N, K, fmt, gs, _ptr(out)) != 0:
        raise ValueError("orc_unpack: invalid arguments")
    return out


def c_code_at(row: np.ndarray, fmt: int, gs: int, k: int) -> int:
    r = np.ascontiguousarray(row, dtype=np.uint8)
    return _c().orc_code_at(_ptr(r), fmt, gs, k)


def c_t5_invalid_bytes(packed: np.ndarray, N: int, K: int, gs: int) -> int:
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    return _c().orc_t5_invalid_bytes(_ptr(p), N, K, gs)


def c_sym_bias(scales, ratio: float) -> np.ndarray:
    s = _bits16(scales)
    f = _c().orc_sym_bias
    out = np.array([f(int(v), float(ratio)) for v in s.ravel()], dtype=np.uint16)
    return out.reshape(s.shape).view(np.float16)


def c_sym_mismatches(scales, biases, ratio: float) -> int:
    s = _bits16(scales)
    b = _bits16(biases)
    N, G = s.shape
    return _c().orc_sym_mismatches(_ptr(s), _ptr(b), N, G, float(ratio))


def c_qmv_rows(x, packed, scales, biases, fmt: int, gs: int, rows=None,
               ratio: float | None = None):
    """(y, bound) float64 [M, len(rows)] for the listed weight rows."""
    xb = _bits16(x)
    M, K = xb.shape
    sb = _bits16(scales)
    N = sb.shape[0]
    bb = None if biases is None else _bits16(biases)
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    r = np.arange(N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    y = np.zeros((M, r.size), dtype=np.float64)
    bound = np.zeros((M, r.size), dtype=np.float64)
    rat = DEFAULT_SYM_RATIO[fmt] if ratio is None else float(ratio)
    rc = _c().orc_qmv_rows(_ptr(xb), _ptr(p), _ptr(sb), None if bb is None else _ptr(bb),
                           rat, M, N, K, fmt, gs, _ptr(r), r.size, _ptr(y), _ptr(bound))
    if rc != 0:
        raise ValueError("orc_qmv_rows: invalid arguments")
    return y, bound
