"""GB300-native low-bit quantized matrix-vector product (QMV).

Thin Python binding over ``libbqd.so`` (the C ABI declared in ``include/bqd.h``).
Every function here only marshals arguments -- torch tensors supply device
memory and the current CUDA stream -- and calls the entry point of the same
name; every step of the computation runs in the library's CUDA kernels.
There is no CPU fallback: if the library is not built, calls raise.

Operation (page "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析",
§二.1-§二.3):  y[m, n] = sum_k x[m, k] * (scale[n, k/gs] * q[n, k] + bias[n, k/gs])
with q packed as 1-bit / 2-bit LSB-first uint32 codes or as "t5" trits
(five per byte, 13/26 bytes per 64/128-weight group).
"""
from __future__ import annotations

import ctypes
import threading
from pathlib import Path

FMT_AFFINE1 = 1
FMT_AFFINE2 = 2
FMT_T5 = 3
FORMATS = {"affine1": FMT_AFFINE1, "affine2": FMT_AFFINE2, "t5": FMT_T5}
DTYPE_F16 = 1
DTYPE_F32 = 2

BQD_OK = 0
OPT_KERNEL, OPT_T5_STAGES, OPT_WAIT_LIMIT_NS, OPT_DEBUG_PLAN = 1, 2, 3, 4
KERNELS = {None: 0, "auto": 0, "generic": 1, "mma": 2, "tma": 3, "qmm": 4}
ABI_VERSION = 1  # must match BQD_ABI_VERSION in include/bqd.h

_PKG = Path(__file__).resolve().parent
LIB_PATH = _PKG / "_lib" / "libbqd.so"

_lock = threading.Lock()
_lib = None


class BqdError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


def load() -> ctypes.CDLL:
    """Load libbqd.so (built by ``_build.build()`` / ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not LIB_PATH.exists():
            raise RuntimeError(f"{LIB_PATH} is not built: run `python -c \"import __graft_entry__ as g; "
                               f"g.build()\"` (nvcc, sm_103a) before using the library")
        lib = ctypes.CDLL(str(LIB_PATH))
        i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        lib.bqd_abi_version.argtypes = []
        lib.bqd_abi_version.restype = i32
        lib.bqd_status_string.argtypes = [i32]
        lib.bqd_status_string.restype = ctypes.c_char_p
        lib.bqd_packed_bytes.argtypes = [i32, i64, i64, i32]
        lib.bqd_packed_bytes.restype = sz
        lib.bqd_qmv.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i32, vp, vp]
        lib.bqd_qmv.restype = i32
        lib.bqd_qmv_sym.argtypes = [vp, vp, vp, ctypes.c_float, i64, i64, i64, i32, i32, vp, vp]
        lib.bqd_qmv_sym.restype = i32
        lib.bqd_pack.argtypes = [vp, i64, i64, i32, i32, vp, vp]
        lib.bqd_pack.restype = i32
        lib.bqd_unpack.argtypes = [vp, i64, i64, i32, i32, vp, vp]
        lib.bqd_unpack.restype = i32
        lib.bqd_repack_2bit_to_t5.argtypes = [vp, i64, i64, i32, vp, vp, vp]
        lib.bqd_repack_2bit_to_t5.restype = i32
        lib.bqd_validate_t5.argtypes = [vp, i64, i64, i32, vp, vp]
        lib.bqd_validate_t5.restype = i32
        lib.bqd_detect_sym.argtypes = [vp, vp, i64, i64, ctypes.c_float, vp, vp]
        lib.bqd_detect_sym.restype = i32
        lib.bqd_spec_decode_verify.argtypes = [vp, i32, vp, i64, i64, i64, vp, vp, vp, vp]
        lib.bqd_spec_decode_verify.restype = i32
        lib.bqd_device_status.argtypes = [vp]
        lib.bqd_device_status.restype = i32
        lib.bqd_set_option.argtypes = [i32, i64]
        lib.bqd_set_option.restype = i32
        lib.bqd_get_option.argtypes = [i32]
        lib.bqd_get_option.restype = i64
        if lib.bqd_abi_version() != ABI_VERSION:
            raise RuntimeError(f"libbqd ABI {lib.bqd_abi_version()} != binding ABI {ABI_VERSION}")
        _lib = lib
        return lib


def _check(fn: str, status: int):
    if status != BQD_OK:
        raise BqdError(fn, status)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def _need(t, name, *, dtype=None, shape=None, nbytes=None, device=None, min_numel=None):
    """Check a tensor argument before its address is handed to the library:
    a CUDA tensor, contiguous, of the expected dtype, shape or byte size, on
    the expected device.  A wrong buffer would otherwise let a kernel read or
    write past an allocation.  Raises ValueError."""
    if t is None:
        raise ValueError(f"{name}: a tensor is required")
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{name}: must be a CUDA tensor (got device {getattr(t, 'device', None)})")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous (row-major, no strides)")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if nbytes is not None and t.numel() * t.element_size() != nbytes:
        raise ValueError(f"{name}: {t.numel() * t.element_size()} bytes, expected {nbytes}")
    if min_numel is not None and t.numel() < min_numel:
        raise ValueError(f"{name}: {t.numel()} elements, expected at least {min_numel}")
    return t


def _check_group(K: int, group_size: int):
    if group_size not in (64, 128):
        raise ValueError(f"group_size must be 64 or 128, got {group_size}")
    if K % group_size != 0:
        raise ValueError(f"K={K} is not a multiple of group_size={group_size}")


def _check_qmv_args(x, w_packed, scales, biases, fmt, group_size, out):
    import torch
    f16 = torch.float16
    if getattr(x, "dim", lambda: 0)() != 2:
        raise ValueError("x must be a 2-D fp16 tensor [M, K]")
    if getattr(scales, "dim", lambda: 0)() != 2:
        raise ValueError("scales must be a 2-D fp16 tensor [N, G]")
    M, K = x.shape
    N, G = scales.shape
    f = _fmt(fmt)
    if f not in FORMATS.values():
        raise ValueError(f"unknown format {fmt!r}")
    _check_group(K, group_size)
    dev = x.device
    _need(x, "x", dtype=f16, device=dev)
    _need(scales, "scales", dtype=f16, shape=(N, K // group_size), device=dev)
    _need(w_packed, "w_packed", nbytes=packed_bytes(f, N, K, group_size), device=dev)
    if biases is not None:
        _need(biases, "biases", dtype=f16, shape=(N, G), device=dev)
    if out is not None:
        _need(out, "out", dtype=f16, shape=(M, N), device=dev)
    return M, N, K


# ---- host-only entry points ----------------------------------------------

def abi_version() -> int:
    return load().bqd_abi_version()


def status_string(status: int) -> str:
    return load().bqd_status_string(int(status)).decode()


def packed_bytes(fmt, N: int, K: int, group_size: int) -> int:
    return int(load().bqd_packed_bytes(_fmt(fmt), N, K, group_size))


def row_bytes(fmt, K: int, group_size: int) -> int:
    return packed_bytes(fmt, 1, K, group_size)


# ---- device entry points ---------------------------------------------------

def qmv(x, w_packed, scales, biases, fmt, group_size: int, out=None, stream=None):
    """y = x @ dequant(W)^T, fp16 [M, N].  ``biases=None`` selects the sym
    path (no bias tensor read, default ratio of the format)."""
    import torch
    M, N, K = _check_qmv_args(x, w_packed, scales, biases, fmt, group_size, out)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _check("bqd_qmv", load().bqd_qmv(_ptr(x), _ptr(w_packed), _ptr(scales), _ptr(biases), M, N, K,
                                     _fmt(fmt), group_size, _ptr(out), _stream(stream)))
    return out


def qmv_sym(x, w_packed, scales, ratio: float, fmt, group_size: int, out=None, stream=None):
    """Sym variant with an explicit ratio (bias = -ratio * scale, not read)."""
    import torch
    M, N, K = _check_qmv_args(x, w_packed, scales, None, fmt, group_size, out)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=x.device)
    _check("bqd_qmv_sym", load().bqd_qmv_sym(_ptr(x), _ptr(w_packed), _ptr(scales), float(ratio), M, N,
                                             K, _fmt(fmt), group_size, _ptr(out), _stream(stream)))
    return out


def pack(codes, fmt, group_size: int, out=None, stream=None):
    """codes uint8 [N, K] (device) -> packed uint8 [N, row_bytes] (device)."""
    import torch
    if getattr(codes, "dim", lambda: 0)() != 2:
        raise ValueError("codes must be a 2-D uint8 tensor [N, K]")
    N, K = codes.shape
    _check_group(K, group_size)
    _need(codes, "codes", dtype=torch.uint8)
    rb = row_bytes(fmt, K, group_size)
    if out is None:
        out = torch.empty((N, rb), dtype=torch.uint8, device=codes.device)
    _need(out, "out", nbytes=N * rb, device=codes.device)
    _check("bqd_pack", load().bqd_pack(_ptr(codes), N, K, _fmt(fmt), group_size, _ptr(out),
                                       _stream(stream)))
    return out


def unpack(w_packed, N: int, K: int, fmt, group_size: int, out=None, stream=None):
    import torch
    _check_group(K, group_size)
    _need(w_packed, "w_packed", nbytes=packed_bytes(fmt, N, K, group_size))
    if out is None:
        out = torch.empty((N, K), dtype=torch.uint8, device=w_packed.device)
    _need(out, "out", dtype=torch.uint8, shape=(N, K), device=w_packed.device)
    _check("bqd_unpack", load().bqd_unpack(_ptr(w_packed), N, K, _fmt(fmt), group_size, _ptr(out),
                                           _stream(stream)))
    return out


def repack_2bit_to_t5(w2, N: int, K: int, group_size: int, out=None, status=None, stream=None):
    """-> (w_t5 uint8 [N, G*ceil(gs/5)], status int32[1] = count of codes equal to 3)."""
    import torch
    _check_group(K, group_size)
    _need(w2, "w2", nbytes=packed_bytes(FMT_AFFINE2, N, K, group_size))
    if out is None:
        out = torch.empty((N, row_bytes(FMT_T5, K, group_size)), dtype=torch.uint8, device=w2.device)
    if status is None:
        status = torch.empty((1,), dtype=torch.int32, device=w2.device)
    _need(out, "out", nbytes=packed_bytes(FMT_T5, N, K, group_size), device=w2.device)
    _need(status, "status", dtype=torch.int32, device=w2.device, min_numel=1)
    _check("bqd_repack_2bit_to_t5", load().bqd_repack_2bit_to_t5(
        _ptr(w2), N, K, group_size, _ptr(out), _ptr(status), _stream(stream)))
    return out, status


def validate_t5(w_t5, N: int, K: int, group_size: int, status=None, stream=None):
    """-> int32[1] device tensor: number of invalid t5 bytes."""
    import torch
    _check_group(K, group_size)
    _need(w_t5, "w_t5", nbytes=packed_bytes(FMT_T5, N, K, group_size))
    if status is None:
        status = torch.empty((1,), dtype=torch.int32, device=w_t5.device)
    _need(status, "status", dtype=torch.int32, device=w_t5.device, min_numel=1)
    _check("bqd_validate_t5", load().bqd_validate_t5(_ptr(w_t5), N, K, group_size, _ptr(status),
                                                     _stream(stream)))
    return status


def detect_sym(scales, biases, ratio: float, out=None, stream=None):
    """-> int32[1] device tensor: number of biases != fp16(-ratio * scale)."""
    import torch
    if getattr(scales, "dim", lambda: 0)() != 2:
        raise ValueError("scales must be a 2-D fp16 tensor [N, G]")
    N, G = scales.shape
    _need(scales, "scales", dtype=torch.float16)
    _need(biases, "biases", dtype=torch.float16, shape=(N, G), device=scales.device)
    if out is None:
        out = torch.empty((1,), dtype=torch.int32, device=scales.device)
    _need(out, "out", dtype=torch.int32, device=scales.device, min_numel=1)
    _check("bqd_detect_sym", load().bqd_detect_sym(_ptr(scales), _ptr(biases), N, G, float(ratio),
                                                   _ptr(out), _stream(stream)))
    return out


def spec_decode_verify(logits, draft, accepted=None, next_token=None, argmax_out=None, stream=None):
    """Greedy speculative-decoding verification (bqd_spec_decode_verify).

    logits fp16|fp32 [B, D+1, V], draft int32 [B, D] (device).  Returns
    (accepted int32 [B], next_token int32 [B]); pass ``argmax_out`` (int32
    [B, D+1]) to also receive every row's argmax."""
    import torch
    if getattr(logits, "dim", lambda: 0)() != 3:
        raise ValueError("logits must be a 3-D tensor [B, D+1, V]")
    B, D1, V = logits.shape
    _need(logits, "logits")
    if logits.dtype == torch.float16:
        dt = DTYPE_F16
    elif logits.dtype == torch.float32:
        dt = DTYPE_F32
    else:
        raise TypeError(f"logits must be float16 or float32, got {logits.dtype}")
    if draft.dtype != torch.int32 or tuple(draft.shape) != (B, D1 - 1):
        raise ValueError(f"draft must be int32 [{B}, {D1 - 1}], got {draft.dtype} {tuple(draft.shape)}")
    dev = logits.device
    if D1 > 1:
        _need(draft, "draft", dtype=torch.int32, device=dev)
    if accepted is not None:
        _need(accepted, "accepted", dtype=torch.int32, shape=(B,), device=dev)
    if next_token is not None:
        _need(next_token, "next_token", dtype=torch.int32, shape=(B,), device=dev)
    if argmax_out is not None:
        _need(argmax_out, "argmax_out", dtype=torch.int32, shape=(B, D1), device=dev)
    if accepted is None:
        accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty((B,), dtype=torch.int32, device=dev)
    _check("bqd_spec_decode_verify", load().bqd_spec_decode_verify(
        _ptr(logits), dt, _ptr(draft) if D1 > 1 else None, B, D1 - 1, V, _ptr(accepted), _ptr(next_token),
        _ptr(argmax_out), _stream(stream)))
    return accepted, next_token


def set_option(option: int, value: int) -> None:
    """Process-wide option (bqd_set_option): OPT_KERNEL (see KERNELS),
    OPT_T5_STAGES, OPT_WAIT_LIMIT_NS, OPT_DEBUG_PLAN."""
    _check("bqd_set_option", load().bqd_set_option(int(option), int(value)))


def get_option(option: int) -> int:
    return int(load().bqd_get_option(int(option)))


def force_kernel(name) -> None:
    """Force one kernel family for every QMV call (None or "auto": the
    dispatcher picks).  For tests and measurements."""
    set_option(OPT_KERNEL, KERNELS[name])


def device_status(stream=None) -> int:
    """Synchronise the stream; BQD_OK, or the status of an expired bounded
    device-side wait since the previous call (see include/bqd.h)."""
    return int(load().bqd_device_status(_stream(stream)))
