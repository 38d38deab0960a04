"""PyTorch drop-in linear layer over the QMV library.

Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析", §三 -- after a
model loads, one patch routes every 1/2-bit affine quantised linear layer to
the fast decode kernels and another lets the loader accept t5 uint8 weights
(and intercepts direct quantised-matmul calls); §二.2 -- a layer whose biases
equal -scale * ratio is served by the sym kernel, which reads no bias tensor;
§二.3 -- t5 weights (and the repack of ternary 2-bit weights into t5).

Here the same roles are a module and a function:

* ``QuantLinear`` holds packed weights, fp16 scales and (unless sym) fp16
  biases as buffers, and its forward is one ``bqd_qmv`` call for any number
  of activation rows; the library's dispatcher picks the kernel (decode
  kernels for M <= 16, the tcgen05 prefill product above).
* ``QuantLinear.from_packed`` runs the load-time checks on the device: sym
  detection (the bias tensor is dropped when every bias is the sym bias) and,
  for t5, byte validation (a bad byte raises instead of decoding to garbage).
* ``QuantLinear.from_2bit_ternary`` repacks 2-bit weights whose codes are all
  in {0, 1, 2} into t5 (a code of 3 raises).
* ``quantized_matmul`` is the functional form for callers that hold the
  tensors themselves.

Everything is argument marshalling: the checks and the products run in the
library's CUDA kernels; the only host work is reading back one count per
check at load time.
"""
from __future__ import annotations

import torch

from . import (FMT_AFFINE1, FMT_AFFINE2, FMT_T5, _fmt, detect_sym, qmv, qmv_sym, repack_2bit_to_t5,
               row_bytes, validate_t5)

# sym ratio r of each format when none is given: bias = -r * scale (the middle
# of the code range: 1-bit {0,1}, 2-bit {0..3}, t5 {0,1,2})
DEFAULT_RATIO = {FMT_AFFINE1: 0.5, FMT_AFFINE2: 1.5, FMT_T5: 1.0}


def _check_layout(fmt: int, in_features: int, out_features: int, group_size: int):
    if fmt not in DEFAULT_RATIO:
        raise ValueError(f"unknown format {fmt}")
    if group_size not in (64, 128):
        raise ValueError(f"group_size must be 64 or 128, got {group_size}")
    if in_features <= 0 or out_features <= 0 or in_features % group_size:
        raise ValueError(f"in_features ({in_features}) must be a positive multiple of group_size "
                         f"({group_size}); out_features ({out_features}) positive")


def _require_cuda(name: str, t):
    if t is not None and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the checks and products run on the device)")


def quantized_matmul(x, weight, scales, biases, fmt, group_size: int, ratio: float | None = None):
    """y[..., n] = sum_k x[..., k] * (scale[n, k/gs] * q[n, k] + bias[n, k/gs]).

    x: fp16 [..., K] on the device; weight: packed uint8 [N, row_bytes];
    scales: fp16 [N, K/gs]; biases: fp16 [N, K/gs] or None (sym: bias =
    -ratio * scale, default ratio of the format).  Returns fp16 [..., N]."""
    fmt = _fmt(fmt)
    K = x.shape[-1]
    x2 = x.reshape(-1, K)
    if not x2.is_contiguous():
        x2 = x2.contiguous()
    if biases is None and ratio is not None and ratio != DEFAULT_RATIO[fmt]:
        y = qmv_sym(x2, weight, scales, ratio, fmt, group_size)
    else:
        y = qmv(x2, weight, scales, biases, fmt, group_size)
    return y.reshape(*x.shape[:-1], scales.shape[0])


class QuantLinear(torch.nn.Module):
    """Linear layer y = x @ W^T with W stored packed (1-bit, 2-bit or t5)."""

    def __init__(self, in_features: int, out_features: int, fmt, group_size: int, sym: bool = False,
                 ratio: float | None = None, device=None):
        super().__init__()
        fmt = _fmt(fmt)
        _check_layout(fmt, in_features, out_features, group_size)
        self.in_features, self.out_features = in_features, out_features
        self.fmt, self.group_size = fmt, group_size
        self.ratio = DEFAULT_RATIO[fmt] if ratio is None else float(ratio)
        G = in_features // group_size
        rb = row_bytes(fmt, in_features, group_size)
        self.register_buffer("weight", torch.zeros((out_features, rb), dtype=torch.uint8, device=device))
        self.register_buffer("scales", torch.zeros((out_features, G), dtype=torch.float16, device=device))
        self.register_buffer("biases", None if sym else
                             torch.zeros((out_features, G), dtype=torch.float16, device=device))

    @property
    def sym(self) -> bool:
        return self.biases is None

    def extra_repr(self) -> str:
        name = {FMT_AFFINE1: "affine1", FMT_AFFINE2: "affine2", FMT_T5: "t5"}[self.fmt]
        return (f"in_features={self.in_features}, out_features={self.out_features}, format={name}, "
                f"group_size={self.group_size}, sym={self.sym}" + (f", ratio={self.ratio}" if self.sym else ""))

    def forward(self, x):
        return quantized_matmul(x, self.weight, self.scales, self.biases, self.fmt, self.group_size,
                                self.ratio if self.sym else None)

    # ---- loading ----------------------------------------------------------------

    @classmethod
    def from_packed(cls, weight, scales, biases, fmt, group_size: int, detect: bool = True,
                    ratio: float | None = None):
        """Layer over already packed device tensors (taken as they are, not copied).

        With ``detect``, biases that all equal fp16(-ratio * scale) are dropped
        so that the sym kernel serves the layer.  t5 weights are validated;
        an invalid byte or padding trit raises ValueError."""
        fmt = _fmt(fmt)
        for name, t in (("weight", weight), ("scales", scales), ("biases", biases)):
            _require_cuda(name, t)
        N, G = scales.shape
        K = G * group_size
        _check_layout(fmt, K, N, group_size)
        if weight.dtype != torch.uint8 or tuple(weight.shape) != (N, row_bytes(fmt, K, group_size)):
            raise ValueError(f"weight must be uint8 [{N}, {row_bytes(fmt, K, group_size)}], "
                             f"got {weight.dtype} {tuple(weight.shape)}")
        if scales.dtype != torch.float16 or (biases is not None and (biases.dtype != torch.float16 or
                                                                     biases.shape != scales.shape)):
            raise ValueError("scales and biases must be fp16 [N, K/group_size]")
        r = DEFAULT_RATIO[fmt] if ratio is None else float(ratio)
        if fmt == FMT_T5:
            bad = int(validate_t5(weight, N, K, group_size).item())
            if bad:
                raise ValueError(f"{bad} invalid t5 bytes (>= 243 or non-zero padding trits)")
        if biases is not None and detect and int(detect_sym(scales, biases, r).item()) == 0:
            biases = None
        layer = cls.__new__(cls)
        torch.nn.Module.__init__(layer)
        layer.in_features, layer.out_features = K, N
        layer.fmt, layer.group_size, layer.ratio = fmt, group_size, r
        layer.register_buffer("weight", weight.contiguous())
        layer.register_buffer("scales", scales.contiguous())
        layer.register_buffer("biases", None if biases is None else biases.contiguous())
        return layer

    @classmethod
    def from_2bit_ternary(cls, w2, scales, biases, group_size: int, detect: bool = True):
        """t5 layer from 2-bit packed weights whose codes are all 0, 1 or 2.

        The codes keep their values (t5 stores them five per byte) and so do
        the scales; biases that equal -scale (the t5 sym ratio 1) are dropped,
        others are kept as the general affine t5 case.  A code of 3 raises."""
        _require_cuda("w2", w2)
        N, G = scales.shape
        K = G * group_size
        w5, status = repack_2bit_to_t5(w2, N, K, group_size)
        n3 = int(status.item())
        if n3:
            raise ValueError(f"{n3} codes equal to 3: the 2-bit weights are not ternary")
        return cls.from_packed(w5, scales, biases, FMT_T5, group_size, detect=detect, ratio=1.0)

    def _load_from_state_dict(self, state_dict, prefix, local_metadata, strict, missing_keys,
                              unexpected_keys, error_msgs):
        super()._load_from_state_dict(state_dict, prefix, local_metadata, strict, missing_keys,
                                      unexpected_keys, error_msgs)
        # t5 weights arriving from a checkpoint are validated like from_packed's
        if self.fmt == FMT_T5 and self.weight.is_cuda and (prefix + "weight") in state_dict:
            bad = int(validate_t5(self.weight, self.out_features, self.in_features, self.group_size).item())
            if bad:
                error_msgs.append(f"{prefix}weight: {bad} invalid t5 bytes (>= 243 or non-zero padding trits)")
