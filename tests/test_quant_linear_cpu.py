"""Host-side logic of the PyTorch drop-in layer (no compute call, no GPU):
layout checks, buffer shapes and dtypes, the sym flag, and that the load-time
constructors refuse host tensors (their checks run on the device).

Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" §三 (the layer
patch and the t5 load patch), §二.2 (sym layers read no bias tensor)."""
import pytest
import torch

import bit_quantized_decode_unpack_gb300 as bqd
from bit_quantized_decode_unpack_gb300 import _build


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return bqd.load()


def QL():
    from bit_quantized_decode_unpack_gb300.quant_linear import QuantLinear
    return QuantLinear


@pytest.mark.parametrize("fmt,gs,rb", [("affine1", 64, 640), ("affine2", 128, 1280), ("t5", 64, 80 * 13),
                                       ("t5", 128, 40 * 26)])
def test_buffers_follow_the_packed_layout(fmt, gs, rb):
    layer = QL()(5120, 300, fmt, gs)
    assert layer.weight.dtype == torch.uint8 and tuple(layer.weight.shape) == (300, rb)
    assert rb == bqd.row_bytes(fmt, 5120, gs)
    assert layer.scales.dtype == torch.float16 and tuple(layer.scales.shape) == (300, 5120 // gs)
    assert tuple(layer.biases.shape) == (300, 5120 // gs) and not layer.sym
    assert set(layer.state_dict()) == {"weight", "scales", "biases"}


def test_sym_layer_has_no_bias_buffer_and_keeps_its_ratio():
    layer = QL()(1024, 16, "affine2", 64, sym=True)
    assert layer.sym and layer.biases is None and layer.ratio == 1.5
    assert set(layer.state_dict()) == {"weight", "scales"}
    assert "sym=True" in repr(layer) and "ratio=1.5" in repr(layer)
    assert QL()(1024, 16, "affine1", 64, sym=True, ratio=0.25).ratio == 0.25
    assert QL()(1024, 16, "t5", 64, sym=True).ratio == 1.0


@pytest.mark.parametrize("args", [(1000, 16, "affine2", 64), (1024, 16, "affine2", 32), (1024, 0, "t5", 64),
                                  (1024, 16, 7, 64)])
def test_bad_layouts_raise(args):
    with pytest.raises((ValueError, KeyError)):
        QL()(*args)


def test_load_time_constructors_refuse_host_tensors():
    w = torch.zeros((16, 256), dtype=torch.uint8)
    s = torch.zeros((16, 16), dtype=torch.float16)
    with pytest.raises(ValueError, match="CUDA"):
        QL().from_packed(w, s, None, "affine2", 64)
    with pytest.raises(ValueError, match="CUDA"):
        QL().from_2bit_ternary(w, s, None, 64)
