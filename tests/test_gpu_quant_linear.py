"""GPU checks of the PyTorch drop-in layer against the float64 oracle.

Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" §三 -- quantised
linear layers routed to the fast kernels for every M (decode kernels for
M <= 16, the fused prefill product above), t5 weights accepted (and checked) at
load time; §二.2 -- load-time sym detection drops a bias tensor that equals
-ratio * scale; §二.3 -- ternary 2-bit weights repacked into t5.
Bar: |y_gpu - y| <= 2e-3 * sum_k |x_k w_k| for every output."""
import numpy as np
import pytest

import oracle
import bit_quantized_decode_unpack_gb300 as bqd
from bit_quantized_decode_unpack_gb300 import synth
from _util import assert_within_tolerance, to_dev

pytestmark = pytest.mark.gpu
F1, F2, T5 = bqd.FMT_AFFINE1, bqd.FMT_AFFINE2, bqd.FMT_T5


def QL():
    from bit_quantized_decode_unpack_gb300.quant_linear import QuantLinear
    return QuantLinear


def layer_of(p, detect=True):
    w = bqd.pack(to_dev(p["codes"]), p["fmt"], p["gs"])
    return QL().from_packed(w, to_dev(p["scales"]), to_dev(p["biases"]), p["fmt"], p["gs"], detect=detect)


def check(p, y2d):
    packed = oracle.c_pack(p["codes"], p["fmt"], p["gs"])
    yr, bound = oracle.c_qmv_rows(p["x"], packed, p["scales"], p["biases"], p["fmt"], p["gs"])
    assert_within_tolerance(y2d.cpu().numpy().astype(np.float64), yr, bound, what=p["key"])


@pytest.mark.parametrize("fmt", [F1, F2, T5])
@pytest.mark.parametrize("M", [1, 3, 5, 12, 24])
def test_forward_any_rows_and_leading_dims(fmt, M):
    import torch
    p = synth.problem(fmt, M, 384, 2048, 128)
    layer = layer_of(p)
    x = to_dev(p["x"])
    y = layer(x)
    assert y.shape == (M, 384) and y.dtype == torch.float16
    check(p, y)
    # leading dimensions are flattened into rows and restored
    y3 = layer(x.reshape(1, M, 2048))
    assert y3.shape == (1, M, 384) and torch.equal(y3.view(torch.int16).reshape(M, 384), y.view(torch.int16))


@pytest.mark.parametrize("fmt", [F1, F2])
def test_sym_detection_drops_a_bias_equal_to_the_sym_bias(fmt):
    import torch
    p = synth.problem(fmt, 4, 256, 1024, 64, sym=True)
    r = {F1: 0.5, F2: 1.5}[fmt]
    p["biases"] = oracle.c_sym_bias(p["scales"], r)  # stored fp16(-r * s)
    with_bias = layer_of(p, detect=False)
    detected = layer_of(p, detect=True)
    assert not with_bias.sym and detected.sym
    x = to_dev(p["x"])
    y0, y1 = with_bias(x), detected(x)
    torch.cuda.synchronize()
    # the sym kernel rebuilds the same fp16 bias: bit-identical outputs
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    check(p, y1)
    # one bias off by one ulp: not sym
    b = p["biases"].copy()
    b.view(np.uint16)[3, 2] ^= 1
    p2 = dict(p, biases=b)
    assert not layer_of(p2).sym


def test_t5_layer_rejects_invalid_bytes():
    import torch
    p = synth.problem(T5, 2, 64, 1024, 64, sym=True)
    w = bqd.pack(to_dev(p["codes"]), T5, 64)
    bad = w.clone()
    bad[5, 7] = 250  # >= 243: not a t5 byte
    with pytest.raises(ValueError, match="invalid t5"):
        QL().from_packed(bad, to_dev(p["scales"]), None, T5, 64)
    # a padding trit (the high trits of a group's last byte) must be zero
    bad = w.clone()
    bad[1, 12] = 81 * 2
    with pytest.raises(ValueError, match="invalid t5"):
        QL().from_packed(bad, to_dev(p["scales"]), None, T5, 64)
    # the same check when the weights arrive through load_state_dict
    good = QL().from_packed(w, to_dev(p["scales"]), None, T5, 64)
    fresh = QL()(1024, 64, T5, 64, sym=True, device="cuda")
    sd = {k: v.clone() for k, v in good.state_dict().items()}
    fresh.load_state_dict(sd)
    sd["weight"][0, 0] = 255
    with pytest.raises(RuntimeError, match="invalid t5"):
        fresh.load_state_dict(sd)
    torch.cuda.synchronize()


@pytest.mark.parametrize("gs", [64, 128])
def test_ternary_2bit_repacks_into_t5(gs):
    import torch
    p = synth.problem(F2, 5, 300, 2048, gs)
    rng = np.random.default_rng(gs)
    p["codes"] = rng.integers(0, 3, size=p["codes"].shape).astype(np.uint8)
    # bias = -scale: t5's sym ratio 1, detected and dropped
    p["biases"] = (-p["scales"].astype(np.float32)).astype(np.float16)
    w2 = bqd.pack(to_dev(p["codes"]), F2, gs)
    t5 = QL().from_2bit_ternary(w2, to_dev(p["scales"]), to_dev(p["biases"]), gs)
    assert t5.fmt == T5 and t5.sym and t5.weight.shape[1] == bqd.row_bytes(T5, 2048, gs)
    assert torch.equal(bqd.unpack(t5.weight, 300, 2048, T5, gs).cpu(), torch.from_numpy(p["codes"]))
    check(p, t5(to_dev(p["x"])))
    # a general bias stays as t5's explicit bias tensor
    p["biases"] = synth.biases(rng, F2, p["scales"])
    t5b = QL().from_2bit_ternary(w2, to_dev(p["scales"]), to_dev(p["biases"]), gs)
    assert not t5b.sym
    check(p, t5b(to_dev(p["x"])))
    # a code of 3 is refused
    c3 = p["codes"].copy()
    c3[7, 100] = 3
    with pytest.raises(ValueError, match="not ternary"):
        QL().from_2bit_ternary(bqd.pack(to_dev(c3), F2, gs), to_dev(p["scales"]), None, gs)


def test_state_dict_round_trip_is_bit_identical():
    import torch
    p = synth.problem(F2, 3, 200, 1024, 64)
    layer = layer_of(p)
    fresh = QL()(1024, 200, F2, 64, device="cuda")
    fresh.load_state_dict(layer.state_dict())
    x = to_dev(p["x"])
    assert torch.equal(layer(x).view(torch.int16), fresh(x).view(torch.int16))


def test_functional_form_with_an_explicit_ratio():
    from bit_quantized_decode_unpack_gb300.quant_linear import quantized_matmul
    p = synth.problem(F1, 2, 130, 1024, 64, sym=True)
    w = bqd.pack(to_dev(p["codes"]), F1, 64)
    y = quantized_matmul(to_dev(p["x"]), w, to_dev(p["scales"]), None, F1, 64, ratio=0.25)
    packed = oracle.c_pack(p["codes"], F1, 64)
    yr, bound = oracle.c_qmv_rows(p["x"], packed, p["scales"], None, F1, 64, ratio=0.25)
    assert_within_tolerance(y.cpu().numpy().astype(np.float64), yr, bound)
