"""CPU checks of the Python binding's argument checks: every tensor handed to
the library must be a CUDA tensor on the activations' device, contiguous, of
the expected dtype and of the exact size the layout implies.  A wrong buffer
(a 1-bit matrix declared as 2-bit, the scales of the other group size, a
transposed view) would otherwise let a kernel read or write past an
allocation.  No GPU is needed: a stand-in object plays a CUDA tensor, and the
checks raise before any device call."""
import pytest
import torch

import bit_quantized_decode_unpack_gb300 as bqd
from bit_quantized_decode_unpack_gb300 import _build


class FakeCuda:
    """Just enough of a torch.Tensor for the binding's checks."""

    def __init__(self, shape, dtype, device="cuda:0", contiguous=True):
        self.shape = torch.Size(shape)
        self.dtype = dtype
        self.device = torch.device(device)
        self.is_cuda = self.device.type == "cuda"
        self._contig = contiguous

    def dim(self):
        return len(self.shape)

    def numel(self):
        n = 1
        for s in self.shape:
            n *= s
        return n

    def element_size(self):
        return torch.empty((), dtype=self.dtype).element_size()

    def is_contiguous(self):
        return self._contig

    def data_ptr(self):  # pragma: no cover - never reached: the checks raise first
        raise AssertionError("a device address was taken before the checks")


F16, U8, I32 = torch.float16, torch.uint8, torch.int32


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return bqd.load()


def good(fmt=2, M=3, N=64, K=512, gs=64):
    return dict(x=FakeCuda((M, K), F16), w=FakeCuda((bqd.packed_bytes(fmt, N, K, gs),), U8),
                s=FakeCuda((N, K // gs), F16), b=FakeCuda((N, K // gs), F16),
                out=FakeCuda((M, N), F16), fmt=fmt, gs=gs)


def call(a):
    return bqd.qmv(a["x"], a["w"], a["s"], a["b"], a["fmt"], a["gs"], out=a["out"])


@pytest.mark.parametrize("field,bad,match", [
    ("x", FakeCuda((3, 512), F16, device="cpu"), "CUDA"),
    ("x", FakeCuda((3, 512), torch.float32), "dtype"),
    ("x", FakeCuda((3, 512), F16, contiguous=False), "contiguous"),
    ("x", FakeCuda((3, 512), F16, device="cuda:1"), "expected"),
    # a 1-bit matrix passed as 2-bit: half the bytes
    ("w", FakeCuda((64 * 512 // 8,), U8), "bytes"),
    # the scales of the other group size
    ("s", FakeCuda((64, 512 // 128), F16), "shape"),
    ("s", FakeCuda((64, 8), torch.bfloat16), "dtype"),
    ("b", FakeCuda((64, 4), F16), "shape"),
    ("b", FakeCuda((64, 8), F16, contiguous=False), "contiguous"),
    ("out", FakeCuda((64, 3), F16), "shape"),
    ("out", FakeCuda((3, 64), torch.float32), "dtype"),
    ("out", FakeCuda((3, 64), F16, contiguous=False), "contiguous"),
])
def test_qmv_rejects_a_wrong_tensor(field, bad, match):
    a = good()
    a[field] = bad
    with pytest.raises(ValueError, match=match):
        call(a)


def test_qmv_rejects_layout_errors():
    a = good()
    a["gs"] = 32
    with pytest.raises(ValueError, match="group_size"):
        call(a)
    a = good(K=512)
    a["x"] = FakeCuda((3, 520), F16)  # K not a multiple of the group size
    with pytest.raises(ValueError, match="multiple"):
        call(a)
    a = good()
    a["fmt"] = 7
    with pytest.raises(ValueError, match="format"):
        call(a)
    a = good()
    a["x"] = FakeCuda((512,), F16)
    with pytest.raises(ValueError, match="2-D"):
        call(a)


def test_t5_weight_size_is_checked():
    a = good(fmt=3)
    a["b"] = None
    a["w"] = FakeCuda((bqd.packed_bytes(2, 64, 512, 64),), U8)  # 2-bit bytes declared as t5
    with pytest.raises(ValueError, match="bytes"):
        call(a)


def test_sym_variant_is_checked_too():
    a = good()
    with pytest.raises(ValueError, match="shape"):
        bqd.qmv_sym(a["x"], a["w"], FakeCuda((64, 4), F16), 1.5, 2, 64, out=a["out"])


def test_layout_entry_points_are_checked():
    with pytest.raises(ValueError, match="dtype"):
        bqd.pack(FakeCuda((4, 128), I32), 2, 64)
    with pytest.raises(ValueError, match="bytes"):
        bqd.pack(FakeCuda((4, 128), U8), 2, 64, out=FakeCuda((4, 16), U8))
    with pytest.raises(ValueError, match="bytes"):
        bqd.unpack(FakeCuda((4, 16), U8), 4, 128, 2, 64)
    with pytest.raises(ValueError, match="shape"):
        bqd.unpack(FakeCuda((4, 32), U8), 4, 128, 2, 64, out=FakeCuda((4, 64), U8))
    with pytest.raises(ValueError, match="bytes"):
        bqd.repack_2bit_to_t5(FakeCuda((4, 16), U8), 4, 128, 64)
    with pytest.raises(ValueError, match="dtype"):
        bqd.repack_2bit_to_t5(FakeCuda((4, 32), U8), 4, 128, 64, out=FakeCuda((4, 26), U8),
                              status=FakeCuda((1,), torch.int64))
    with pytest.raises(ValueError, match="bytes"):
        bqd.validate_t5(FakeCuda((4, 25), U8), 4, 128, 64)
    with pytest.raises(ValueError, match="shape"):
        bqd.detect_sym(FakeCuda((4, 2), F16), FakeCuda((4, 3), F16), 1.5)
    with pytest.raises(ValueError, match="at least"):
        bqd.detect_sym(FakeCuda((4, 2), F16), FakeCuda((4, 2), F16), 1.5, out=FakeCuda((0,), I32))


def test_verification_outputs_are_checked():
    lg = FakeCuda((2, 3, 10), F16)
    d = FakeCuda((2, 2), I32)
    with pytest.raises(ValueError, match="shape"):
        bqd.spec_decode_verify(lg, d, accepted=FakeCuda((3,), I32))
    with pytest.raises(ValueError, match="int32"):
        bqd.spec_decode_verify(lg, FakeCuda((2, 2), torch.int64))
    with pytest.raises(ValueError, match="shape"):
        bqd.spec_decode_verify(lg, d, argmax_out=FakeCuda((2, 2), I32))
