"""CPU-side checks of the C ABI: the library loads, exports every symbol that
include/bqd.h declares, and its host-only entry points and host-side argument
validation behave as documented.  No compute call is made (no GPU here)."""
import ctypes
import re
from pathlib import Path

import pytest

import bit_quantized_decode_unpack_gb300 as bqd
from bit_quantized_decode_unpack_gb300 import _build

ROOT = Path(__file__).resolve().parent.parent
HEADERS = sorted((ROOT / "include").glob("*.h"))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return bqd.load()


def _declared_symbols():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names |= set(re.findall(r"\b(bqd_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared_symbols()
    for want in ["bqd_abi_version", "bqd_status_string", "bqd_packed_bytes", "bqd_qmv", "bqd_qmv_sym",
                 "bqd_pack", "bqd_unpack", "bqd_repack_2bit_to_t5", "bqd_validate_t5", "bqd_detect_sym"]:
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_symbols():
        assert hasattr(lib, name), name
        # and as a plain C symbol (extern "C", not mangled)
        ctypes.cast(getattr(lib, name), ctypes.c_void_p)


def test_abi_version_matches_header(lib):
    text = (ROOT / "include" / "bqd.h").read_text()
    v = int(re.search(r"#define BQD_ABI_VERSION (\d+)", text).group(1))
    assert lib.bqd_abi_version() == v == bqd.ABI_VERSION


def test_status_strings(lib):
    for st in range(0, 9):
        assert bqd.status_string(st)
    assert bqd.status_string(0) == "ok"
    assert "unknown" in bqd.status_string(99)


@pytest.mark.parametrize("fmt,N,K,gs,want", [
    (1, 256, 512, 64, 256 * 512 // 8),
    (2, 17408, 5120, 64, 17408 * 5120 // 4),
    (3, 17408, 5120, 64, 17408 * 80 * 13),
    (3, 5120, 17408, 128, 5120 * 136 * 26),
    (3, 1, 64, 64, 13),
    (3, 1, 128, 128, 26),
    (1, 0, 512, 64, 0),
    (2, 5, 0, 64, 0),
])
def test_packed_bytes(lib, fmt, N, K, gs, want):
    assert bqd.packed_bytes(fmt, N, K, gs) == want


@pytest.mark.parametrize("args", [(0, 1, 64, 64), (4, 1, 64, 64), (2, 1, 96, 64), (2, 1, 64, 32),
                                  (2, -1, 64, 64), (2, 1, -64, 64)])
def test_packed_bytes_invalid(lib, args):
    assert bqd.packed_bytes(*args) == 0


def _qmv(lib, x=1, w=1, s=1, b=None, M=1, N=1, K=64, fmt=2, gs=64, out=1):
    vp = lambda v: None if v is None else ctypes.c_void_p(v)
    return lib.bqd_qmv(vp(x and 0x1000), vp(w and 0x2000), vp(s and 0x3000), vp(b), M, N, K, fmt, gs,
                       vp(out and 0x4000), None)


def test_qmv_host_validation_rejects_before_any_launch(lib):
    INV, ALIGN = 1, 3
    assert _qmv(lib, fmt=0) == INV
    assert _qmv(lib, gs=32) == INV
    assert _qmv(lib, K=96) == INV           # K % gs != 0
    assert _qmv(lib, M=-1) == INV
    assert _qmv(lib, out=0) == INV          # null output
    assert _qmv(lib, x=0) == INV            # null input
    assert _qmv(lib, w=0) == INV
    assert _qmv(lib, s=0) == INV
    vp = ctypes.c_void_p
    # misaligned x / out / weights
    assert lib.bqd_qmv(vp(0x1001), vp(0x2000), vp(0x3000), None, 1, 1, 64, 2, 64, vp(0x4000), None) == ALIGN
    assert lib.bqd_qmv(vp(0x1000), vp(0x2000), vp(0x3000), None, 1, 1, 64, 2, 64, vp(0x4008), None) == ALIGN
    assert lib.bqd_qmv(vp(0x1000), vp(0x2004), vp(0x3000), None, 1, 1, 64, 2, 64, vp(0x4000), None) == ALIGN
    assert lib.bqd_qmv(vp(0x1000), vp(0x2000), vp(0x3001), None, 1, 1, 64, 2, 64, vp(0x4000), None) == ALIGN
    # empty problems are valid no-ops: nothing is launched, no pointer needed
    assert lib.bqd_qmv(None, None, None, None, 0, 7, 64, 2, 64, None, None) == 0
    assert lib.bqd_qmv(None, None, None, None, 3, 0, 64, 2, 64, None, None) == 0
    # non-finite sym ratio
    assert lib.bqd_qmv_sym(vp(0x1000), vp(0x2000), vp(0x3000), ctypes.c_float(float("nan")), 1, 1, 64,
                           2, 64, vp(0x4000), None) == INV


def test_other_entry_points_validate_on_host(lib):
    INV = 1
    vp = ctypes.c_void_p
    assert lib.bqd_pack(None, 4, 64, 2, 64, vp(0x1000), None) == INV
    assert lib.bqd_pack(vp(0x1000), 4, 96, 2, 64, vp(0x2000), None) == INV
    assert lib.bqd_pack(None, 0, 64, 2, 64, None, None) == 0
    assert lib.bqd_unpack(vp(0x1000), 4, 64, 9, 64, vp(0x2000), None) == INV
    assert lib.bqd_repack_2bit_to_t5(vp(0x1000), 4, 64, 64, vp(0x2000), None, None) == INV
    assert lib.bqd_validate_t5(vp(0x1000), 4, 64, 48, vp(0x2000), None) == INV
    assert lib.bqd_detect_sym(vp(0x1000), None, 4, 2, ctypes.c_float(1.5), vp(0x2000), None) == INV
    assert lib.bqd_detect_sym(vp(0x1000), vp(0x1000), 4, 2, ctypes.c_float(1.5), None, None) == INV


def test_binding_names_match_the_c_abi():
    for name in _declared_symbols():
        assert hasattr(bqd, name[len("bqd_"):]), name


def test_spec_decode_verify_validates_on_host(lib):
    """bqd_spec_decode_verify rejects bad arguments before any launch (no GPU
    is touched for these), and B == 0 is a no-op."""
    INV, ALIGN = 1, 3
    vp = ctypes.c_void_p
    f = lib.bqd_spec_decode_verify
    ok = dict(lg=0x1000, dt=1, dr=0x2000, B=2, D=3, V=100, a=0x3000, n=0x4000, am=None)

    def call(**kw):
        a = dict(ok, **kw)
        p = lambda v: None if v is None else vp(v)
        return f(p(a["lg"]), a["dt"], p(a["dr"]), a["B"], a["D"], a["V"], p(a["a"]), p(a["n"]), p(a["am"]), None)

    assert call(dt=3) == INV               # unknown logits type
    assert call(B=-1) == INV
    assert call(D=-1) == INV
    assert call(D=4096) == INV             # above the documented maximum
    assert call(V=0) == INV
    assert call(V=(1 << 31)) == INV
    assert call(lg=None) == INV
    assert call(a=None) == INV
    assert call(n=None) == INV
    assert call(dr=None) == INV            # drafts are needed when D > 0
    assert call(lg=0x1001) == ALIGN        # fp16 logits need 2-byte alignment
    assert call(lg=0x1002, dt=2) == ALIGN  # fp32 logits need 4-byte alignment
    assert call(a=0x3002) == ALIGN
    assert call(B=0, lg=None, dr=None, a=None, n=None) == 0


def test_options_set_get_and_validate(lib):
    """bqd_set_option / bqd_get_option: process-wide controls for tests and
    measurements, validated on the host."""
    INV = 1
    old = {o: lib.bqd_get_option(o) for o in (1, 2, 3, 4)}
    try:
        for k in (0, 1, 2, 3, 4):
            assert lib.bqd_set_option(1, k) == 0 and lib.bqd_get_option(1) == k
        assert lib.bqd_set_option(1, 5) == INV and lib.bqd_set_option(1, -1) == INV
        assert lib.bqd_set_option(2, 2) == 0 and lib.bqd_get_option(2) == 2
        assert lib.bqd_set_option(2, 3) == INV
        assert lib.bqd_set_option(3, 250) == 0 and lib.bqd_get_option(3) == 250
        assert lib.bqd_set_option(3, 0) == 0 and lib.bqd_get_option(3) == 1_000_000_000  # default restored
        assert lib.bqd_set_option(3, -5) == INV
        assert lib.bqd_set_option(99, 1) == INV and lib.bqd_get_option(99) == -1
        # the binding's names map onto the same values
        bqd.force_kernel("qmm")
        assert lib.bqd_get_option(bqd.OPT_KERNEL) == bqd.KERNELS["qmm"]
        bqd.force_kernel(None)
        assert lib.bqd_get_option(bqd.OPT_KERNEL) == 0
    finally:
        for o, v in old.items():
            lib.bqd_set_option(o, v)
