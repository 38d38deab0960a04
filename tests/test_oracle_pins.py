"""Pins for the float64 oracle: checks against what the page and mathematics
fix, never against the oracle's own formula retyped.

Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" (oMLX Bonsai custom
kernels: the fast QMV path for the Qwen family), §二.1-§二.3, §四.

Each pin is chosen so that a plausible slip in the oracle (bit order, trit
order, a dropped bias, a wrong sign, a transposed operand, a wrong group
index) fails at least one of them; ``test_planted_mistakes_are_caught`` plants
such slips in a copy of the NumPy oracle and checks that they are caught.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from oracle import oracle as npo
from bit_quantized_decode_unpack_gb300 import synth
from conftest import read_golden

F1, F2, T5 = oracle.FMT_AFFINE1, oracle.FMT_AFFINE2, oracle.FMT_T5


# ---- fp16 conversions: against NumPy's own IEEE half implementation --------

def test_half_to_double_all_bit_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.c_half_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)])


def test_float_to_half_rne_matches_numpy():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.normal(0, 1, 20000), rng.normal(0, 1e-5, 5000), rng.normal(0, 3e4, 5000),
        # exact ties between neighbouring halves, subnormal ties, overflow edge
        (np.arange(1024, 2048, dtype=np.float64) + 0.5) * 2.0 ** -10,
        (np.arange(0, 1024, dtype=np.float64) + 0.5) * 2.0 ** -24,
        [65504.0, 65519.0, 65520.0, 1e9, -1e9, 0.0, -0.0, 2.0 ** -25, 2.0 ** -26],
    ]).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.c_float_to_half_bits(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---- t5 byte code: exhaustive ------------------------------------------------

def test_t5_all_243_bytes_are_a_bijection_on_trit_tuples():
    seen = {}
    for b in range(243):
        t = tuple(int(v) for v in oracle.c_t5_decode(b))
        assert all(v in (0, 1, 2) for v in t)
        assert oracle.c_t5_encode(np.array(t)) == b
        seen[t] = b
    assert set(seen) == set(itertools.product(range(3), repeat=5))
    # base-3 numeral with the first weight as the least significant digit,
    # parsed by Python's own int(..., 3)
    for t, b in seen.items():
        assert int("".join(str(d) for d in reversed(t)), 3) == b


def test_t5_golden_bytes():
    for line in read_golden("t5_bytes.txt"):
        *t, b = (int(v) for v in line.split())
        assert oracle.c_t5_encode(np.array(t)) == b
        assert tuple(oracle.c_t5_decode(b)) == tuple(t)
        # NumPy twin on a one-group row with these trits first
        codes = np.zeros((1, 64), dtype=np.uint8)
        codes[0, :5] = t
        assert npo.pack(codes, T5, 64)[0, 0] == b


# ---- packing: golden rows, single-bit probes, round trips --------------------

def _hexbytes(s):
    return np.array([int(v, 16) for v in s.split()], dtype=np.uint8)


def test_pack_1bit_golden():
    lines = dict(l.split(":", 1) for l in read_golden("pack_1bit.txt"))
    codes = np.zeros((1, 64), dtype=np.uint8)
    codes[0, [int(v) for v in lines["ones"].split()]] = 1
    want = _hexbytes(lines["bytes"])
    assert np.array_equal(oracle.c_pack(codes, F1, 64)[0], want)
    assert np.array_equal(npo.pack(codes, F1, 64)[0], want)
    assert np.array_equal(oracle.c_unpack(want[None], 1, 64, F1, 64), codes)
    assert np.array_equal(npo.unpack(want[None], 1, 64, F1, 64), codes)


def test_pack_2bit_golden():
    lines = dict(l.split(":", 1) for l in read_golden("pack_2bit.txt"))
    codes = np.array([[int(v) for v in lines["codes"].split()]], dtype=np.uint8)
    want = _hexbytes(lines["bytes"])
    assert np.array_equal(oracle.c_pack(codes, F2, 64)[0], want)
    assert np.array_equal(npo.pack(codes, F2, 64)[0], want)
    assert np.array_equal(oracle.c_unpack(want[None], 1, 64, F2, 64), codes)
    assert np.array_equal(npo.unpack(want[None], 1, 64, F2, 64), codes)


@pytest.mark.parametrize("gs", [64, 128])
def test_pack_t5_golden(gs):
    lines = dict(l.split(":", 1) for l in read_golden("pack_t5.txt"))
    codes = np.zeros((1, gs), dtype=np.uint8)
    for item in lines[f"gs{gs}_trits"].split():
        k, v = item.split("=")
        codes[0, int(k)] = int(v)
    want = _hexbytes(lines[f"gs{gs}_bytes"])
    assert np.array_equal(oracle.c_pack(codes, T5, gs)[0], want)
    assert np.array_equal(npo.pack(codes, T5, gs)[0], want)
    assert np.array_equal(oracle.c_unpack(want[None], 1, gs, T5, gs), codes)
    assert np.array_equal(npo.unpack(want[None], 1, gs, T5, gs), codes)


@pytest.mark.parametrize("fmt,bits", [(F1, 1), (F2, 2)])
def test_single_code_probes(fmt, bits):
    """A single non-zero code at k sets exactly the bits of word k // (32/bits)
    given by integer arithmetic (LSB-first)."""
    K = 128
    per_word = 32 // bits
    for k in range(K):
        for c in range(1, 2 ** bits):
            codes = np.zeros((1, K), dtype=np.uint8)
            codes[0, k] = c
            words = oracle.c_pack(codes, fmt, 64).view("<u4")[0]
            want = np.zeros(K // per_word, dtype=np.uint64)
            want[k // per_word] = c << (bits * (k % per_word))
            assert np.array_equal(words.astype(np.uint64), want), (k, c)


@pytest.mark.parametrize("fmt", [F1, F2, T5])
@pytest.mark.parametrize("gs", [64, 128])
def test_pack_round_trip_and_c_numpy_agree(fmt, gs):
    rng = np.random.default_rng(fmt * 10 + gs)
    for N, K in [(1, gs), (3, 2 * gs), (7, 5 * gs), (16, 640)]:
        if K % gs:
            continue
        codes = synth.codes(rng, fmt, N, K)
        pc, pn = oracle.c_pack(codes, fmt, gs), npo.pack(codes, fmt, gs)
        assert pc.shape == (N, npo.row_bytes(fmt, K, gs))
        assert np.array_equal(pc, pn)
        assert np.array_equal(oracle.c_unpack(pc, N, K, fmt, gs), codes)
        assert np.array_equal(npo.unpack(pc, N, K, fmt, gs), codes)
        for k in [0, K // 3, K - 1]:
            assert oracle.c_code_at(pc[N - 1], fmt, gs, k) == codes[N - 1, k]


# ---- byte-size facts printed on the page -----------------------------------

def test_sizes_printed_on_the_page():
    # §二.1: one uint32 holds 32 1-bit values
    assert oracle.c_row_bytes(F1, 32 * 7 * 64 // 32, 64) == 7 * 64 // 8 * 1
    assert oracle.c_row_bytes(F1, 64, 64) == 8
    assert oracle.c_row_bytes(F2, 64, 64) == 16
    # §二.3: 13 / 26 bytes per 64 / 128 weight group
    assert oracle.c_row_bytes(T5, 64, 64) == 13
    assert oracle.c_row_bytes(T5, 128, 128) == 26
    assert oracle.c_row_bytes(T5, 5120, 128) == 40 * 26
    # §二.3: about 1.585 bit/weight = log2(3) of information; stored 1.625
    assert abs(math.log2(3) - 1.585) < 5e-4
    assert 13 * 8 / 64 == 1.625 and 26 * 8 / 128 == 1.625
    # §二.3: about 23% less RAM than the 2-bit uint32 format (codes + fp16
    # scales for t5, codes + fp16 scales + fp16 biases for 2-bit)
    for gs in (64, 128):
        t5 = oracle.c_row_bytes(T5, gs, gs) + 2
        two = oracle.c_row_bytes(F2, gs, gs) + 2 + 2
        assert 0.20 <= 1 - t5 / two <= 0.26
    assert oracle.c_row_bytes(T5, 65, 64) == -1
    assert oracle.c_row_bytes(F2, 64, 32) == -1


# ---- the product: hand example, brute force, closed forms, identities ------

def test_qmv_hand_worked_example():
    rows = [l.split() for l in read_golden("qmv_tiny.txt")]
    codes = np.zeros((2, 64), dtype=np.uint8)
    codes[:, :4] = [0, 1, 2, 3]
    packed = oracle.c_pack(codes, F2, 64)
    s = np.array([[float(r[1])] for r in rows], dtype=np.float16)
    b = np.array([[float(r[2])] for r in rows], dtype=np.float16)
    x = np.zeros((1, 64), dtype=np.float16)
    x[0, :4] = 1
    y, bound = oracle.c_qmv_rows(x, packed, s, b, F2, 64)
    yn, bn = npo.qmv(x, packed, s, b, F2, 64)
    for r in rows:
        n = int(r[0])
        assert y[0, n] == float(r[3]) and bound[0, n] == float(r[4])
        assert yn[0, n] == float(r[3]) and bn[0, n] == float(r[4])


def _brute_force_y(x, codes, s, b, gs):
    """Pure-Python loops on the codes (no packed bytes involved)."""
    M, K = x.shape
    N = codes.shape[0]
    y = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                g = k // gs
                acc += float(x[m, k]) * (float(s[n, g]) * int(codes[n, k]) + float(b[n, g]))
            y[m, n] = acc
    return y


@pytest.mark.parametrize("fmt", [F1, F2, T5])
@pytest.mark.parametrize("gs", [64, 128])
def test_qmv_brute_force_tiny(fmt, gs):
    for N, K, M in [(1, gs, 1), (2, 2 * gs, 3), (3, gs, 5)]:
        p = synth.problem(fmt, M, N, K, gs, sym=False, key=f"bf{fmt}{gs}{N}{K}{M}")
        packed = oracle.c_pack(p["codes"], fmt, gs)
        b = p["biases"] if p["biases"] is not None else npo.sym_bias(p["scales"], 1.0)
        want = _brute_force_y(p["x"], p["codes"], p["scales"], b, gs)
        yc, bc = oracle.c_qmv_rows(p["x"], packed, p["scales"], b, fmt, gs)
        yn, bn = npo.qmv(p["x"], packed, p["scales"], b, fmt, gs)
        scale = np.abs(want).max() + 1e-300
        assert np.abs(yc - want).max() <= 1e-12 * scale
        assert np.abs(yn - want).max() <= 1e-12 * scale
        assert np.abs(bc - bn).max() <= 1e-12 * (np.abs(bn).max() + 1e-300)
        assert np.all(bc >= np.abs(yc) - 1e-12)


def test_1bit_closed_form_config1():
    """1-bit: y = sum_g (scale_g * sum_{k in g, bit set} x_k + bias_g * sum_{k in g} x_k)."""
    p = synth.problem(F1, 1, 256, 512, 64, key="affine1_m1_256x512_gs64")
    packed = oracle.c_pack(p["codes"], F1, 64)
    x = p["x"].astype(np.float64)
    s, b = p["scales"].astype(np.float64), p["biases"].astype(np.float64)
    want = np.zeros((1, 256))
    for n in range(256):
        for g in range(512 // 64):
            sl = slice(64 * g, 64 * (g + 1))
            set_sum = x[0, sl][p["codes"][n, sl] == 1].sum()
            want[0, n] += s[n, g] * set_sum + b[n, g] * x[0, sl].sum()
    yc, _ = oracle.c_qmv_rows(p["x"], packed, p["scales"], p["biases"], F1, 64)
    yn, _ = npo.qmv(p["x"], packed, p["scales"], p["biases"], F1, 64)
    assert np.abs(yc - want).max() <= 1e-12 * np.abs(want).max()
    assert np.abs(yn - want).max() <= 1e-12 * np.abs(want).max()


@pytest.mark.parametrize("fmt", [F1, F2, T5])
def test_one_hot_x_recovers_each_dequantized_weight(fmt):
    gs, N, K = 64, 4, 128
    p = synth.problem(fmt, 1, N, K, gs, key=f"onehot{fmt}")
    b = p["biases"] if p["biases"] is not None else npo.sym_bias(p["scales"], 1.0)
    packed = oracle.c_pack(p["codes"], fmt, gs)
    for k in range(0, K, 7):
        x = np.zeros((1, K), dtype=np.float16)
        x[0, k] = 1
        y, _ = oracle.c_qmv_rows(x, packed, p["scales"], b, fmt, gs)
        for n in range(N):
            g = k // gs
            assert y[0, n] == float(p["scales"][n, g]) * int(p["codes"][n, k]) + float(b[n, g])


@pytest.mark.parametrize("fmt", [F1, F2, T5])
def test_integer_case_is_a_sum_of_codes(fmt):
    """scale = 1, bias = 0, x = 1: y = sum of codes; for 1-bit a popcount of
    the packed words (Python's own bit counting)."""
    gs, N, K = 64, 5, 512
    rng = np.random.default_rng(7)
    codes = synth.codes(rng, fmt, N, K)
    packed = oracle.c_pack(codes, fmt, gs)
    s = np.ones((N, K // gs), dtype=np.float16)
    b = np.zeros((N, K // gs), dtype=np.float16)
    x = np.ones((1, K), dtype=np.float16)
    y, _ = oracle.c_qmv_rows(x, packed, s, b, fmt, gs)
    yn, _ = npo.qmv(x, packed, s, b, fmt, gs)
    assert np.array_equal(y[0], codes.sum(axis=1).astype(np.float64))
    assert np.array_equal(yn[0], codes.sum(axis=1).astype(np.float64))
    if fmt == F1:
        words = packed.view("<u4")
        pop = [sum(bin(int(w)).count("1") for w in row) for row in words]
        assert np.array_equal(y[0], np.array(pop, dtype=np.float64))


@pytest.mark.parametrize("fmt,ratio", [(F1, 0.5), (F2, 1.5), (T5, 1.0)])
def test_sym_identity_bias_free_equals_stored_bias(fmt, ratio):
    """§二.2 identity I-B: with bias = -scale*ratio stored, the bias-free path
    gives the identical result."""
    p = synth.problem(fmt, 3, 9, 256, 64, sym=True, key=f"sym{fmt}")
    packed = oracle.c_pack(p["codes"], fmt, 64)
    # the stored bias, formed the way a quantiser would: float32 product, fp16
    stored = (np.float32(-ratio) * p["scales"].astype(np.float32)).astype(np.float16)
    assert np.array_equal(oracle.c_sym_bias(p["scales"], ratio).view(np.uint16), stored.view(np.uint16))
    assert oracle.c_sym_mismatches(p["scales"], stored, ratio) == 0
    y0, b0 = oracle.c_qmv_rows(p["x"], packed, p["scales"], None, fmt, 64)
    y1, b1 = oracle.c_qmv_rows(p["x"], packed, p["scales"], stored, fmt, 64)
    assert np.array_equal(y0, y1) and np.array_equal(b0, b1)
    yn, _ = npo.qmv(p["x"], packed, p["scales"], None, fmt, 64)
    assert np.abs(yn - y0).max() <= 1e-12 * np.abs(y0).max()
    # t5 without a bias tensor: w = scale*t - scale, so t = 1 gives w = 0
    if fmt == T5:
        W = npo.dequantize(packed, p["scales"], None, 9, 256, T5, 64)
        assert np.all(W[p["codes"] == 1] == 0)
        assert np.all(W[p["codes"] == 0] < 0) and np.all(W[p["codes"] == 2] > 0)


def test_sym_mismatch_counts_a_changed_bias():
    s = np.full((2, 3), 0.01, dtype=np.float16)
    b = oracle.c_sym_bias(s, 1.5).copy()
    assert oracle.c_sym_mismatches(s, b, 1.5) == 0
    b[1, 2] = np.float16(0.5)
    b[0, 0] = -b[0, 0]
    assert oracle.c_sym_mismatches(s, b, 1.5) == 2


def test_linearity_in_x():
    """y(2 x1 + x2) = 2 y(x1) + y(x2), with integer x so that fp16 is exact."""
    rng = np.random.default_rng(3)
    for fmt in (F1, F2, T5):
        p = synth.problem(fmt, 2, 6, 192, 64, key=f"lin{fmt}")
        b = p["biases"] if p["biases"] is not None else npo.sym_bias(p["scales"], 1.0)
        packed = oracle.c_pack(p["codes"], fmt, 64)
        x1 = rng.integers(-8, 9, size=(2, 192)).astype(np.float16)
        x2 = rng.integers(-8, 9, size=(2, 192)).astype(np.float16)
        y1, _ = oracle.c_qmv_rows(x1, packed, p["scales"], b, fmt, 64)
        y2, _ = oracle.c_qmv_rows(x2, packed, p["scales"], b, fmt, 64)
        y3, _ = oracle.c_qmv_rows((2 * x1 + x2).astype(np.float16), packed, p["scales"], b, fmt, 64)
        assert np.abs(y3 - (2 * y1 + y2)).max() <= 1e-12 * (np.abs(y3).max() + 1)


def test_rows_subset_matches_full():
    p = synth.problem(F2, 5, 40, 320, 64, key="rows")
    packed = oracle.c_pack(p["codes"], F2, 64)
    y, bd = oracle.c_qmv_rows(p["x"], packed, p["scales"], p["biases"], F2, 64)
    rows = np.array([39, 0, 17, 17, 5])
    ys, bs = oracle.c_qmv_rows(p["x"], packed, p["scales"], p["biases"], F2, 64, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(bs, bd[:, rows])


# ---- t5 validation -----------------------------------------------------------

@pytest.mark.parametrize("gs", [64, 128])
def test_t5_invalid_bytes(gs):
    B = oracle.t5_bytes_per_group(gs)
    N, K = 3, 2 * gs
    codes = synth.codes(np.random.default_rng(gs), T5, N, K)
    packed = oracle.c_pack(codes, T5, gs)
    assert oracle.c_t5_invalid_bytes(packed, N, K, gs) == 0
    assert npo.t5_invalid_bytes(packed, N, K, gs) == 0
    bad = packed.copy()
    bad[0, 0] = 243            # out of range
    bad[1, 3] = 255            # out of range
    live = gs - 5 * (B - 1)    # trits used in a group's last byte
    bad[2, B - 1] = 3 ** live  # first padding trit set to 1
    bad[2, 2 * B - 1] = 242    # all trits set: padding non-zero
    assert oracle.c_t5_invalid_bytes(bad, N, K, gs) == 4
    assert npo.t5_invalid_bytes(bad, N, K, gs) == 4
    ok = packed.copy()
    ok[0, B - 1] = 3 ** live - 1  # largest byte with zero padding
    assert oracle.c_t5_invalid_bytes(ok, N, K, gs) == 0


# ---- planted mistakes: a slipped oracle must fail the pins above ------------

def test_planted_mistakes_are_caught():
    """Plant plausible slips in copies of the NumPy oracle's pieces and check
    that the independent pins reject each of them."""
    lines = dict(l.split(":", 1) for l in read_golden("pack_2bit.txt"))
    codes = np.array([[int(v) for v in lines["codes"].split()]], dtype=np.uint8)
    want = _hexbytes(lines["bytes"])

    # (1) MSB-first 2-bit packing
    q = codes.reshape(1, 16, 4)
    msb = (q[..., 3] | (q[..., 2] << 2) | (q[..., 1] << 4) | (q[..., 0] << 6)).astype(np.uint8)
    assert not np.array_equal(msb[0], want)

    # (2) t5 with the first weight most significant
    for line in read_golden("t5_bytes.txt"):
        *t, b = (int(v) for v in line.split())
        rev = sum(v * 3 ** (4 - i) for i, v in enumerate(t))
        if len(set(t)) > 1 and t != t[::-1]:
            assert rev != b

    # (3) dropped bias / wrong sign of bias / transposed group index
    rows = [l.split() for l in read_golden("qmv_tiny.txt")]
    x = np.zeros(64)
    x[:4] = 1
    q0 = np.array([0, 1, 2, 3] + [0] * 60, dtype=np.float64)
    for r in rows:
        s, b, y = float(r[1]), float(r[2]), float(r[3])
        assert (x * (s * q0 + b)).sum() == y
        assert (x * (s * q0)).sum() != y          # dropped bias
        assert (x * (s * q0 - b)).sum() != y      # bias sign flipped
        assert (x * (b * q0 + s)).sum() != y      # scale/bias swapped

    # (4) transposed product (W x instead of x W^T) on a non-square case is
    # rejected by the brute-force comparison's shape check
    p = synth.problem(F2, 3, 2, 128, 64, key="transpose")
    packed = oracle.c_pack(p["codes"], F2, 64)
    y, _ = npo.qmv(p["x"], packed, p["scales"], p["biases"], F2, 64)
    assert y.shape == (3, 2)
