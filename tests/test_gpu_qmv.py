"""GPU parity of the QMV path against the float64 oracle, through the C ABI.

Bar: every output within |y_gpu - y| <= 2e-3 * sum_k |x_k w_k| (fp16 in,
fp32 accumulate, fp16 out).  Small shapes span several tiles and ragged tails
and are checked element by element on every row; the full-size shapes of the
decode sweep are checked on sampled rows, in the same dispatch the benchmark
times.  Both kernels (tensor-core decode and generic) are exercised.
"""
import numpy as np
import pytest

import oracle
from oracle import oracle as npo
import bit_quantized_decode_unpack_gb300 as bqd
from bit_quantized_decode_unpack_gb300 import synth
from _util import assert_within_tolerance, forced_kernel, to_dev

pytestmark = pytest.mark.gpu
F1, F2, T5 = bqd.FMT_AFFINE1, bqd.FMT_AFFINE2, bqd.FMT_T5
KERNELS = [None, "generic"]  # None = the dispatcher's choice; "mma"/"tma" force the tensor-core paths


def run_case(p, kernel=None, rows=None, explicit_ratio=None):
    import torch
    fmt, gs = p["fmt"], p["gs"]
    packed = oracle.c_pack(p["codes"], fmt, gs)
    w = bqd.pack(to_dev(p["codes"]), fmt, gs)
    x, s, b = to_dev(p["x"]), to_dev(p["scales"]), to_dev(p["biases"])
    with forced_kernel(kernel):
        if explicit_ratio is None:
            y = bqd.qmv(x, w, s, b, fmt, gs)
        else:
            y = bqd.qmv_sym(x, w, s, explicit_ratio, fmt, gs)
    torch.cuda.synchronize()
    yr, bound = oracle.c_qmv_rows(p["x"], packed, p["scales"], p["biases"], fmt, gs, rows=rows,
                                  ratio=explicit_ratio)
    yg = y.cpu().numpy().astype(np.float64)
    if rows is not None:
        yg = yg[:, rows]
    return assert_within_tolerance(yg, yr, bound, what=p["key"])


SMALL = [(1, 1, 1), (2, 17, 2), (3, 130, 5), (4, 64, 3), (5, 1000, 20), (8, 259, 32), (11, 64, 10),
         (16, 33, 6)]  # (M, N, K in groups)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("fmt", [F1, F2, T5])
@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("sym", [False, True])
def test_small_shapes_all_rows(kernel, fmt, gs, sym):
    for M, N, G in SMALL:
        p = synth.problem(fmt, M, N, G * gs, gs, sym=sym)
        if fmt == T5 and not sym:
            # t5 with an explicit bias tensor: the general affine case
            p["biases"] = synth.biases(np.random.default_rng(M), F2, p["scales"])
        run_case(p, kernel)


# shapes inside the tensor-core paths' envelope (t5: K a multiple of 1024),
# spanning several row tiles, K-slices and ragged row tails
MMA_SHAPES = [(1, 17, 1024), (2, 300, 2048), (3, 130, 3072), (5, 1000, 1024), (8, 259, 2048), (11, 40, 1024),
              (4, 16, 5120), (6, 1, 1024)]


@pytest.mark.parametrize("kernel,fmt", [("mma", F1), ("mma", F2), ("mma", T5), ("tma", F1), ("tma", F2), ("tma", T5)])
@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("sym", [False, True])
def test_tensor_core_paths_forced(kernel, fmt, gs, sym):
    """A forced kernel family makes an unsupported request an error instead
    of a fallback, so these cases are known to run on the named kernel."""
    for M, N, K in MMA_SHAPES:
        p = synth.problem(fmt, M, N, K, gs, sym=sym)
        if fmt == T5 and not sym:
            p["biases"] = synth.biases(np.random.default_rng(N), F2, p["scales"])
        run_case(p, kernel)


# TMA-ring kernel: its envelope is K a multiple of 256 (with K/gs a multiple of
# 8 the scale rows are 16-byte multiples and come by TMA); shapes span row blocks of 128 (N <= 2048) and 256
# (larger N) with ragged tails, both sides of N = 2048, split-K clusters of
# many sizes (portable and not; 300 x 17408 would take 14 ranks, which leave
# one of them no rows of a 128-row block, so the planner skips that split), M
# up to 8 in one pass and passes of 8 rows (grid rows of one launch) beyond
# (every M from 9 to 16, and 27 and 33), the last one ragged
TMA_SHAPES = [(1, 2048, 2048), (3, 2100, 1024), (1, 1, 1024), (2, 127, 1024), (3, 256, 2048), (4, 257, 3072), (5, 383, 4096), (7, 1024, 5120),
              (8, 2000, 1024), (9, 200, 2048), (16, 130, 1024), (1, 5120, 17408), (5, 300, 17408), (2, 4096, 6144),
              (27, 300, 2048), (6, 70, 1024), (10, 513, 2048), (11, 64, 5120), (12, 300, 3072), (13, 257, 1024),
              (14, 1000, 2048), (15, 33, 4096), (33, 129, 1024)]


@pytest.mark.parametrize("fmt", [F1, F2])
@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("sym", [False, True])
def test_tma_kernel_shapes(fmt, gs, sym):
    shapes = TMA_SHAPES + ([(3, 257, 512), (1, 40, 512)] if gs == 64 else [])
    for M, N, K in shapes:
        p = synth.problem(fmt, M, N, K, gs, sym=sym)
        run_case(p, "tma")


# t5 TMA-ring kernel: K a multiple of 1024; ragged 128-row blocks (narrow
# layers) and 256-row blocks (4353 x 5120, 4100 x 17408, 5120 x 17408), split-K
# clusters, the column split (M <= 2) and the scaled path (M >= 3), passes of
# at most 8 x rows (grid rows of one launch; M = 12, 16, 23 take several, the
# last one ragged); K = 28672 (28 chunks) is where 14 ranks would leave one
# of them no rows of a 128-row block: the planner skips that split
T5R_SHAPES = [(1, 300, 28672), (4, 200, 28672), (1, 1, 1024), (2, 127, 1024), (2, 255, 1024), (3, 129, 2048), (3, 257, 2048), (4, 300, 3072),
              (4, 513, 1024), (5, 1000, 5120), (6, 383, 4096), (6, 511, 3072), (7, 260, 2048), (12, 64, 1024),
              (16, 130, 2048), (1, 5120, 17408), (5, 200, 17408), (23, 129, 2048), (1, 4353, 5120),
              (2, 4100, 17408), (3, 4353, 5120), (8, 4100, 17408)]


@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("sym", [False, True])
def test_t5_tma_kernel_shapes(gs, sym):
    for M, N, K in T5R_SHAPES:
        p = synth.problem(T5, M, N, K, gs, sym=sym)
        if not sym:
            p["biases"] = synth.biases(np.random.default_rng(N + M), F2, p["scales"])
        run_case(p, "tma")


# K a multiple of 256 whose scale rows (K/gs fp16) are no multiple of 16 bytes:
# the scale and bias boxes come by 4-byte copies instead of TMA.  K = 2304 at
# gs = 128 gives 36-byte rows (4-byte aligned only); split-K clusters, passes of
# 8 rows, 128- and 256-row blocks and ragged tails as above
TMA_COPY_SHAPES = {64: [(1, 300, 768), (5, 1000, 1280), (3, 2100, 2304), (8, 129, 4864), (12, 257, 3840),
                        (2, 4100, 2816), (1, 40, 768)],
                   128: [(1, 300, 1280), (5, 1000, 2304), (3, 2100, 2560), (8, 129, 1536), (12, 257, 3584),
                         (2, 4100, 2304), (1, 5120, 13824), (4, 64, 256)]}


@pytest.mark.parametrize("fmt", [F1, F2])
@pytest.mark.parametrize("gs", [64, 128])
@pytest.mark.parametrize("sym", [False, True])
def test_tma_kernel_scale_rows_by_copies(fmt, gs, sym):
    for M, N, K in TMA_COPY_SHAPES[gs]:
        assert (K // gs) % 8 != 0 and K % 256 == 0
        run_case(synth.problem(fmt, M, N, K, gs, sym=sym), "tma")


@pytest.mark.parametrize("fmt", [F1, F2])
@pytest.mark.parametrize("sym", [False, True])
def test_tma_kernel_scales_at_4_byte_offsets(fmt, sym):
    """Scale (and bias) tensors whose storage starts 4 bytes past a 16-byte
    boundary: the boxes come by copies although their rows are 16-byte
    multiples."""
    import torch
    gs = 64
    for M, N, K in [(3, 300, 2048), (5, 4100, 5120), (1, 129, 17408)]:
        p = synth.problem(fmt, M, N, K, gs, sym=sym)
        packed = oracle.c_pack(p["codes"], fmt, gs)
        w = bqd.pack(to_dev(p["codes"]), fmt, gs)

        def offset_copy(a):
            if a is None:
                return None
            buf = torch.empty(a.size + 2, dtype=torch.float16, device="cuda")
            t = buf[2:].view(a.shape)
            t.copy_(torch.from_numpy(a))
            assert t.data_ptr() % 16 == 4 and t.is_contiguous()
            return t

        with forced_kernel("tma"):
            y = bqd.qmv(to_dev(p["x"]), w, offset_copy(p["scales"]), offset_copy(p["biases"]), fmt, gs)
        torch.cuda.synchronize()
        yr, bound = oracle.c_qmv_rows(p["x"], packed, p["scales"], p["biases"], fmt, gs)
        assert_within_tolerance(y.cpu().numpy().astype(np.float64), yr, bound, what=p["key"])


@pytest.mark.parametrize("fmt", [F1, F2])
def test_tma_envelope_and_fallback(fmt):
    """Outside the TMA kernel's envelope (here K = 640, no whole number of
    256-code chunks) a forced call reports "unsupported" and the default
    dispatch still gives parity."""
    p = synth.problem(fmt, 3, 100, 640, 64)
    with pytest.raises(bqd.BqdError) as ei:
        run_case(p, "tma")
    assert ei.value.status == 2  # BQD_ERR_UNSUPPORTED
    run_case(p, None)


@pytest.mark.parametrize("kernel", ["tma", "mma", "generic"])
@pytest.mark.parametrize("fmt", [F1, F2, T5])
def test_zero_codes_zero_bias_give_exact_zeros(kernel, fmt):
    """w = s*0 + 0 everywhere: y is exactly 0 whatever x and s are (the ring
    kernels' offset cancellation is exact for code-free groups: the offset
    sums come from the same MMA sequence as the weights' products)."""
    import torch
    M, N, K, gs = 5, 300, 2048, 64
    p = synth.problem(fmt, M, N, K, gs)
    codes = np.zeros_like(p["codes"])
    w = bqd.pack(to_dev(codes), fmt, gs)
    b = torch.zeros((N, K // gs), dtype=torch.float16, device="cuda")
    with forced_kernel(kernel):
        y = bqd.qmv(to_dev(p["x"]), w, to_dev(p["scales"]), b, fmt, gs)
    torch.cuda.synchronize()
    assert torch.all(y == 0)


@pytest.mark.parametrize("stages", ["1", "2"])
@pytest.mark.parametrize("gs", [64, 128])
def test_t5_stage_ring_depths(stages, gs):
    """The t5 kernel's weight ring with one and with two stages per warp."""
    bqd.set_option(bqd.OPT_T5_STAGES, int(stages))
    try:
        for M, N, K in [(1, 300, 3072), (5, 1000, 2048), (8, 40, 5120)]:
            run_case(synth.problem(T5, M, N, K, gs, sym=True), "mma")
    finally:
        bqd.set_option(bqd.OPT_T5_STAGES, 0)


@pytest.mark.parametrize("kernel", KERNELS)
def test_config1_all_rows(kernel):
    """1-bit, M=1, N=256, K=512, gs=64, seed 0."""
    p = synth.problem(F1, 1, 256, 512, 64, key="affine1_m1_256x512_gs64")
    run_case(p, kernel)


def _sample_rows(N, n=48, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, 1, 15, 16, N - 1], rng.integers(0, N, n)]))


FULL = []
for (N, K) in [(5120, 5120), (1024, 5120), (17408, 5120), (5120, 17408)]:
    for gs in (64, 128):
        for M in (1, 5):
            FULL.append((F2, M, N, K, gs, False))
    FULL.append((F2, 3, N, K, 64, True))
for (N, K) in [(17408, 5120), (5120, 17408)]:
    for gs in (64, 128):
        for M in (1, 3, 5):
            FULL.append((T5, M, N, K, gs, True))
for (N, K) in [(6144, 5120), (5120, 6144), (17408, 5120)]:
    FULL.append((F1, 1, N, K, 64, False))
    FULL.append((F1, 5, N, K, 128, False))


@pytest.mark.slow
@pytest.mark.parametrize("fmt,M,N,K,gs,sym", FULL)
def test_full_size_sampled_rows(fmt, M, N, K, gs, sym):
    p = synth.problem(fmt, M, N, K, gs, sym=sym)
    run_case(p, None, rows=_sample_rows(N, seed=N + K + M))


@pytest.mark.parametrize("kernel", KERNELS + ["mma"])
@pytest.mark.parametrize("fmt,ratio", [(F1, 0.5), (F2, 1.5), (T5, 1.0)])
def test_sym_identity_on_gpu_is_bit_identical(kernel, fmt, ratio):
    """§二.2 identity I-B: the bias-free path equals the path reading the
    stored bias fp16(-ratio*scale), bit for bit."""
    import torch
    p = synth.problem(fmt, 5, 777, 2048, 64, sym=True)
    stored = npo.sym_bias(p["scales"], ratio)
    w = bqd.pack(to_dev(p["codes"]), fmt, 64)
    x, s = to_dev(p["x"]), to_dev(p["scales"])
    with forced_kernel(kernel):
        y0 = bqd.qmv(x, w, s, None, fmt, 64)
        y1 = bqd.qmv(x, w, s, to_dev(stored), fmt, 64)
        y2 = bqd.qmv_sym(x, w, s, ratio, fmt, 64)
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))
    assert torch.equal(y0.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("kernel", KERNELS)
def test_explicit_ratio(kernel):
    p = synth.problem(F2, 4, 300, 1024, 128, sym=True)
    run_case(p, kernel, explicit_ratio=0.7)


@pytest.mark.parametrize("kernel", KERNELS + ["mma"])
def test_kernels_agree_and_are_deterministic(kernel):
    import torch
    p = synth.problem(F2, 5, 2048, 5120, 64)
    w = bqd.pack(to_dev(p["codes"]), F2, 64)
    x, s, b = to_dev(p["x"]), to_dev(p["scales"]), to_dev(p["biases"])
    with forced_kernel(kernel):
        y0 = bqd.qmv(x, w, s, b, F2, 64)
        y1 = bqd.qmv(x, w, s, b, F2, 64)
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int16), y1.view(torch.int16))


def test_empty_and_degenerate_inputs():
    import torch
    dev = "cuda"
    poison = torch.full((4, 8), 7.0, dtype=torch.float16, device=dev)
    x = torch.zeros((4, 64), dtype=torch.float16, device=dev)
    s = torch.ones((8, 1), dtype=torch.float16, device=dev)
    w = torch.zeros((8, 16), dtype=torch.uint8, device=dev)
    # M = 0 / N = 0: valid no-ops
    bqd.qmv(x[:0], w, s, None, F2, 64, out=poison[:0])
    lib = bqd.load()
    assert lib.bqd_qmv(None, None, None, None, 4, 0, 64, F2, 64, None, None) == 0
    torch.cuda.synchronize()
    assert torch.all(poison == 7.0)
    # K = 0: zeros
    out = torch.full((4, 8), 7.0, dtype=torch.float16, device=dev)
    assert lib.bqd_qmv(None, None, None, None, 4, 8, 0, F2, 64,
                       __import__("ctypes").c_void_p(out.data_ptr()), None) == 0
    torch.cuda.synchronize()
    assert torch.all(out == 0)
    # x = 0: exact zeros for every format (bias times a zero sum)
    for fmt in (F1, F2, T5):
        p = synth.problem(fmt, 3, 70, 640, 64)
        wd = bqd.pack(to_dev(p["codes"]), fmt, 64)
        for kernel in KERNELS:
            with forced_kernel(kernel):
                y = bqd.qmv(torch.zeros((3, 640), dtype=torch.float16, device=dev), wd,
                            to_dev(p["scales"]), to_dev(p["biases"]), fmt, 64)
            torch.cuda.synchronize()
            assert torch.all(y == 0)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("fmt", [F1, F2, T5])
def test_one_hot_x_recovers_dequantized_weights(kernel, fmt):
    import torch
    gs, N, K = 64, 96, 256
    p = synth.problem(fmt, 8, N, K, gs)
    ks = [0, 1, 63, 64, 130, 255, 200, 17]
    x = np.zeros((8, K), dtype=np.float16)
    for m, k in enumerate(ks):
        x[m, k] = 1
    p["x"] = x
    run_case(p, kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_output_guard_band_untouched(kernel):
    import torch
    p = synth.problem(F2, 5, 1000, 1280, 64)
    w = bqd.pack(to_dev(p["codes"]), F2, 64)
    M, N = 5, 1000
    buf = torch.full((M * N + 2048,), 1234.0, dtype=torch.float16, device="cuda")
    out = buf[:M * N].view(M, N)
    with forced_kernel(kernel):
        bqd.qmv(to_dev(p["x"]), w, to_dev(p["scales"]), to_dev(p["biases"]), F2, 64, out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[M * N:] == 1234.0)


@pytest.mark.parametrize("fmt", [F1, F2, T5])
def test_large_scales_take_the_exact_unpack(fmt):
    """Scales far above the fast unpack's range (|s| up to ~600) must still be
    exact on the tensor-core paths (they switch to the exact unpack)."""
    rng = np.random.default_rng(4)
    p = synth.problem(fmt, 2, 96, 2048, 64, sym=True)
    p["scales"] = (np.abs(rng.normal(0, 200, size=p["scales"].shape)) + 1).astype(np.float16)
    p["x"] = (p["x"].astype(np.float32) * 1e-3).astype(np.float16)
    run_case(p, "mma")
    run_case(p, None)
    run_case(p, "tma")


def test_large_magnitudes_stay_within_tolerance():
    """Scales near 8, x up to +-60: fp16 output stays finite and within bound."""
    rng = np.random.default_rng(9)
    p = synth.problem(F2, 3, 200, 640, 64)
    p["scales"] = (np.abs(rng.normal(0, 2, size=p["scales"].shape)) + 6).astype(np.float16)
    p["biases"] = (-p["scales"].astype(np.float32) * 1.5).astype(np.float16)
    p["x"] = (rng.normal(0, 20, size=p["x"].shape)).clip(-60, 60).astype(np.float16) * np.float16(0.01)
    for kernel in KERNELS:
        run_case(p, kernel)


def test_non_default_stream():
    import torch
    p = synth.problem(T5, 5, 500, 1280, 128, sym=True)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        w = bqd.pack(to_dev(p["codes"]), T5, 128)
        y = bqd.qmv(to_dev(p["x"]), w, to_dev(p["scales"]), None, T5, 128)
    st.synchronize()
    packed = oracle.c_pack(p["codes"], T5, 128)
    yr, bound = oracle.c_qmv_rows(p["x"], packed, p["scales"], None, T5, 128)
    assert_within_tolerance(y.cpu().numpy(), yr, bound)


MID_M = [(F2, M, N, K, gs) for M in (9, 12, 16) for (N, K) in [(17408, 5120), (5120, 17408)] for gs in (64, 128)]
MID_M += [(F1, M, 17408, 5120, 64) for M in (10, 16)]


@pytest.mark.slow
@pytest.mark.parametrize("fmt,M,N,K,gs", MID_M)
def test_mid_m_one_pass_full_size_sampled_rows(fmt, M, N, K, gs):
    """9 <= M <= 16 (two passes of x rows in one launch of the decode kernel)
    at the layer sizes, on sampled rows (the dispatcher's choice there)."""
    p = synth.problem(fmt, M, N, K, gs)
    run_case(p, None, rows=_sample_rows(N, seed=N + M))
