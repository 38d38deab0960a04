"""GPU parity of the speculative-decoding verification kernel against the
oracle, through the C ABI: accepted lengths, next tokens and every row's
argmax must be identical (integer results).

Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" §三 --
spec_decode_verify (compare drafts, count the accepted length, produce the
correction token), greedy reading."""

import numpy as np
import pytest

import oracle
import bit_quantized_decode_unpack_gb300 as bqd

pytestmark = pytest.mark.gpu


def make_case(seed, B, D, V, dtype, plant=True):
    """Gaussian logits; drafts that follow the target's tokens for a spread of
    leading lengths (the target tokens come from the oracle's argmax)."""
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((B, D + 1, V)).astype(dtype)
    draft = rng.integers(0, V, size=(B, D)).astype(np.int32)
    if plant and D > 0:
        t = np.array([[oracle.spec_verify.row_argmax(logits[b, i]) for i in range(D)] for b in range(B)])
        for b in range(B):
            j = b % (D + 1)
            draft[b, :j] = t[b, :j]
            if j < D:
                draft[b, j] = (t[b, j] + 1) % V if V > 1 else -5
    return logits, draft


def run(logits, draft, offset=0):
    import torch
    B, D1, V = logits.shape
    flat = torch.from_numpy(logits.reshape(-1))
    if offset:  # start the tensor off a 16-byte boundary
        buf = torch.empty(flat.numel() + offset, dtype=flat.dtype, device="cuda")
        buf[offset:].copy_(flat.cuda())
        lg = buf[offset:].view(B, D1, V)
    else:
        lg = flat.cuda().view(B, D1, V)
    dr = torch.from_numpy(draft).cuda()
    amax = torch.full((B, D1), -7, dtype=torch.int32, device="cuda")
    a, n = bqd.spec_decode_verify(lg, dr, argmax_out=amax)
    torch.cuda.synchronize()
    wa, wn, wt = oracle.spec_decode_verify(logits, draft)
    assert np.array_equal(amax.cpu().numpy(), wt), "argmax rows"
    assert np.array_equal(a.cpu().numpy(), wa), "accepted lengths"
    assert np.array_equal(n.cpu().numpy(), wn), "next tokens"
    return wa


# (B, D, V): single values, ragged V (rows off 16-byte boundaries), D+1 beyond
# the 16-CTA cluster (rows shared round-robin), many sequences
SHAPES = [(1, 0, 1), (3, 1, 7), (5, 4, 1000), (8, 8, 4099), (2, 20, 513), (40, 3, 32000), (17, 15, 257)]


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
@pytest.mark.parametrize("B,D,V", SHAPES)
def test_random_logits(dtype, B, D, V):
    logits, draft = make_case(B * 100 + D + V, B, D, V, dtype)
    acc = run(logits, draft)
    if B > D:
        assert set(acc.tolist()) == set(range(D + 1))  # every accepted length occurs


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_unaligned_base(dtype):
    logits, draft = make_case(3, 6, 5, 3001, dtype)
    run(logits, draft, offset=3)


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_ties_nan_and_infinities(dtype):
    B, D, V = 6, 3, 600
    logits, draft = make_case(11, B, D, V, dtype, plant=False)
    logits[0, 0, [17, 300, 599]] = 50.0            # a three-way tie: 17 wins
    logits[1, :, :] = np.nan                       # rows of NaN: -1, never matched
    draft[1, 0] = -1
    logits[2, 1, :] = -np.inf                      # all -inf: token 0
    logits[2, 1, 5] = np.nan
    logits[3, 2, ::2] = np.nan                     # NaNs among values
    logits[3, 2, 401] = 40.0
    logits[4, 0, 599] = np.inf                     # +inf at the last token
    draft[4, 0] = 599
    logits[5, 1, 0] = 60.0                         # the first token
    logits[5, 0, 7] = 60.0
    draft[5, :2] = [7, 0]
    acc = run(logits, draft)
    assert acc[4] >= 1 and acc[5] >= 2


def test_full_size_fp16():
    """64 sequences, 8 draft tokens, a 151,936-token vocabulary (the size the
    benchmark times)."""
    logits, draft = make_case(99, 64, 8, 151936, np.float16)
    run(logits, draft)


def test_argument_errors():
    import torch
    lg = torch.zeros((2, 3, 10), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(TypeError):
        bqd.spec_decode_verify(lg, torch.zeros((2, 2), dtype=torch.int32, device="cuda"))
    lg = torch.zeros((2, 3, 10), dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        bqd.spec_decode_verify(lg, torch.zeros((2, 3), dtype=torch.int32, device="cuda"))
    # B = 0 launches nothing
    a, n = bqd.spec_decode_verify(torch.zeros((0, 3, 10), dtype=torch.float16, device="cuda"),
                                  torch.zeros((0, 2), dtype=torch.int32, device="cuda"))
    assert a.numel() == 0 and n.numel() == 0


@pytest.mark.parametrize("dtype", [np.float16, np.float32])
def test_rows_split_over_the_cluster(dtype):
    """Few rows: each row's vocabulary is split into parts reduced by different
    CTAs (here 2 rows x 4 parts of ~5000, boundaries off 16-byte alignment).
    Ties across parts go to the smaller token; NaN-only parts are ignored."""
    B, D, V = 4, 1, 20003
    logits, draft = make_case(21, B, D, V, dtype, plant=False)
    logits[0, 0, [100, 12000, 20002]] = 30.0        # tie across parts 0, 2, 3: token 100
    logits[1, 0, :5000] = np.nan                   # part 0 all NaN; maximum in part 3
    logits[1, 0, 19000] = 30.0
    draft[1, 0] = 19000
    logits[2, :, :] = np.nan                       # every part NaN: -1
    logits[3, 1, 10001] = 30.0                     # maximum at a part's first value
    acc = run(logits, draft)
    assert acc[1] == 1


def test_small_batch_full_vocabulary():
    """One sequence, 4 draft tokens, a 151,936-token vocabulary: the five rows
    are split over the cluster's 15 CTAs."""
    logits, draft = make_case(5, 1, 4, 151936, np.float16)
    run(logits, draft)
