"""Pins of the speculative-decoding verification oracle (CPU), by construction.

Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析" §三 --
spec_decode_verify: compare the draft tokens, count the accepted length,
produce the correction token (greedy reading: argmax of each target row, the
leading run of equal draft tokens, the target's token after it).

Each case plants the answer: logits with a known largest entry per row, and
drafts that agree with the planted tokens for exactly j leading positions."""
import math

import numpy as np
import pytest

import oracle


def planted(rng, B, D, V, js):
    """Rows whose maximum (1.0) sits at a random token T[b, i]; drafts equal
    to T for the first js[b] positions, then one that differs."""
    T = rng.integers(0, V, size=(B, D + 1))
    logits = rng.uniform(-3.0, 0.5, size=(B, D + 1, V))
    logits[np.arange(B)[:, None], np.arange(D + 1)[None, :], T] = 1.0
    draft = rng.integers(0, V, size=(B, D))
    for b, j in enumerate(js):
        draft[b, :j] = T[b, :j]
        if j < D:
            draft[b, j] = (T[b, j] + 1) % V
    return logits, draft, T


@pytest.mark.parametrize("D", [0, 1, 4, 9])
def test_planted_accepted_lengths(D):
    rng = np.random.default_rng(D)
    js = list(range(D + 1))
    logits, draft, T = planted(rng, D + 1, D, 11, js)
    a, nxt, t = oracle.spec_decode_verify(logits, draft)
    assert t.tolist() == T.tolist()
    assert a.tolist() == js
    # the correction (j < D) or bonus (j = D) token is the target's at position j
    assert nxt.tolist() == [int(T[b, j]) for b, j in enumerate(js)]


def test_a_later_match_does_not_extend_the_run():
    logits, draft, T = planted(np.random.default_rng(1), 1, 4, 9, [1])
    draft[0, 2:] = T[0, 2:4]  # positions 2, 3 agree again after the miss at 1
    a, nxt, _ = oracle.spec_decode_verify(logits, draft)
    assert a[0] == 1 and nxt[0] == T[0, 1]


def test_ties_go_to_the_smallest_token():
    row = np.array([0.5, 2.0, -1.0, 2.0, 2.0])
    assert oracle.spec_verify.row_argmax(row) == 1
    logits = np.stack([row, row[::-1]])[None]          # [1, 2, 5]
    a, nxt, t = oracle.spec_decode_verify(logits, [[1]])
    assert t.tolist() == [[1, 0]] and a[0] == 1 and nxt[0] == 0


def test_nan_entries_are_never_chosen():
    nan, inf = math.nan, math.inf
    assert oracle.spec_verify.row_argmax([nan, 1.0, nan, 3.0, nan]) == 3
    assert oracle.spec_verify.row_argmax([nan, nan]) == -1
    assert oracle.spec_verify.row_argmax([-inf, -inf, nan]) == 0
    assert oracle.spec_verify.row_argmax([nan, -inf, 5.0, inf]) == 3
    # a row of NaNs gives -1, which no draft matches (not even a draft of -1)
    logits = np.array([[[nan, nan], [0.0, 1.0]]])
    a, nxt, t = oracle.spec_decode_verify(logits, [[-1]])
    assert t.tolist() == [[-1, 1]] and a[0] == 0 and nxt[0] == -1


def test_fp16_logits_compare_as_stored():
    # 1.0009765625 is the fp16 successor of 1.0: distinct, and the larger wins
    row = np.array([1.0, 1.0009765625, 1.0], dtype=np.float16)
    assert oracle.spec_verify.row_argmax(row) == 1


def test_brute_force_against_sorted_order():
    """Small random cases: the argmax agrees with the first index of a stable
    descending sort, and the accepted run with a direct prefix comparison."""
    rng = np.random.default_rng(5)
    for _ in range(50):
        B, D, V = 3, int(rng.integers(0, 5)), int(rng.integers(1, 6))
        logits = rng.integers(-2, 3, size=(B, D + 1, V)).astype(np.float64)  # many ties
        draft = rng.integers(0, V, size=(B, D))
        a, nxt, t = oracle.spec_decode_verify(logits, draft)
        for b in range(B):
            want = [int(np.argsort(-logits[b, i], kind="stable")[0]) for i in range(D + 1)]
            assert t[b].tolist() == want
            run = 0
            while run < D and draft[b, run] == want[run]:
                run += 1
            assert a[b] == run and nxt[b] == want[run]
