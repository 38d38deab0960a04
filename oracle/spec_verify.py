"""Oracle of the speculative-decoding verification step (test infrastructure
only, like the rest of ``oracle/``).

Page: "oMLX Bonsai 自定义内核:Qwen 系列快速 QMV 路径完整解析", §三 --
spec_decode_verify fuses three steps: compare the draft tokens, count the
accepted length, produce the correction token.  The page states no formula;
the greedy reading, step by step in the page's order:

1. compare: the target's token at position i is the argmax of its logits
   row i (i = 0 .. D); ties go to the smallest token id, NaN entries are
   never chosen, a row without a comparable value gives -1;
2. count: the accepted length is the number of leading draft tokens equal to
   the target's tokens (a -1 from a row of NaNs matches no draft token);
3. correct: the next token is the target's token at that position (the
   correction where the draft was rejected, the bonus token when all D drafts
   were accepted).

Plain loops over sequences and rows; within a row, NumPy's max of the
non-NaN values and the first index holding it, comparing the logits as they
are stored (fp16 values widened exactly to float64).
"""
from __future__ import annotations

import numpy as np


def row_argmax(row) -> int:
    """Index of the largest non-NaN value; the smallest such index on ties;
    -1 if every value is NaN."""
    r = np.asarray(row, dtype=np.float64)
    comparable = ~np.isnan(r)
    if not comparable.any():
        return -1
    largest = r[comparable].max()
    return int(np.flatnonzero(r == largest)[0])


def spec_decode_verify(logits, draft):
    """logits [B, D+1, V], draft int [B, D] -> (accepted [B], next_token [B],
    target tokens [B, D+1]), all int64."""
    logits = np.asarray(logits)
    B, D1, _ = logits.shape
    draft = np.asarray(draft).reshape(B, D1 - 1)
    t = np.array([[row_argmax(logits[b, i]) for i in range(D1)] for b in range(B)], dtype=np.int64).reshape(B, D1)
    accepted = np.zeros(B, dtype=np.int64)
    nxt = np.zeros(B, dtype=np.int64)
    for b in range(B):
        a = 0
        while a < D1 - 1 and t[b, a] >= 0 and int(draft[b, a]) == int(t[b, a]):
            a += 1
        accepted[b] = a
        nxt[b] = t[b, a]
    return accepted, nxt, t
