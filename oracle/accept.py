"""Greedy acceptance of a drafted block (oracle).  TEST INFRASTRUCTURE: see
oracle/common.py for who may use this package.

Source: flashmap_drafter.js (diskformer 0.6.6), ``specGenerate``, the verify
step: the target's argmax rows for [anchor, drafts...] are compared with the
drafts; the accepted count is the longest prefix on which they agree (capped by
the verify length K), and the next token is the target's own token at the
first disagreement (or at K).  The MTP runner on ternary_bonsai_2_mtp.js
(``MTPRunner.generate``) uses the same rule.
"""
from __future__ import annotations

from typing import Sequence, Tuple


def accept(draft: Sequence[int], target: Sequence[int], k: int) -> Tuple[int, int]:
    """Return (n_accepted, bonus).  draft has >= k entries, target k + 1."""
    acc = 0
    while acc < k and int(draft[acc]) == int(target[acc]):
        acc += 1
    return acc, int(target[acc])
