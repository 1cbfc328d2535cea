"""Adaptive draft length: a plain CPU restatement (test infrastructure).

TEST INFRASTRUCTURE.  Only `tests/` may import this module; the product path
(the CUDA library and its binding) never does.

Follows sxl-space.tk "【大模型】- 推测解码", 自适应推测解码
(AdaptiveSpeculativeDecoder: __init__ and adapt_k), one controller per
sequence of a batch:

  * current_k starts at (min_k + max_k) // 2;
  * each round appends acceptance_rate = accepted / current_k to a history
    that keeps its last history_size = 100 entries;
  * once the history holds at least 10 rates, the mean of the last 10
    decides: above 0.8 current_k = min(current_k + 1, max_k); below 0.5
    current_k = max(current_k - 1, min_k).

Readings (the pages are silent): rates are exact fractions, so a mean of
exactly 0.8 or 0.5 changes nothing (the pages' Python floats round such
ties); a round without a rate (accepted < 0, current_k = 0 or
accepted > current_k) leaves the controller as it was.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

HISTORY_SIZE = 100
WINDOW = 10
HIGH = Fraction(4, 5)
LOW = Fraction(1, 2)


class AdaptiveK:
    """One sequence's controller, in the pages' order of steps."""

    def __init__(self, min_k: int = 1, max_k: int = 10):
        self.min_k = min_k
        self.max_k = max_k
        self.current_k = (min_k + max_k) // 2
        self.acceptance_history: list[Fraction] = []

    def adapt(self, accepted: int) -> int:
        """Record one round (accepted drafted tokens at the current length)
        and return the length for the next round."""
        k = self.current_k
        if accepted < 0 or k <= 0 or accepted > k:
            return self.current_k
        self.acceptance_history.append(Fraction(accepted, k))
        if len(self.acceptance_history) > HISTORY_SIZE:
            self.acceptance_history.pop(0)
        if len(self.acceptance_history) >= WINDOW:
            avg = sum(self.acceptance_history[-WINDOW:]) / WINDOW
            if avg > HIGH:
                self.current_k = min(self.current_k + 1, self.max_k)
            elif avg < LOW:
                self.current_k = max(self.current_k - 1, self.min_k)
        return self.current_k


def offsets(ks) -> np.ndarray:
    """k_offsets of a batch from its per-sequence lengths."""
    return np.concatenate([[0], np.cumsum(np.asarray(ks, dtype=np.int64))]).astype(np.int32)


def run_batch(num_accepted_rounds, B: int, min_k: int = 1, max_k: int = 10):
    """k_offsets after init and after each round of accept counts
    (a list of [B] arrays); returns the list of k_offsets arrays."""
    ctl = [AdaptiveK(min_k, max_k) for _ in range(B)]
    out = [offsets([c.current_k for c in ctl])]
    for counts in num_accepted_rounds:
        out.append(offsets([c.adapt(int(n)) for c, n in zip(ctl, counts)]))
    return out
