"""Pins of the budget-preset and re-eviction oracles:

- StreamingLLM's kept set is the top-k of the order "sinks first, then the most recent"
  (topk_positions over a score that encodes that order), and has the closed form
  {0..s-1} U {C-(k-s)..C-1};
- re-evicting a cache that has no appended rows keeps the top-k of the held candidates,
  which by nestedness is topk_positions over all candidates when the held rows came from a
  larger top-k; appended rows (-1) and window rows always stay.
"""
import numpy as np
import pytest

import oracle as O


@pytest.mark.parametrize("C,k,s", [(50, 0, 4), (50, 3, 4), (50, 4, 4), (50, 20, 4), (50, 50, 4),
                                   (10, 7, 0)])
def test_streaming_is_topk_of_sinks_then_recency(C, k, s):
    score = np.arange(C, dtype=np.float64) + 1.0
    score[:s] = 1e9                                   # sinks first
    np.testing.assert_array_equal(O.streaming_positions(C, k, s), O.topk_positions(score, k))
    got = O.streaming_positions(C, k, s)
    assert len(got) == k and np.all(np.diff(got) > 0)


def test_reevict_nested_and_forced_rows_stay():
    rng = np.random.default_rng(2)
    C, w = 60, 4
    s = rng.random(C)
    for big in (10, 30, 60):
        kept = O.topk_positions(s, big)
        held = list(kept) + list(range(C, C + w)) + [-1, -1, -1]      # window, then 3 appends
        for small in range(0, big + 1, 7):
            rows = O.reevict_rows(held, s, small + w + 3)
            pos = np.asarray(held)[rows]
            np.testing.assert_array_equal(pos[:small], O.topk_positions(s, small))
            np.testing.assert_array_equal(pos[small:], list(range(C, C + w)) + [-1, -1, -1])
