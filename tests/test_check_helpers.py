"""The parity helpers themselves, on the CPU: they accept the oracle's own result and reject a
planted wrong one, so a GPU test that passes through them has been checked for something."""
import numpy as np
import pytest

import oracle as O
from tests.kvpath import assert_decode_close, oracle_crit_kept_check, oracle_kept_check


def _head(seed, C=400):
    rng = np.random.default_rng(seed)
    s = rng.random(C) ** 3
    c = rng.random(C) + 0.1
    return s, c


def test_crit_check_accepts_the_oracle_selection():
    s, c = _head(1)
    for k in (0, 1, 37, 200, 400):
        kept = O.critical_positions(s, c, k, 1, 2, 1e-6)
        assert oracle_crit_kept_check(s, c, s.astype(np.float32), kept, k, 1, 2, 1e-6) == 0


def test_crit_check_rejects_a_swapped_stage2_row():
    s, c = _head(2)
    k = 100
    kept = O.critical_positions(s, c, k, 1, 2, 1e-6)
    kappa = (s + 1e-6) * c
    out = np.setdiff1d(np.arange(len(s)), kept)
    # drop the kept row of largest kappa that stage 1 did not take, add the worst row left
    st1 = O.topk_positions(s, k // 2)
    st2 = np.setdiff1d(kept, st1)
    best = st2[np.argmax(kappa[st2])]
    worst = out[np.argmin(kappa[out])]
    bad = np.sort(np.concatenate([np.setdiff1d(kept, [best]), [worst]]))
    with pytest.raises(AssertionError):
        oracle_crit_kept_check(s, c, s.astype(np.float32), bad, k, 1, 2, 1e-6)


def test_crit_check_rejects_a_swapped_stage1_row():
    s, c = _head(3)
    k = 100
    kept = O.critical_positions(s, c, k, 1, 2, 1e-6)
    top = int(np.argmax(s))
    assert top in kept
    out = np.setdiff1d(np.arange(len(s)), kept)
    bad = np.sort(np.concatenate([np.setdiff1d(kept, [top]), [out[0]]]))
    with pytest.raises(AssertionError):
        oracle_crit_kept_check(s, c, s.astype(np.float32), bad, k, 1, 2, 1e-6)


def test_topk_check_allows_only_near_ties():
    s = np.array([0.5, 0.4, 0.3, 0.3 * (1 + 1e-7), 0.1])
    assert oracle_kept_check(s, np.array([0, 1, 2]), 3) == 2      # 2 and 3 tie within 1e-5
    with pytest.raises(AssertionError):
        oracle_kept_check(s, np.array([0, 1, 4]), 3)


def test_decode_bar():
    ref = np.array([0.5, -3.9, 5.0, 100.0])
    got = ref + np.array([0.0099, -0.0099, 0.0099 + 2.0 ** -8 * 5.0, 0.3])
    assert assert_decode_close(got, ref, "bf16") == pytest.approx(0.3)
    with pytest.raises(AssertionError):
        assert_decode_close(ref + np.array([0.0, 0.0101, 0.0, 0.0]), ref, "bf16")
    with pytest.raises(AssertionError):
        assert_decode_close(ref + np.array([0.0, 0.0, 0.0, 0.5]), ref, "bf16")
    with pytest.raises(AssertionError):
        assert_decode_close(ref + 2e-4, ref, "f32")
