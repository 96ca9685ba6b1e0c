"""The host n-gram drafter (CPU): hand cases, agreement with a brute-force
restatement of the rule on random histories, the ragged batch form, and
argument errors."""
import os

import numpy as np
import pytest


@pytest.fixture(scope="module")
def dr():
    from speculative_decoding_verify_ragged_gb300 import _abi
    if not os.path.exists(_abi.LIB_PATH):
        from speculative_decoding_verify_ragged_gb300 import build
        build.build()
    from speculative_decoding_verify_ragged_gb300 import draft
    return draft


def _brute(h, gamma, min_n, max_n):
    """The rule, spelled out: longest suffix first, most recent earlier occurrence
    that leaves a token after it, copy what followed (<= gamma, <= end)."""
    h = list(h)
    L = len(h)
    for n in range(min(max_n, L - 1), min_n - 1, -1):
        suf = h[L - n:]
        for i in range(L - n - 1, -1, -1):
            if h[i:i + n] == suf:
                return h[i + n:i + n + gamma]
    return []


def test_hand_cases(dr):
    assert dr.ngram_draft([1, 2, 3, 4, 1, 2, 3], 2, 1, 4).tolist() == [4, 1]
    assert dr.ngram_draft([5, 9, 5, 7, 5], 2, 1, 3).tolist() == [7, 5]          # most recent occurrence
    assert dr.ngram_draft([1, 2, 9, 2, 8, 1, 2], 3, 1, 3).tolist() == [9, 2, 8]  # the longer suffix wins
    assert dr.ngram_draft([1, 2, 3, 4], 3, 1, 4).tolist() == []                 # nothing repeats
    assert dr.ngram_draft([7, 7], 5, 1, 4).tolist() == [7]                      # bounded by the end
    assert dr.ngram_draft([3, 1, 3], 4, 2, 4).tolist() == []                    # min_n excludes the 1-gram
    assert dr.ngram_draft([], 4, 1, 2).tolist() == []
    assert dr.ngram_draft([4, 4, 4], 0, 1, 2).tolist() == []


def test_periodic_history_is_continued_exactly(dr):
    period = [11, 12, 13, 14, 15]
    h = period * 4 + period[:2]
    # the most recent earlier occurrence is one period back: the copy runs to the end of the history
    assert dr.ngram_draft(h, 6, 1, 4).tolist() == [13, 14, 15, 11, 12]
    assert dr.ngram_draft(h, 3, 1, 4).tolist() == [13, 14, 15]


def test_agrees_with_brute_force(dr):
    g = np.random.default_rng(0)
    for trial in range(600):
        L = int(g.integers(0, 60))
        V = int(g.integers(2, 6))
        h = g.integers(0, V, size=L).tolist()
        gamma = int(g.integers(0, 8))
        min_n = int(g.integers(1, 4))
        max_n = min_n + int(g.integers(0, 4))
        assert dr.ngram_draft(h, gamma, min_n, max_n).tolist() == _brute(h, gamma, min_n, max_n), (h, gamma)


def test_batch_is_ragged_and_padded(dr):
    g = np.random.default_rng(1)
    hs = [g.integers(0, 4, size=int(n)).tolist() for n in (0, 1, 9, 30, 200)]
    lens, drafts = dr.ngram_draft_batch(hs, 5, 1, 3)
    assert drafts.shape == (5, 5)
    for b, h in enumerate(hs):
        want = _brute(h, 5, 1, 3)
        assert lens[b] == len(want)
        assert drafts[b, :lens[b]].tolist() == want
        assert (drafts[b, lens[b]:] == -1).all()


def test_bad_arguments(dr):
    from speculative_decoding_verify_ragged_gb300 import SdvError
    with pytest.raises(ValueError):
        dr.ngram_draft([1, 2], 2, 0, 3)
    with pytest.raises(ValueError):
        dr.ngram_draft([1, 2], 2, 3, 2)
    with pytest.raises(SdvError):
        dr.ngram_draft_batch([[1, 2]], 2, 2, 1)
