"""Pins of the oracle's reuse-interval choice (EvoCG §3.4, interval reuse scheduling), and the
library's host implementation against it. Codes: 0 = FP64, 1 = FP32, 2 = BF16; an upward
transition is a drop of a block's code from one iteration to the next; under reuse interval K
the decision of iteration K*floor(k/K) is in force at iteration k."""
import numpy as np
import pytest

import oracle


def _col(seq):
    return np.array(seq, np.uint8).reshape(-1, 1)


def test_transitions_inside_windows_are_delayed():
    # ups at k = 3 (2 -> 1) and k = 5 (1 -> 0); K = 2 keeps iterations 2 and 4 (codes 2, 1)
    ks, f = oracle.kstar_select(_col([2, 2, 2, 1, 1, 0, 0, 0]))
    assert list(f) == [0.0, 1.0, 1.0, 1.0] and ks == 1


def test_transitions_on_window_starts_are_not_delayed():
    # ups at k = 2 and k = 4: on the starts of K = 2 windows; K = 4 delays the one at k = 2
    ks, f = oracle.kstar_select(_col([2, 2, 1, 1, 0, 0, 0, 0]))
    assert list(f) == [0.0, 0.0, 0.5, 1.0] and ks == 2


def test_no_upward_transition_takes_the_largest_interval():
    ks, f = oracle.kstar_select(_col([0, 0, 1, 1, 2, 2]))   # only downward moves
    assert list(f) == [0.0, 0.0, 0.0] and ks == 4             # powers of two up to 6 rows


def test_the_limit_is_strict_and_counts_over_all_blocks():
    # block 0 goes up at k = 1 (delayed for K >= 2); blocks 1..10 at k = 2 (delayed for K = 4)
    log = np.zeros((4, 11), np.uint8)
    log[0, 0] = 1
    log[:2, 1:] = 2
    log[2:, 1:] = 1
    ks, f = oracle.kstar_select(log, 0.1)
    assert f[1] == pytest.approx(1 / 11) and f[2] == 1.0 and ks == 2
    ks, _ = oracle.kstar_select(log, 1 / 11)                  # "below" the limit: strict
    assert ks == 1


def test_a_window_decision_already_at_the_higher_precision_delays_nothing():
    # down at k = 1, back up at k = 2: K = 4 reuses iteration 0, which already has code 1
    ks, f = oracle.kstar_select(_col([1, 2, 1, 1]))
    assert list(f) == [0.0, 0.0, 0.0] and ks == 4


def test_empty_and_single_row_logs():
    assert oracle.kstar_select(np.zeros((0, 3), np.uint8))[0] == 1
    assert oracle.kstar_select(np.zeros((1, 3), np.uint8))[0] == 1


def test_library_host_selection_equals_oracle():
    from mixed_precision_sparse_gb300 import build, evocg
    build.build()
    rng = np.random.default_rng(3)
    for _ in range(300):
        rows, ncb = int(rng.integers(0, 50)), int(rng.integers(1, 8))
        p = rng.dirichlet([1, 1, 1])
        log = rng.choice(3, size=(rows, ncb), p=p).astype(np.uint8)
        if rows > 4 and rng.random() < 0.5:   # persistent patterns, as real runs show
            log = np.repeat(log[: rows // 4 + 1], 4, axis=0)[:rows]
        a, b = evocg.kstar_select(log), oracle.kstar_select(log)
        assert a[0] == b[0] and np.array_equal(a[1], b[1])
    with pytest.raises(evocg.EvocgError):
        evocg.kstar_select(np.full((2, 2), 3, np.uint8))      # codes are 0, 1, 2
