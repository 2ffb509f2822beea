"""Pins of the oracle's approximate expert substitution (MoE-CORE), CPU only."""
import numpy as np

from oracle.aes import aes_substitute


def _res(E, on):
    r = np.zeros(E, bool)
    r[list(on)] = True
    return r


def test_low_score_miss_within_alpha_takes_the_best_resident_unselected():
    # top-2 = experts 0, 1; the rank-3 boundary is expert 2's logit 1.9; expert 1 is missing and
    # float32(2.0) - float32(1.9) = 0.100000024: within alpha = 0.2, outside alpha = 0.05
    z = np.array([[3.0, 2.0, 1.9, 1.0, 0.5, 0.0]], np.float32)
    ids = np.array([[0, 1]])
    res = _res(6, [0, 3, 5])
    new, n = aes_substitute(z, ids, res, 0.2)
    assert new.tolist() == [[0, 3]] and n == 1          # expert 3: the best resident unselected
    new, n = aes_substitute(z, ids, res, 0.05)
    assert new.tolist() == [[0, 1]] and n == 0


def test_several_misses_in_rank_order_and_running_out_of_substitutes():
    z = np.array([[2.0, 1.95, 1.9, 1.85, 1.0, 0.9]], np.float32)
    ids = np.array([[0, 1, 2]])                          # boundary: 1.85
    new, n = aes_substitute(z, ids, _res(6, [4, 5]), 0.12)
    assert new.tolist() == [[0, 4, 5]] and n == 2         # 0 is 0.15 above: a high-score miss, kept
    new, n = aes_substitute(z, ids, _res(6, [5]), 0.12)
    assert new.tolist() == [[0, 5, 2]] and n == 1         # one substitute only


def test_resident_selected_and_full_k_are_untouched():
    rng = np.random.default_rng(0)
    z = rng.standard_normal((5, 8)).astype(np.float32)
    ids = np.argsort(-z, axis=1, kind="stable")[:, :3]
    new, n = aes_substitute(z, ids, np.ones(8, bool), 10.0)      # everything resident
    assert n == 0 and np.array_equal(new, ids)
    ids8 = np.argsort(-z, axis=1, kind="stable")
    new, n = aes_substitute(z, ids8, np.zeros(8, bool), 10.0)    # k = E: no boundary
    assert n == 0 and np.array_equal(new, ids8)


def test_alpha_zero_substitutes_only_exact_boundary_ties():
    z = np.array([[1.0, 0.5, 0.5, 0.1]], np.float32)     # expert 1 ties the boundary (expert 2)
    ids = np.array([[0, 1]])
    new, n = aes_substitute(z, ids, _res(4, [0, 3]), 0.0)
    assert new.tolist() == [[0, 3]] and n == 1
