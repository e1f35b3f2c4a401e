"""The acceptance rule for greedy choices over GPU logits (CPU)."""
import numpy as np

from tests.argmax_rule import acceptable


def test_clear_top_admits_only_the_oracle_argmax():
    y = np.array([1.0, 3.0, 2.0, -5.0])
    b = np.full(4, 1e-3)
    assert [acceptable(y, b, t) for t in range(4)] == [False, True, False, False]


def test_near_tie_admits_either_of_the_top_two():
    y = np.array([1.0, 3.0, 3.0 - 1e-5, 2.0])
    b = np.full(4, 1e-4)
    assert [acceptable(y, b, t) for t in range(4)] == [False, True, True, False]


def test_exact_tie_admits_both():
    y = np.array([0.5, 2.0, 2.0])
    assert acceptable(y, np.zeros(3), 1) and acceptable(y, np.zeros(3), 2) and not acceptable(y, np.zeros(3), 0)


def test_bounds_decide_at_the_margin():
    y = np.array([3.0, 2.875])
    assert not acceptable(y, np.array([0.03125, 0.03125]), 1)   # 2.90625 < 2.96875
    assert acceptable(y, np.array([0.0625, 0.0625]), 1)         # 2.9375 >= 2.9375
