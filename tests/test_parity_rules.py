"""The comparison rules themselves, on the CPU: each rule accepts what the
reading allows and rejects a planted mistake in a made-up GPU result. No GPU."""
import numpy as np
import pytest
import torch

import oracle
from parity import certain_zero_scores, check_kept_set


def _row(pos, K):
    r = np.full(K, -1, dtype=np.int64)
    r[:len(pos)] = sorted(pos)
    return r


def test_kept_set_accepts_the_oracle_set_and_near_ties():
    s = np.array([5.0, 1.0, 3.0, 3.002, 0.5, 2.999])
    check_kept_set(_row([0, 2, 3], 3), s, 3)               # the exact top 3 (K-th = 3.0)
    check_kept_set(_row([0, 3, 5], 3), s, 3)               # 2.999 lies within 1e-3 of the K-th
    with pytest.raises(AssertionError):                     # 1.0 does not
        check_kept_set(_row([0, 1, 3], 3), s, 3)


def test_kept_set_rejects_a_tie_broken_out_of_order_at_zero():
    # the K-th best is exactly 0 and positions 1, 3, 4, 6 tie there; K leaves
    # room for two of them: 1 and 3 by the tie rule
    s = np.array([2.0, 0.0, 1.0, 0.0, 0.0, 3.0, 0.0])
    cz = np.array([False, True, False, True, True, False, True])
    check_kept_set(_row([0, 1, 2, 3, 5], 5), s, 5, "ok", cz)
    with pytest.raises(AssertionError, match="position order"):
        check_kept_set(_row([0, 1, 2, 4, 5], 5), s, 5, "planted", cz)
    # without certain ties (signs too close to call), the near-tie rule alone applies
    check_kept_set(_row([0, 1, 2, 4, 5], 5), s, 5, "uncertain", np.zeros(7, dtype=bool))


def test_kept_set_structure_rules():
    s = np.arange(10, dtype=np.float64)
    with pytest.raises(AssertionError, match="ascending"):
        check_kept_set(np.array([9, 8, 7]), s, 3)
    with pytest.raises(AssertionError, match="padding"):
        check_kept_set(np.array([0, 1, 2, 3]), s[:3], 4)
    with pytest.raises(AssertionError, match="out of range"):    # a short row keeps every position
        check_kept_set(np.array([0, 2, -1, -1]), s[:3], 4)


def test_certain_zero_marks_only_clearly_negative_dots():
    # one head; key 0 gives a dot of -4 (certain), key 1 a dot of -1e-6 of a
    # magnitude sum of 2 (too close to call), key 2 a positive dot
    q = torch.tensor([[[1.0, 1.0]]])
    k = torch.tensor([[-2.0, -2.0], [1.0, -1.000001], [1.0, 0.5]])
    w = torch.tensor([[1.0]])
    cz = certain_zero_scores(q, w, k, np.array([0]), np.array([0]), np.array([3]))[0]
    assert cz.tolist() == [True, False, False]
    s = oracle.indexer(q, w, k, np.array([0]), np.array([0]), np.array([3]))[0]
    assert s[0] == 0 and s[1] == 0 and s[2] == 1.5


def test_certain_zero_needs_every_head_negative():
    q = torch.tensor([[[1.0, 0.0], [0.0, 1.0]]])             # two heads
    k = torch.tensor([[-1.0, -1.0], [-1.0, 1.0]])
    w = torch.tensor([[0.5, -0.5]])                           # signed weights
    cz = certain_zero_scores(q, w, k, np.array([0]), np.array([0]), np.array([2]))[0]
    assert cz.tolist() == [True, False]


def test_certain_zero_on_fp8_codes():
    from workloads import quantize_rows_e4m3
    qf = torch.tensor([[[1.0, 2.0]]])
    kf = torch.tensor([[-3.0, -1.0], [3.0, 1.0]])
    q8, qs = quantize_rows_e4m3(qf)
    k8, ks = quantize_rows_e4m3(kf)
    w = torch.tensor([[1.0]])
    cz = certain_zero_scores(q8, w, k8, np.array([0]), np.array([0]), np.array([2]), qs, ks)[0]
    assert cz.tolist() == [True, False]
