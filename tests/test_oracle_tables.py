"""Pins of the oracle's score-table step (decay 0.95, threshold, expansion)."""
import json
import math
import os

import numpy as np

from oracle import sparse_attention_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_recurrence_handworked():
    g = json.load(open(os.path.join(GOLDEN, "score_table_recurrence.json")))
    v = np.zeros(8)
    s = np.zeros(8)
    for want in g["expected"]:
        v, s = orc.table_update(v, s, 4, [2], [g["a"]], r=g["r"])
        assert abs(v[2] - want) < 1e-15
        assert abs(s[4 - 1 - 2] - want) < 1e-15       # slash entry of offset 1


def test_closed_form_constant_weight():
    rng = np.random.default_rng(0)
    T0 = rng.random(16)
    a = rng.random(16)
    v, s = T0.copy(), np.zeros(16)
    for n in range(1, 40):
        v, s = orc.table_update(v, s, 16, np.arange(16), a)
        assert np.allclose(v, 0.95 ** n * T0 + (1 - 0.95 ** n) * a, atol=1e-14, rtol=0)


def test_unattended_entries_only_decay_and_mass_is_conserved():
    rng = np.random.default_rng(1)
    v, s = rng.random(100), rng.random(100)
    w = rng.random(7)
    w /= w.sum()
    pos = np.array([0, 1, 50, 60, 61, 97, 98])
    v2, s2 = orc.table_update(v, s, 99, pos, w)
    mask = np.ones(100, bool)
    mask[pos] = False
    assert np.allclose(v2[mask], 0.95 * v[mask], atol=1e-15)
    # the step adds (1 - r) of total weight 1 to each table
    assert abs((v2.sum() - 0.95 * v.sum()) - 0.05) < 1e-12
    assert abs((s2.sum() - 0.95 * s.sum()) - 0.05) < 1e-12


def test_slash_offset_moves_by_one_per_step():
    # weight on position 10 at length 40 lands on offset 29; at length 41 the
    # same position is offset 30
    v, s = np.zeros(64), np.zeros(64)
    v, s = orc.table_update(v, s, 40, [10], [1.0])
    assert abs(s[29] - 0.05) < 1e-15 and np.count_nonzero(s) == 1
    v, s = orc.table_update(v, s, 41, [10], [1.0])
    assert abs(s[30] - 0.05) < 1e-15 and abs(s[29] - 0.95 * 0.05) < 1e-15


def test_expansion_clipped_to_middle_region():
    # L = 40, S = 4, W = 20: M = [4, 20); seeds at 4 and 19
    L, S, W = 40, 4, 20
    v = np.zeros(64, np.float32)
    s = np.zeros(64, np.float32)
    v[4] = 1.0
    s[L - 1 - 19] = 1.0
    c, over = orc.table_candidates(v, s, L, S, W, beta=1.0, kcap=100)
    assert c.tolist() == [4, 5, 6, 18, 19] and not over


def test_threshold_is_strict_and_fp32():
    L, S, W = 100, 4, 16          # |I| = 20, tau = fp32(1)/fp32(20)
    tau = np.float32(1.0) / np.float32(20.0)
    v = np.zeros(128, np.float32)
    s = np.zeros(128, np.float32)
    v[30] = tau                                   # equal: not a seed
    v[50] = np.nextafter(tau, np.float32(1))      # just above: a seed
    c, _ = orc.table_candidates(v, s, L, S, W, beta=1.0, kcap=100)
    assert c.tolist() == [49, 50, 51, 52]


def test_capacity_keeps_lowest_positions():
    L, S, W = 200, 4, 16
    v = np.ones(256, np.float32)
    s = np.zeros(256, np.float32)
    c, over = orc.table_candidates(v, s, L, S, W, beta=1.0, kcap=10)
    assert over and c.tolist() == list(range(4, 14))


def test_merged_weights_are_a_softmax_over_the_attended_set():
    rng = np.random.default_rng(2)
    L = 300
    K = rng.standard_normal((L, 128))
    q = rng.standard_normal(128)
    pos, w = orc.merged_weights(q, K, L, 4, 32, [50, 50, 7, 299, 2], 0.1)
    assert pos.tolist() == list(range(4)) + [7, 50] + list(range(268, 300))
    assert abs(w.sum() - 1) < 1e-12
    z = 0.1 * K[pos] @ q
    assert np.allclose(w, np.exp(z) / np.exp(z).sum(), rtol=1e-12)
