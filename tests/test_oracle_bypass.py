"""Pins of the oracle's head-sparsity estimate and mean-value bypass
(reading R11 of LFPS Algorithm 1 step 1, Eq. (5), Eq. (6), App. B.1).

Each pin fixes the estimate by something other than its own formula: the
cases where the estimate is exact (one token; every global key equal), the
closed form for all-zero keys, and the log-normal mean it stands for, checked
against the brute-force sum over many normal keys."""
import math

import numpy as np
import pytest

from oracle import sparse_attention_oracle as orc

D = 128
SCALE = 1.0 / math.sqrt(D)


def _exact_lse_and_sink_weight(q, K, L):
    z = SCALE * (np.asarray(K[:L], dtype=np.float64) @ np.asarray(q, dtype=np.float64))
    m = z.max()
    lse = m + math.log(np.exp(z - m).sum())
    return lse, math.exp(z[0] - lse)


def test_single_token_is_exact():
    rng = np.random.default_rng(1)
    q, K, V = rng.normal(size=D), rng.normal(size=(1, D)), rng.normal(size=(1, D))
    rho, lse = orc.head_sparsity(q, K, 1, SCALE)
    assert rho == 1.0
    assert lse == SCALE * float(K[0] @ q)
    O, l = orc.attend(q, K, V, np.array([0]), SCALE)
    assert np.allclose(orc.bypass_output(V, 1), O, atol=1e-14)
    assert abs(l - lse) < 1e-12


@pytest.mark.parametrize("L", [1, 2, 6, 7, 8, 9, 100])
def test_zero_keys_closed_form(L):
    # every logit 0: sink mass 1, local min(6, L-1), global n = max(0, L-7)
    q = np.random.default_rng(L).normal(size=D)
    rho, lse = orc.head_sparsity(q, np.zeros((L, D)), L, SCALE)
    assert abs(rho - 1.0 / L) < 1e-15
    assert abs(lse - math.log(L)) < 1e-12


@pytest.mark.parametrize("L", [8, 9, 13, 50, 300])
def test_constant_global_keys_make_the_estimate_exact(L):
    # With one global key value the variance is 0 and n e^{z} is the exact
    # global mass; the sink and the six local keys are distinct random rows,
    # so a local window one token short or long, or the sink counted among
    # the global keys, moves the result away from the exact softmax.
    rng = np.random.default_rng(100 + L)
    q = rng.normal(size=D)
    K = np.repeat(rng.normal(size=(1, D)), L, axis=0)
    K[0] = rng.normal(size=D) * 2.0
    K[L - 6:] = rng.normal(size=(6, D)) * 2.0
    rho, lse = orc.head_sparsity(q, K, L, SCALE)
    lse_x, w0 = _exact_lse_and_sink_weight(q, K, L)
    assert abs(lse - lse_x) < 1e-12
    assert abs(rho - w0) < 1e-12


def test_global_mass_is_the_lognormal_mean():
    # n normal keys with mean mu and per-dim std sigma: sum_t e^{z_t} tends to
    # n exp(scale q.mu + scale^2 |q|^2 sigma^2 / 2).  Exponent variance 1 here,
    # so the sample mean is within about 0.5 % at this n; a dropped 1/2 or a
    # missing scale^2 is off by 40 % or more.
    rng = np.random.default_rng(7)
    n = 100_000
    q = rng.normal(size=D)
    q *= math.sqrt(D) / np.linalg.norm(q)              # scale^2 |q|^2 = 1
    mu = rng.normal(size=D) * 0.1
    K = mu[None, :] + rng.normal(size=(n + 7, D))       # sigma = 1
    K[0] = 0.0                                           # sink and local keys: logit 0
    K[n + 1:] = 0.0
    rho, lse = orc.head_sparsity(q, K, n + 7, SCALE)
    lse_x, _ = _exact_lse_and_sink_weight(q, K, n + 7)
    assert abs(lse - lse_x) < 0.02
    # and the closed form itself
    kbar = K[1:n + 1].mean(axis=0)
    expect = math.log(7 + n * math.exp(SCALE * float(kbar @ q) + 0.5 * 1.0 * K[1:n + 1].var(axis=0).mean()))
    assert abs(lse - expect) < 1e-9


def test_planted_sink_is_bypassed_and_a_plain_head_is_not():
    rng = np.random.default_rng(3)
    L = 4096
    K = rng.normal(size=(L, D))
    q_plain = rng.normal(size=D)
    rho_plain, _ = orc.head_sparsity(q_plain, K, L, SCALE)
    assert not orc.is_bypassed(rho_plain)
    q_sink = 20.0 * K[0] / np.linalg.norm(K[0]) * math.sqrt(D) / 8.0
    rho_sink, lse = orc.head_sparsity(q_sink, K, L, SCALE)
    assert orc.is_bypassed(rho_sink)
    lse_x, w0 = _exact_lse_and_sink_weight(q_sink, K, L)
    assert abs(rho_sink - w0) < 0.01          # the estimate tracks the true sink weight
    assert orc.is_bypassed(0.85 + 1e-12) and not orc.is_bypassed(0.85)


def test_empty_sequence():
    rho, lse = orc.head_sparsity(np.ones(D), np.zeros((0, D)), 0, SCALE)
    assert rho == 0.0 and lse == -math.inf
    assert np.array_equal(orc.bypass_output(np.zeros((0, D)), 0), np.zeros(D))


def test_partition_covers_every_token_once():
    for L in range(1, 20):
        loc, glo = orc.sparsity_partition(L)
        allt = np.concatenate([[0], glo, loc])
        assert np.array_equal(np.sort(allt), np.arange(L))
        assert len(loc) == min(6, L - 1)


@pytest.mark.parametrize("L", [2, 3, 7, 64, 1000])
def test_bypass_output_is_the_mean_over_all_L_rows(L):
    # V row t = t e_0 (plus rows beyond L that must not count): the mean over
    # rows 0..L-1 is (L-1)/2 e_0 by the arithmetic-series sum, so a mean over
    # a shorter or shifted range, or one that includes a row past L, fails.
    V = np.zeros((L + 5, D))
    V[:, 0] = np.arange(L + 5, dtype=np.float64)
    V[L:, 1] = 1e6
    got = orc.bypass_output(V, L)
    want = np.zeros(D)
    want[0] = (L - 1) / 2.0
    assert np.array_equal(got, want)
