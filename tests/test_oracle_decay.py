"""Pins for the oracle's causal form with a per-head decay (CPU only, fp64).

RetNet's update ("Linear Attention/es", "Variantes y extensiones"):
S_t = gamma S_{t-1} + phi(k_t) v_t^T, z_t decayed the same way.
"""
import numpy as np
import pytest

import oracle


def _phi(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def brute_decay(q, k, v, gamma, eps=1e-6, S_in=None, z_in=None):
    """y_t = (gamma^(t+1) phi(q_t)^T S_in + sum_{j<=t} gamma^(t-j) w_tj v_j)
             / max(gamma^(t+1) phi(q_t)^T z_in + sum_{j<=t} gamma^(t-j) w_tj, eps)."""
    fq, fk = _phi(q), _phi(k)
    N = q.shape[0]
    y = np.zeros((N, v.shape[1]))
    for t in range(N):
        p = gamma ** (t - np.arange(t + 1))
        w = (fk[:t + 1] @ fq[t]) * p
        num, den = w @ v[:t + 1], w.sum()
        if S_in is not None:
            num = num + gamma ** (t + 1) * (fq[t] @ S_in)
            den = den + gamma ** (t + 1) * (fq[t] @ z_in)
        y[t] = num / max(den, eps)
    return y


def test_hand_example():
    """d = dv = 1, phi(q) = 1, phi(k) = (1, 2), v = (1, 4), gamma = 1/2:
    S = 1, z = 1 -> y_0 = 1; S = 1/2 + 8, z = 1/2 + 2 -> y_1 = 8.5 / 2.5 = 3.4."""
    q = np.zeros((2, 1))
    k = np.array([[0.0], [1.0]])
    v = np.array([[1.0], [4.0]])
    y, S, z = oracle.causal_recurrent_decay(q, k, v, [0.5], return_state=True)
    np.testing.assert_allclose(y[:, 0], [1.0, 3.4], rtol=1e-15)
    np.testing.assert_allclose(S.reshape(-1), [8.5], rtol=1e-15)
    np.testing.assert_allclose(z.reshape(-1), [2.5], rtol=1e-15)


@pytest.mark.parametrize("gamma", [0.5, 0.9, 0.999])
@pytest.mark.parametrize("with_state", [False, True])
def test_matches_bruteforce(gamma, with_state):
    r = np.random.default_rng(int(gamma * 1000) + with_state)
    q, k = r.standard_normal((2, 37, 5))
    v = r.standard_normal((37, 3))
    S_in = r.standard_normal((5, 3)) if with_state else None
    z_in = np.abs(r.standard_normal(5)) + 0.5 if with_state else None
    got = oracle.causal_recurrent_decay(q, k, v, [gamma], S_in=S_in, z_in=z_in)
    np.testing.assert_allclose(got, brute_decay(q, k, v, gamma, S_in=S_in, z_in=z_in),
                               rtol=1e-11, atol=1e-12)


def test_gamma_one_is_the_plain_form_and_gamma_zero_returns_v():
    r = np.random.default_rng(3)
    q, k = r.standard_normal((2, 2, 3, 20, 4))
    v = r.standard_normal((2, 3, 20, 6))
    assert np.array_equal(oracle.causal_recurrent_decay(q, k, v, np.ones(3)),
                          oracle.causal_recurrent(q, k, v))
    # gamma = 0 forgets everything but the current token: y_t = v_t
    np.testing.assert_allclose(oracle.causal_recurrent_decay(q, k, v, np.zeros(3)), v,
                               rtol=1e-13, atol=1e-14)


def test_per_head_gamma_and_constant_v():
    r = np.random.default_rng(4)
    q, k = r.standard_normal((2, 2, 3, 30, 4))
    v = np.broadcast_to(r.standard_normal(5), (2, 3, 30, 5)).copy()
    gam = np.array([0.3, 0.8, 0.99])
    # a normalised average of a constant is that constant
    np.testing.assert_allclose(oracle.causal_recurrent_decay(q, k, v, gam), v, rtol=1e-12)
    v = r.standard_normal((2, 3, 30, 5))
    y = oracle.causal_recurrent_decay(q, k, v, gam)
    for b in range(2):
        for h in range(3):
            np.testing.assert_allclose(y[b, h], brute_decay(q[b, h], k[b, h], v[b, h], gam[h]),
                                       rtol=1e-11, atol=1e-12)


def test_state_carries_across_a_split():
    """Running the first half, then the second from its final state, equals one run."""
    r = np.random.default_rng(5)
    q, k = r.standard_normal((2, 4, 50, 8))
    v = r.standard_normal((4, 50, 8))
    gam = np.array([0.6, 0.9, 0.95, 1.0])
    y = oracle.causal_recurrent_decay(q, k, v, gam)
    y1, S, z = oracle.causal_recurrent_decay(q[:, :20], k[:, :20], v[:, :20], gam,
                                             return_state=True)
    y2 = oracle.causal_recurrent_decay(q[:, 20:], k[:, 20:], v[:, 20:], gam, S_in=S, z_in=z)
    np.testing.assert_allclose(np.concatenate([y1, y2], axis=1), y, rtol=1e-12)
