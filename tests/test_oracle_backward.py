"""Pins for the oracle's gradients of the causal form (CPU only, fp64).

The oracle's backward is checked against things it does not share code
with: central differences of the (separately pinned) forward, torch
autograd through the pairwise form, closed forms for one token, and
invariants of the normalised output.
"""
import numpy as np
import pytest

import oracle
from tests import backward_pins as bp


def _phi(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _dphi(x):
    return np.where(x > 0, 1.0, np.exp(np.minimum(x, 0.0)))


@pytest.mark.parametrize("N,d,dv,with_state,seed", [
    (6, 3, 2, False, 0), (5, 2, 4, True, 1), (9, 4, 4, False, 2), (1, 3, 3, True, 3)])
def test_backward_matches_finite_differences(N, d, dv, with_state, seed):
    r = np.random.default_rng(seed)
    q, k = r.standard_normal((2, 2, N, d))
    v, dy = r.standard_normal((2, 2, N, dv))
    S_in = r.standard_normal((2, d, dv)) if with_state else None
    z_in = np.abs(r.standard_normal((2, d))) + 0.5 if with_state else None
    want = bp.finite_difference_grads(q, k, v, dy, 1e-6, S_in, z_in)
    got = oracle.causal_backward(q, k, v, dy, eps=1e-6, S_in=S_in, z_in=z_in,
                                 return_state_grad=True, nthreads=1)
    for name, g, w in zip(("dq", "dk", "dv", "dS_in", "dz_in"), got, want):
        if w is None:
            continue
        np.testing.assert_allclose(g, w, rtol=1e-6, atol=1e-7 * np.abs(w).max(), err_msg=name)


def test_backward_with_partly_active_clamp():
    """Tokens whose denominator is below eps pass no gradient through it."""
    assert bp.fd_pin_passes(seed=3)
    assert bp.fd_pin_passes(seed=4)


def test_backward_fully_clamped_is_linear_in_dy_over_eps():
    """With eps above every denominator, y = num / eps and dv_t = sum_{s>=t} w_st dy_s / eps."""
    r = np.random.default_rng(7)
    q, k = r.standard_normal((2, 7, 3))
    v, dy = r.standard_normal((2, 7, 2))
    eps = 1e3
    dq, dk, dvv = oracle.causal_backward(q, k, v, dy, eps=eps, nthreads=1)
    fq, fk = _phi(q), _phi(k)
    w = np.tril(fq @ fk.T)                       # w[s, t] = phi(q_s).phi(k_t), t <= s
    np.testing.assert_allclose(dvv, w.T @ dy / eps, rtol=1e-12)
    # dL/dphi(q_s) = sum_{t<=s} phi(k_t) (v_t . dy_s) / eps
    dfq = (np.tril(dy @ v.T) @ fk) / eps
    np.testing.assert_allclose(dq, dfq * _dphi(q), rtol=1e-12)
    want = bp.finite_difference_grads(q, k, v, dy, eps)
    np.testing.assert_allclose(dk, want[1], rtol=1e-6, atol=1e-9)


@pytest.mark.parametrize("N,d,dv,seed", [(12, 4, 3, 0), (33, 8, 8, 1)])
def test_backward_matches_autograd_of_pairwise_form(N, d, dv, seed):
    r = np.random.default_rng(seed)
    q, k = 0.7 * r.standard_normal((2, 3, N, d))
    v, dy = r.standard_normal((2, 3, N, dv))
    S_in = r.standard_normal((3, d, dv))
    z_in = np.abs(r.standard_normal((3, d))) + 0.1
    want = bp.autograd_grads(q, k, v, dy, 1e-6, S_in, z_in)
    got = oracle.causal_backward(q, k, v, dy, eps=1e-6, S_in=S_in, z_in=z_in,
                                 return_state_grad=True)
    for name, g, w in zip(("dq", "dk", "dv", "dS_in", "dz_in"), got, want):
        np.testing.assert_allclose(g, w, rtol=1e-10, atol=1e-12 * np.abs(w).max(), err_msg=name)


def test_single_token_closed_form():
    """N = 1 from a zero state: y_1 = v_1 whatever q and k are, so dv = dy, dq = dk = 0."""
    r = np.random.default_rng(11)
    q, k = r.standard_normal((2, 4, 1, 5))
    v, dy = r.standard_normal((2, 4, 1, 3))
    dq, dk, dvv = oracle.causal_backward(q, k, v, dy)
    np.testing.assert_allclose(dvv, dy, rtol=1e-13)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13


def test_backward_invariants():
    """Shift of v by c shifts every y by c: sum_t dv_t = sum_t dy_t.
    y_t is homogeneous of degree 0 in phi(q_t): phi(q_t) . dL/dphi(q_t) = 0."""
    r = np.random.default_rng(5)
    q, k = r.standard_normal((2, 3, 64, 6))
    v, dy = r.standard_normal((2, 3, 64, 4))
    dq, dk, dvv = oracle.causal_backward(q, k, v, dy)
    np.testing.assert_allclose(dvv.sum(-2), dy.sum(-2), rtol=1e-11, atol=1e-11)
    dfq = dq / _dphi(q)
    proj = (dfq * _phi(q)).sum(-1)
    assert np.abs(proj).max() < 1e-11 * np.abs(dfq).max() * 6


def test_backward_empty_sequence_and_zero_dy():
    q = np.zeros((2, 0, 3))
    v = np.zeros((2, 0, 2))
    dq, dk, dvv, dS, dz = oracle.causal_backward(q, q, v, v, return_state_grad=True)
    assert dq.shape == (2, 0, 3) and dvv.shape == (2, 0, 2)
    assert not dS.any() and not dz.any()
    r = np.random.default_rng(1)
    q, k = r.standard_normal((2, 2, 9, 3))
    v = r.standard_normal((2, 9, 2))
    for g in oracle.causal_backward(q, k, v, np.zeros_like(v)):
        assert not g.any()


def test_backward_threads_do_not_change_results():
    r = np.random.default_rng(2)
    q, k = r.standard_normal((2, 5, 20, 4))
    v, dy = r.standard_normal((2, 5, 20, 3))
    a = oracle.causal_backward(q, k, v, dy, nthreads=1)
    b = oracle.causal_backward(q, k, v, dy, nthreads=4)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("seed", [5, 6])
def test_backward_with_decay_matches_finite_differences(seed):
    """With per-head decays (RetNet's update) and an initial state."""
    assert bp.fd_decay_pin_passes(seed=seed)


def test_backward_with_decay_one_is_the_plain_backward():
    r = np.random.default_rng(8)
    q, k = r.standard_normal((2, 2, 3, 15, 4))
    v, dy = r.standard_normal((2, 2, 3, 15, 5))
    a = oracle.causal_backward(q, k, v, dy)
    b = oracle.causal_backward(q, k, v, dy, gamma=np.ones(3))
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_backward_with_decay_matches_autograd():
    """The pairwise form with gamma^(t-j) weights, differentiated by torch."""
    import torch
    r = np.random.default_rng(9)
    N, d, dv, gam = 14, 4, 3, 0.8
    q, k = 0.7 * r.standard_normal((2, N, d))
    v, dy = r.standard_normal((2, N, dv))
    t = [torch.tensor(x, requires_grad=True) for x in (q, k, v)]
    phi = lambda x: torch.where(x > 0, x + 1.0, torch.exp(torch.clamp(x, max=0.0)))
    i = torch.arange(N, dtype=torch.float64)
    mask = torch.tril(torch.pow(gam, (i[:, None] - i[None, :]).clamp(min=0)))
    w = (phi(t[0]) @ phi(t[1]).T) * mask
    y = (w @ t[2]) / w.sum(-1).clamp_min(1e-6)[:, None]
    (y * torch.tensor(dy)).sum().backward()
    got = oracle.causal_backward(q, k, v, dy, gamma=[gam])
    for g, x in zip(got, t):
        np.testing.assert_allclose(g, x.grad.numpy(), rtol=1e-10, atol=1e-12)
