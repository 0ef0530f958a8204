"""Pins for the fp64 oracle, against things other than the oracle itself.

* hand-derived worked examples (tests/golden/hand_examples.json);
* closed forms of phi;
* a brute-force pairwise evaluation written here in numpy (phi as x+1 / e^x,
  not elu+1), for the causal and non-causal forms;
* torch float64 library routines (expm1, batched matmul, tril): the output
  as an explicit masked N x N kernel matrix, a route with no prefix sums and
  no state, which the "Linear Transformer" page says gives the recurrent
  result ("Comprobar la equivalencia entre cálculo recurrente y cálculo
  causal vectorizado");
* the blockwise form at several block lengths ("Linear Attention/es",
  "Entrenamiento: forma paralela");
* invariants that follow from the equations.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def _rng(seed):
    return np.random.default_rng(seed)


def _phi_np(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _bruteforce(q, k, v, causal, eps=1e-6):
    """Pairwise form, one query at a time, written independently of the oracle."""
    N = q.shape[0]
    fq, fk = _phi_np(q), _phi_np(k)
    y = np.zeros((N, v.shape[1]))
    for i in range(N):
        jmax = i + 1 if causal else N
        w = fk[:jmax] @ fq[i]
        y[i] = (w @ v[:jmax]) / max(w.sum(), eps)
    return y


def _rel(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


# --------------------------------------------------------------------------
# phi
# --------------------------------------------------------------------------
def test_phi_closed_form():
    x = np.array([0.0, 1.0, -1.0, 2.5, -50.0, 1e-300, -1e-300, 3.0])
    want = np.array([1.0, 2.0, math.exp(-1.0), 3.5, math.exp(-50.0), 1.0, 1.0, 4.0])
    got = oracle.phi(x)
    np.testing.assert_allclose(got, want, rtol=1e-15, atol=0)
    # positivity on both branches, continuity at 0
    xs = np.linspace(-30, 30, 6001)
    f = oracle.phi(xs)
    assert (f > 0).all()
    assert abs(oracle.phi([1e-12])[0] - oracle.phi([-1e-12])[0]) < 1e-11


# --------------------------------------------------------------------------
# hand-derived golden cases
# --------------------------------------------------------------------------
def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_hand_examples(case):
    q, k, v = (np.array(case[x], dtype=np.float64) for x in ("q", "k", "v"))
    eps = case["eps"]
    want = np.array(case["y"])
    if case["mode"] == "causal":
        y, S, z = oracle.causal_recurrent(q, k, v, eps=eps, return_state=True)
        np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-300)
        for C in (1, 2, 3):
            yc = oracle.causal_chunked(q, k, v, C, eps=eps)
            np.testing.assert_allclose(yc, want, rtol=1e-13, atol=1e-300)
        np.testing.assert_allclose(oracle.quadratic(q, k, v, causal=True, eps=eps), want,
                                   rtol=1e-13, atol=1e-300)
        # the same tokens fed one decode step at a time
        Sd = np.zeros((q.shape[1], v.shape[1]))
        zd = np.zeros(q.shape[1])
        for t in range(q.shape[0]):
            yt, Sd, zd = oracle.decode_step(q[t], k[t], v[t], Sd, zd, eps=eps)
            np.testing.assert_allclose(yt, want[t], rtol=1e-13, atol=1e-300)
    else:
        y, S, z = oracle.noncausal(q, k, v, eps=eps, return_state=True)
        np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-300)
        np.testing.assert_allclose(oracle.quadratic(q, k, v, causal=False, eps=eps), want,
                                   rtol=1e-13, atol=1e-300)
    if "S_final" in case:
        np.testing.assert_allclose(S, np.array(case["S_final"]), rtol=1e-14)
        np.testing.assert_allclose(z, np.array(case["z_final"]), rtol=1e-14)


# --------------------------------------------------------------------------
# brute force and library cross-checks
# --------------------------------------------------------------------------
@pytest.mark.parametrize("N,d,dv,scale,seed", [
    (1, 1, 1, 1.0, 0), (17, 1, 3, 1.0, 1), (64, 4, 5, 1.0, 2), (96, 32, 32, 0.3, 3),
    (256, 32, 16, 1.0, 4), (200, 8, 8, 3.0, 5)])
def test_recurrent_matches_bruteforce(N, d, dv, scale, seed):
    r = _rng(seed)
    q, k, v = (r.standard_normal((N, n)) * scale for n in (d, d, dv))
    y = oracle.causal_recurrent(q, k, v)
    assert _rel(y, _bruteforce(q, k, v, True)) < 1e-12
    yq = oracle.quadratic(q, k, v, causal=True)
    assert _rel(yq, _bruteforce(q, k, v, True)) < 1e-12
    yn = oracle.noncausal(q, k, v)
    assert _rel(yn, _bruteforce(q, k, v, False)) < 1e-12
    assert _rel(oracle.quadratic(q, k, v, causal=False), _bruteforce(q, k, v, False)) < 1e-12


def _torch_phi(x):
    """elu(x) + 1 from torch's expm1: x + 1 for x > 0, expm1(x) + 1 otherwise."""
    return torch.where(x > 0, x, torch.special.expm1(torch.clamp(x, max=0.0))) + 1.0


def _torch_kernel_matrix(q, k, v, causal, eps=1e-6):
    """The output as an explicit N x N kernel matrix, float64 torch routines:
    A = Phi(Q) Phi(K)^T (lower triangle only when causal, by torch.tril), then
    y = A V / max(A 1, eps) with batched matmuls.  No prefix sums and no state:
    a different route to the same numbers than the oracle's recurrence."""
    Q, K, V = (torch.from_numpy(np.ascontiguousarray(x)) for x in (q, k, v))
    A = torch.bmm(_torch_phi(Q), _torch_phi(K).transpose(1, 2))
    if causal:
        A = torch.tril(A)
    den = torch.maximum(A.sum(dim=2, keepdim=True), torch.tensor(eps, dtype=A.dtype))
    return (torch.bmm(A, V) / den).numpy()


@pytest.mark.parametrize("B,N,d,dv,seed", [(2, 64, 16, 16, 7), (3, 50, 8, 12, 8), (1, 128, 32, 32, 9)])
def test_library_cross_check(B, N, d, dv, seed):
    r = _rng(seed)
    q, k, v = (r.standard_normal((B, N, n)) for n in (d, d, dv))
    assert _rel(oracle.causal_recurrent(q, k, v), _torch_kernel_matrix(q, k, v, True)) < 1e-12
    assert _rel(oracle.noncausal(q, k, v), _torch_kernel_matrix(q, k, v, False)) < 1e-12


@pytest.mark.parametrize("C", [1, 3, 7, 64, 128, 300])
def test_chunked_equals_recurrent(C):
    r = _rng(11)
    N, d, dv = 300, 16, 24
    q, k, v = (r.standard_normal((2, N, n)) for n in (d, d, dv))
    y, S, z = oracle.causal_recurrent(q, k, v, return_state=True)
    yc, Sc, zc = oracle.causal_chunked(q, k, v, C, return_state=True)
    assert _rel(yc, y) < 1e-12
    assert _rel(Sc, S) < 1e-12 and _rel(zc, z) < 1e-12


# --------------------------------------------------------------------------
# invariants
# --------------------------------------------------------------------------
def test_noncausal_equals_last_causal_row():
    r = _rng(21)
    q, k, v = (r.standard_normal((3, 77, n)) for n in (8, 8, 5))
    yc, Sc, zc = oracle.causal_recurrent(q, k, v, return_state=True)
    yn, Sn, zn = oracle.noncausal(q, k, v, return_state=True)
    assert _rel(yn[:, -1], yc[:, -1]) < 1e-12
    assert _rel(Sn, Sc) < 1e-12 and _rel(zn, zc) < 1e-12


def test_constant_v_returns_v():
    r = _rng(22)
    q, k = (r.standard_normal((2, 90, 6)) for _ in range(2))
    c = np.array([1.5, -0.25, 3.0])
    v = np.broadcast_to(c, (2, 90, 3)).copy()
    for y in (oracle.causal_recurrent(q, k, v), oracle.noncausal(q, k, v),
              oracle.causal_chunked(q, k, v, 16)):
        np.testing.assert_allclose(y, np.broadcast_to(c, y.shape), rtol=1e-13, atol=1e-13)


def test_affine_equivariance_in_v():
    r = _rng(23)
    q, k, v = (r.standard_normal((2, 60, n)) for n in (5, 5, 4))
    a, b = -2.5, 0.75
    y = oracle.causal_recurrent(q, k, v)
    y2 = oracle.causal_recurrent(q, k, a * v + b)
    np.testing.assert_allclose(y2, a * y + b, rtol=1e-12, atol=1e-12)


def test_first_token_returns_v1_and_d1_cancels_q():
    r = _rng(24)
    q, k, v = (r.standard_normal((4, 1, n)) for n in (7, 7, 3))
    np.testing.assert_allclose(oracle.causal_recurrent(q, k, v), v, rtol=1e-14)
    # d = 1: y_i = sum_{j<=i} phi(k_j) v_j / sum_{j<=i} phi(k_j), independent of q
    q1, k1, v1 = (r.standard_normal((40, n)) for n in (1, 1, 2))
    fk = _phi_np(k1[:, 0])
    want = np.cumsum(fk[:, None] * v1, 0) / np.cumsum(fk)[:, None]
    np.testing.assert_allclose(oracle.causal_recurrent(q1, k1, v1), want, rtol=1e-12)
    np.testing.assert_allclose(oracle.causal_recurrent(q1 * 5 - 1, k1, v1), want, rtol=1e-12)


def test_noncausal_permutation_invariance():
    r = _rng(25)
    q, k, v = (r.standard_normal((50, n)) for n in (6, 6, 3))
    p = r.permutation(50)
    y = oracle.noncausal(q, k, v)
    np.testing.assert_allclose(oracle.noncausal(q, k[p], v[p]), y, rtol=1e-12)


def test_denominators_positive_and_outputs_convex():
    # y_t is a convex combination of v_1..v_t (all weights phi.phi > 0).
    r = _rng(26)
    q, k, v = (r.standard_normal((1, 120, n)) * 2 for n in (4, 4, 1))
    y = oracle.causal_recurrent(q, k, v)[0, :, 0]
    vv = v[0, :, 0]
    for t in range(120):
        assert vv[: t + 1].min() - 1e-12 <= y[t] <= vv[: t + 1].max() + 1e-12


def test_state_additive_over_segments():
    r = _rng(27)
    q, k, v = (r.standard_normal((2, 150, n)) for n in (8, 8, 6))
    y, S, z = oracle.causal_recurrent(q, k, v, return_state=True)
    cut = 61
    y1, S1, z1 = oracle.causal_recurrent(q[:, :cut], k[:, :cut], v[:, :cut], return_state=True)
    y2, S2, z2 = oracle.causal_recurrent(q[:, cut:], k[:, cut:], v[:, cut:], S_in=S1, z_in=z1,
                                         return_state=True)
    assert _rel(np.concatenate([y1, y2], 1), y) < 1e-12
    assert _rel(S2, S) < 1e-12 and _rel(z2, z) < 1e-12
    # and the segment sums add: S = S(first) + S(second from zero)
    _, S2b, z2b = oracle.causal_recurrent(q[:, cut:], k[:, cut:], v[:, cut:], return_state=True)
    assert _rel(S1 + S2b, S) < 1e-12 and _rel(z1 + z2b, z) < 1e-12
    # the chunked form continues from an initial state too
    yc2, Sc2, zc2 = oracle.causal_chunked(q[:, cut:], k[:, cut:], v[:, cut:], 16, S_in=S1,
                                          z_in=z1, return_state=True)
    assert _rel(yc2, y2) < 1e-12 and _rel(Sc2, S) < 1e-12


def test_prefill_then_decode_equals_causal():
    r = _rng(28)
    Np, M = 40, 12
    q, k, v = (r.standard_normal((3, Np + M, n)) for n in (8, 8, 8))
    y, S, z = oracle.causal_recurrent(q, k, v, return_state=True)
    _, Sd, zd = oracle.causal_recurrent(q[:, :Np], k[:, :Np], v[:, :Np], return_state=True)
    for t in range(Np, Np + M):
        yt, Sd, zd = oracle.decode_step(q[:, t], k[:, t], v[:, t], Sd, zd)
        assert _rel(yt, y[:, t]) < 1e-12
    assert _rel(Sd, S) < 1e-12 and _rel(zd, z) < 1e-12


def test_threads_do_not_change_results():
    r = _rng(29)
    q, k, v = (r.standard_normal((7, 33, n)) for n in (4, 4, 4))
    a = oracle.causal_recurrent(q, k, v, nthreads=1)
    b = oracle.causal_recurrent(q, k, v, nthreads=5)
    assert np.array_equal(a, b)


def test_empty_sequence():
    q = np.zeros((2, 0, 4)); v = np.zeros((2, 0, 3))
    y, S, z = oracle.causal_recurrent(q, q, v, return_state=True)
    assert y.shape == (2, 0, 3) and not S.any() and not z.any()
