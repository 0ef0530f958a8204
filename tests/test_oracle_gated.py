"""Pins of the oracle's gated form, its feature-map choice and the random-feature
map (CPU, fp64) -- "Linear Attention/es", "Variantes y extensiones" (gated
linear attention) and "Mapas de características" (identity and random-feature
maps).  Each check compares the oracle with something it does not share
arithmetic with: hand-worked values, the closed-form pairwise weights with
products of gates (``gated_pins.brute_gated``), the plain and decayed forms
it must reduce to, and the softmax kernel the random features estimate.
"""
import json
import os

import numpy as np
import pytest

import oracle
from tests.gated_pins import brute_gated, phi_np, random_features_np

HERE = os.path.dirname(__file__)


def _rng(s):
    return np.random.default_rng(s)


def _rel(a, b):
    return float(np.abs(np.asarray(a) - np.asarray(b)).max() / max(np.abs(b).max(), 1e-300))


def test_hand_examples():
    with open(os.path.join(HERE, "golden", "gated_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q, k, v = (np.array(c[x], dtype=np.float64) for x in ("q", "k", "v"))
        y = oracle.causal_gated(q, k, v, gate=np.array(c["gate"]), phi=c["phi"], eps=c["eps"])
        np.testing.assert_allclose(y, np.array(c["y"]), rtol=1e-14, err_msg=c["name"])


@pytest.mark.parametrize("kind", ["elu1", "identity"])
@pytest.mark.parametrize("per_feature", [False, True])
@pytest.mark.parametrize("N,d,dv,seed", [(1, 1, 1, 0), (23, 3, 2, 1), (64, 8, 5, 2)])
def test_matches_closed_form(kind, per_feature, N, d, dv, seed):
    r = _rng(seed)
    q, k, v = (r.standard_normal((N, n)) for n in (d, d, dv))
    if kind == "identity":   # keep the denominators away from the clamp
        q, k = np.abs(q) + 0.1, np.abs(k) + 0.1
    g = r.uniform(0.0, 1.0, (N, d) if per_feature else (N,))
    S_in = r.standard_normal((d, dv))
    z_in = r.uniform(0.5, 2.0, d)
    y = oracle.causal_gated(q, k, v, gate=g, phi=kind, S_in=S_in, z_in=z_in)
    assert _rel(y, brute_gated(q, k, v, g, kind, S_in=S_in, z_in=z_in)) < 1e-12
    y0 = oracle.causal_gated(q, k, v, gate=g, phi=kind)
    assert _rel(y0, brute_gated(q, k, v, g, kind)) < 1e-12


def test_reduces_to_plain_and_decayed_forms():
    r = _rng(3)
    q, k, v = (r.standard_normal((2, 3, 40, n)) for n in (6, 6, 4))
    ones = np.ones((2, 3, 40))
    np.testing.assert_allclose(oracle.causal_gated(q, k, v, gate=ones),
                               oracle.causal_recurrent(q, k, v), rtol=1e-13)
    np.testing.assert_allclose(oracle.causal_gated(q, k, v), oracle.causal_recurrent(q, k, v),
                               rtol=1e-13)
    gam = np.array([0.5, 0.9, 0.99])
    g = np.broadcast_to(gam[None, :, None], (2, 3, 40))
    np.testing.assert_allclose(oracle.causal_gated(q, k, v, gate=g),
                               oracle.causal_recurrent_decay(q, k, v, gam), rtol=1e-12)
    gf = np.broadcast_to(gam[None, :, None, None], (2, 3, 40, 6))
    np.testing.assert_allclose(oracle.causal_gated(q, k, v, gate=gf),
                               oracle.causal_recurrent_decay(q, k, v, gam), rtol=1e-12)


def test_closed_gate_keeps_only_the_current_token():
    r = _rng(4)
    q, k, v = (r.standard_normal((30, n)) for n in (5, 5, 3))
    g = r.uniform(0.2, 1.0, 30)
    g[[0, 7, 19]] = 0.0
    y = oracle.causal_gated(q, k, v, gate=g)
    for t in (0, 7, 19):   # the state restarts: y_t = v_t
        np.testing.assert_allclose(y[t], v[t], rtol=1e-13)
    # and the final state after a closed gate at the last token is phi(k) v^T
    g[-1] = 0.0
    _, S, z = oracle.causal_gated(q, k, v, gate=g, return_state=True)
    np.testing.assert_allclose(S, np.outer(phi_np(k[-1]), v[-1]), rtol=1e-13)
    np.testing.assert_allclose(z, phi_np(k[-1]), rtol=1e-13)


def test_identity_map_matches_bilinear_pairwise_forms():
    r = _rng(5)
    q, k = (np.abs(r.standard_normal((2, 50, 4))) + 0.05 for _ in range(2))
    v = r.standard_normal((2, 50, 3))
    for causal in (True, False):
        want = np.stack([
            np.stack([(np.tril(q[b] @ k[b].T) if causal else q[b] @ k[b].T)[i] @ v[b]
                      / (np.tril(q[b] @ k[b].T) if causal else q[b] @ k[b].T)[i].sum()
                      for i in range(50)]) for b in range(2)])
        got = (oracle.causal_gated(q, k, v, phi="identity") if causal
               else oracle.noncausal(q, k, v, phi="identity"))
        assert _rel(got, want) < 1e-12
        assert _rel(oracle.quadratic(q, k, v, causal, phi="identity"), want) < 1e-12


def test_gate_state_is_additive_over_a_split():
    """prefill(N1) -> (S, z); continuing from it over N2 equals the tail of
    the whole run (the gate of a token multiplies the state it receives)."""
    r = _rng(6)
    q, k, v = (r.standard_normal((3, 70, n)) for n in (4, 4, 2))
    g = r.uniform(0.3, 1.0, (3, 70, 4))
    y, S, z = oracle.causal_gated(q, k, v, gate=g, return_state=True)
    _, S1, z1 = oracle.causal_gated(q[:, :30], k[:, :30], v[:, :30], gate=g[:, :30],
                                    return_state=True)
    y2, S2, z2 = oracle.causal_gated(q[:, 30:], k[:, 30:], v[:, 30:], gate=g[:, 30:],
                                     S_in=S1, z_in=z1, return_state=True)
    np.testing.assert_allclose(y2, y[:, 30:], rtol=1e-12)
    np.testing.assert_allclose(S2, S, rtol=1e-12)
    np.testing.assert_allclose(z2, z, rtol=1e-12)


def test_random_features_closed_form_and_positivity():
    r = _rng(7)
    x = r.standard_normal((3, 20, 8)) * 0.5
    W = r.standard_normal((32, 8))
    f = oracle.random_features(x, W)
    assert f.shape == (3, 20, 32) and (f > 0).all()
    np.testing.assert_allclose(f, random_features_np(x, W), rtol=1e-13)


def test_random_features_estimate_the_softmax_kernel():
    """With Gaussian rows w ~ N(0, I), phi(q) . phi(k) averages exp(w.(q+k) -
    (|q|^2 + |k|^2)/2) over the rows, whose expectation is exp(q . k); with
    2^17 rows the estimate is within a few 1/sqrt(m) of it."""
    r = _rng(8)
    d, m = 4, 1 << 17
    W = r.standard_normal((m, d))
    qs = r.standard_normal((5, d)) * 0.4
    ks = r.standard_normal((5, d)) * 0.4
    est = np.sum(oracle.random_features(qs, W) * oracle.random_features(ks, W), axis=1)
    want = np.exp(np.sum(qs * ks, axis=1))
    assert np.all(np.abs(est / want - 1) < 0.03), est / want
