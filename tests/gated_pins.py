"""Independent checks for the gated and feature-map forms of the oracle (CPU, fp64).

``brute_gated`` writes the causal output from its closed form rather than the
recurrence: unrolling S_t = diag(g_t) S_{t-1} + phi(k_t) v_t^T gives

  S_i = diag(prod_{u=0..i} g_u) S_in + sum_{j<=i} diag(prod_{u=j+1..i} g_u) phi(k_j) v_j^T,

so y_i = phi(q_i)^T S_i / max(phi(q_i)^T z_i, eps) with pair weights
w_ij = sum_a phi(q_i)_a phi(k_j)_a prod_{u=j+1..i} g_{u,a}, formed here with
numpy products of the gates (no running state).
"""
import numpy as np


def phi_np(x, kind="elu1"):
    x = np.asarray(x, np.float64)
    if kind == "identity":
        return x
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def brute_gated(q, k, v, gate=None, kind="elu1", eps=1e-6, S_in=None, z_in=None):
    """One head: q, k [N, d], v [N, dv], gate None, [N] or [N, d]."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    N, d = q.shape
    g = np.ones((N, d)) if gate is None else np.asarray(gate, np.float64)
    if g.ndim == 1:
        g = np.repeat(g[:, None], d, axis=1)
    fq, fk = phi_np(q, kind), phi_np(k, kind)
    y = np.zeros((N, v.shape[1]))
    for i in range(N):
        num = np.zeros(v.shape[1])
        den = 0.0
        for j in range(i + 1):
            prod = np.prod(g[j + 1:i + 1], axis=0)          # per feature, empty product = 1
            w = float(np.sum(fq[i] * fk[j] * prod))
            num += w * v[j]
            den += w
        if S_in is not None:
            pin = np.prod(g[:i + 1], axis=0)
            num += (fq[i] * pin) @ np.asarray(S_in, np.float64)
            den += float(np.sum(fq[i] * pin * np.asarray(z_in, np.float64)))
        y[i] = num / max(den, eps)
    return y


def random_features_np(x, W):
    x, W = np.asarray(x, np.float64), np.asarray(W, np.float64)
    return np.exp(x @ W.T - 0.5 * np.sum(x * x, axis=-1, keepdims=True)) / np.sqrt(W.shape[0])
