"""Independent checks for the oracle's gradients (CPU, fp64).

Neither helper shares arithmetic with ``oracle.causal_backward``:

* ``finite_difference_grads`` perturbs each input of the oracle's forward
  (``oracle.causal_recurrent``, pinned on its own) and takes central
  differences of the loss sum_t dy_t . y_t;
* ``autograd_grads`` writes the causal output in the pairwise form
  y_i = (phi(q_i)^T S_in + sum_{j<=i} w_ij v_j) / max(phi(q_i)^T z_in + sum_{j<=i} w_ij, eps),
  w_ij = phi(q_i)^T phi(k_j), as plain float64 torch operations and lets
  autograd differentiate it.
"""
import numpy as np

import oracle


def loss(q, k, v, dy, eps, S_in=None, z_in=None, gamma=None) -> float:
    if gamma is None:
        y = oracle.causal_recurrent(q, k, v, eps=eps, S_in=S_in, z_in=z_in, nthreads=1)
    else:
        y = oracle.causal_recurrent_decay(q, k, v, gamma, eps=eps, S_in=S_in, z_in=z_in,
                                          nthreads=1)
    return float((y * dy).sum())


def finite_difference_grads(q, k, v, dy, eps, S_in=None, z_in=None, h=1e-6, gamma=None):
    """Central differences of the loss for every element of q, k, v (and S_in, z_in)."""
    args = [np.array(a, dtype=np.float64) for a in (q, k, v)]
    state = [None if a is None else np.array(a, dtype=np.float64) for a in (S_in, z_in)]
    grads = []
    for which in range(5):
        x = args[which] if which < 3 else state[which - 3]
        if x is None:
            grads.append(None)
            continue
        g = np.empty_like(x)
        flat, gflat = x.reshape(-1), g.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp = loss(*args, dy, eps, *state, gamma=gamma)
            flat[i] = old - h
            lm = loss(*args, dy, eps, *state, gamma=gamma)
            flat[i] = old
            gflat[i] = (lp - lm) / (2 * h)
        grads.append(g)
    return grads


def autograd_grads(q, k, v, dy, eps, S_in=None, z_in=None):
    """Gradients of the pairwise form through torch autograd (float64, CPU)."""
    import torch

    t = [torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True) for a in (q, k, v)]
    N, d = t[0].shape[-2], t[0].shape[-1]
    dv = t[2].shape[-1]
    lead = t[0].shape[:-2]
    Si = (torch.zeros(lead + (d, dv), dtype=torch.float64) if S_in is None
          else torch.tensor(np.asarray(S_in, dtype=np.float64)))
    zi = (torch.zeros(lead + (d,), dtype=torch.float64) if z_in is None
          else torch.tensor(np.asarray(z_in, dtype=np.float64)))
    Si.requires_grad_(True)
    zi.requires_grad_(True)

    def phi(x):
        return torch.where(x > 0, x + 1.0, torch.exp(torch.clamp(x, max=0.0)))

    fq, fk = phi(t[0]), phi(t[1])
    mask = torch.tril(torch.ones(N, N, dtype=torch.float64))
    w = (fq @ fk.transpose(-1, -2)) * mask
    num = w @ t[2] + fq @ Si
    den = w.sum(-1) + (fq * zi.unsqueeze(-2)).sum(-1)
    y = num / den.clamp_min(eps).unsqueeze(-1)
    (y * torch.tensor(np.asarray(dy, dtype=np.float64))).sum().backward()
    return [x.grad.numpy() for x in t] + [Si.grad.numpy(), zi.grad.numpy()]


def dens(q, k, z_in=None):
    """phi(q_t)^T z_t for every token (numpy, for choosing a clamp threshold)."""
    def phi(x):
        return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))
    fq, fk = phi(np.asarray(q, np.float64)), phi(np.asarray(k, np.float64))
    z = np.cumsum(fk, axis=-2)
    if z_in is not None:
        z = z + np.asarray(z_in, np.float64)[..., None, :]
    return (fq * z).sum(-1)


def eps_between_dens(q, k, z_in=None, margin=1e-3) -> float:
    """An eps that clamps some tokens and not others, away from every den."""
    dd = np.sort(dens(q, k, z_in=z_in).reshape(-1))
    gaps = np.diff(dd)
    mid = len(dd) // 2
    order = sorted(range(len(gaps)), key=lambda i: abs(i - mid))
    for i in order:
        if gaps[i] > 2 * margin:
            return float((dd[i] + dd[i + 1]) / 2)
    raise ValueError("no gap between denominators")


def fd_decay_pin_passes(seed=5, rtol=1e-6) -> bool:
    """One small case with per-head decays and an initial state."""
    r = np.random.default_rng(seed)
    q, k = r.standard_normal((2, 2, 6, 3))
    v, dy = r.standard_normal((2, 2, 6, 2))
    S_in = r.standard_normal((2, 3, 2))
    z_in = np.abs(r.standard_normal((2, 3))) + 0.5
    gam = np.array([0.6, 0.95])
    want = finite_difference_grads(q, k, v, dy, 1e-6, S_in, z_in, gamma=gam)
    got = oracle.causal_backward(q, k, v, dy, eps=1e-6, S_in=S_in, z_in=z_in,
                                 return_state_grad=True, nthreads=1, gamma=gam)
    for g, w in zip(got, want):
        if not np.abs(g - w).max() <= rtol * max(np.abs(w).max(), 1e-12):
            return False
    return True


def fd_pin_passes(seed=3, rtol=1e-6) -> bool:
    """One small case with an initial state and a partly active clamp."""
    r = np.random.default_rng(seed)
    q, k = r.standard_normal((2, 2, 5, 3))
    v, dy = r.standard_normal((2, 2, 5, 2))
    S_in = r.standard_normal((2, 3, 2))
    z_in = np.abs(r.standard_normal((2, 3))) + 0.5
    eps = eps_between_dens(q, k, z_in=z_in)
    want = finite_difference_grads(q, k, v, dy, eps, S_in, z_in)
    got = oracle.causal_backward(q, k, v, dy, eps=eps, S_in=S_in, z_in=z_in,
                                 return_state_grad=True, nthreads=1)
    for g, w in zip(got, want):
        scale = max(np.abs(w).max(), 1e-12)
        if not np.abs(g - w).max() <= rtol * scale:
            return False
    return True
