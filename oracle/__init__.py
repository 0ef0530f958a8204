"""fp64 CPU oracle for elu(x)+1 kernelized linear attention.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python
binding) never imports this package; only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` do.  The C source
``linattn_oracle.c`` shares nothing with the CUDA sources.

Each function widens its inputs to float64 numpy arrays and calls the plain
C loops in ``linattn_oracle.c``:

* ``phi(x)``                       -- elu(x) + 1 ("Linear Attention/es",
  "Mapas de características"; "Linear Transformer", "La función ELU + 1").
* ``causal_recurrent(q, k, v)``    -- token-by-token recurrent form
  ("Linear Attention/es", "Forma recurrente e inferencia autorregresiva").
* ``noncausal(q, k, v)``           -- matrix form with S, z summed over the
  whole sequence ("Linear Attention/es", "Reformulación con núcleos").
* ``quadratic(q, k, v, causal)``   -- brute-force pairwise form (first
  equality of the same equation), O(N^2).
* ``causal_chunked(q, k, v, C)``   -- blockwise form ("Linear Attention/es",
  "Entrenamiento: forma paralela").
* ``decode_step(q, k, v, S, z)``   -- one recurrent step on a stored state.
* ``causal_recurrent_decay(q, k, v, gamma)`` -- the recurrent form with a
  per-head decay, S_t = gamma S_{t-1} + phi(k_t) v_t^T and likewise z_t
  ("Linear Attention/es", "Variantes y extensiones", RetNet).
* ``causal_backward(q, k, v, dy)`` -- gradients of sum_t dy_t . y_t of the
  causal form with respect to q, k, v (and the initial state), by the chain
  rule through the recurrence ("Linear Attention/es", "Entrenamiento: forma
  paralela" motivates it; the recurrence is "Forma recurrente ...").
* ``causal_gated(q, k, v, gate, phi)`` -- the recurrent form with a
  data-dependent gate per token (one value, or one per feature row of S) in
  place of the decay ("Variantes y extensiones", gated linear attention), and
  the feature map "elu1" or "identity" ("Mapas de características").
* ``noncausal(..., phi=)`` and ``quadratic(..., phi=)`` take the same choice
  of feature map.
* ``random_features(x, W)`` -- the positive random-feature map
  exp(W x - ||x||^2 / 2) / sqrt(m) of the same section (Performer), W given.

Shapes: q, k ``[..., N, d]``; v ``[..., N, dv]``; leading dims are flattened
into independent heads.  States: S ``[..., d, dv]``, z ``[..., d]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "linattn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liblinattn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math) into oracle/_build."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    """Declare the C signatures on a loaded oracle library."""
    P = ctypes.POINTER(ctypes.c_double)
    i, dbl = ctypes.c_int, ctypes.c_double
    lib.oracle_phi.argtypes = [P, P, ctypes.c_long]
    lib.oracle_phi.restype = None
    lib.oracle_causal_recurrent.argtypes = [P, P, P, P, i, i, i, i, dbl, P, P, P, P, i]
    lib.oracle_causal_recurrent.restype = i
    lib.oracle_noncausal.argtypes = [P, P, P, P, i, i, i, i, dbl, P, P, i]
    lib.oracle_noncausal.restype = i
    lib.oracle_quadratic.argtypes = [P, P, P, P, i, i, i, i, dbl, i, i]
    lib.oracle_quadratic.restype = i
    lib.oracle_causal_chunked.argtypes = [P, P, P, P, i, i, i, i, dbl, i, P, P, P, P, i]
    lib.oracle_causal_chunked.restype = i
    lib.oracle_decode_step.argtypes = [P, P, P, P, P, P, i, i, i, dbl, i]
    lib.oracle_decode_step.restype = i
    lib.oracle_causal_recurrent_decay.argtypes = [P, P, P, P, i, i, i, i, dbl, P, P, P, P, P, i]
    lib.oracle_causal_recurrent_decay.restype = i
    lib.oracle_causal_backward.argtypes = [P, P, P, P, P, P, P, i, i, i, i, dbl, P, P, P, P, i]
    lib.oracle_causal_backward.restype = i
    lib.oracle_causal_backward_decay.argtypes = [P, P, P, P, P, P, P, i, i, i, i, dbl, P, P, P,
                                                 P, P, i]
    lib.oracle_causal_backward_decay.restype = i
    lib.oracle_causal_gated.argtypes = [P, P, P, P, i, i, i, i, dbl, i, P, i, P, P, P, P, i]
    lib.oracle_causal_gated.restype = i
    lib.oracle_noncausal_phi.argtypes = [P, P, P, P, i, i, i, i, dbl, i, P, P, i]
    lib.oracle_noncausal_phi.restype = i
    lib.oracle_quadratic_phi.argtypes = [P, P, P, P, i, i, i, i, dbl, i, i, i]
    lib.oracle_quadratic_phi.restype = i
    lib.oracle_random_features.argtypes = [P, P, P, ctypes.c_long, i, i]
    lib.oracle_random_features.restype = i
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(x) -> np.ndarray:
    """Widen any array-like (numpy, or a CPU torch tensor via numpy()) to C-contiguous f64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _split(q, k, v):
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.shape != k.shape or q.shape[:-1] != v.shape[:-1] or q.ndim < 2:
        raise ValueError(f"bad shapes q{q.shape} k{k.shape} v{v.shape}")
    lead = q.shape[:-2]
    N, d, dv = q.shape[-2], q.shape[-1], v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    return q, k, v, lead, BH, N, d, dv


def phi(x) -> np.ndarray:
    x = _f64(x)
    out = np.empty_like(x)
    _load().oracle_phi(_ptr(x), _ptr(out), x.size)
    return out


def causal_recurrent(q, k, v, eps: float = 1e-6, S_in=None, z_in=None,
                     return_state: bool = False, nthreads: int | None = None):
    q, k, v, lead, BH, N, d, dv = _split(q, k, v)
    y = np.empty(lead + (N, dv))
    S_in = None if S_in is None else _f64(S_in).reshape(BH, d, dv)
    z_in = None if z_in is None else _f64(z_in).reshape(BH, d)
    S = np.empty(lead + (d, dv)) if return_state else None
    z = np.empty(lead + (d,)) if return_state else None
    rc = _load().oracle_causal_recurrent(_ptr(q), _ptr(k), _ptr(v), _ptr(y), BH, N, d, dv,
                                         float(eps), _ptr(S_in), _ptr(z_in), _ptr(S), _ptr(z),
                                         nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_causal_recurrent failed")
    return (y, S, z) if return_state else y


PHI_KINDS = {"elu1": 0, "identity": 1}


def noncausal(q, k, v, eps: float = 1e-6, return_state: bool = False,
              nthreads: int | None = None, phi: str = "elu1"):
    q, k, v, lead, BH, N, d, dv = _split(q, k, v)
    y = np.empty(lead + (N, dv))
    S = np.empty(lead + (d, dv)) if return_state else None
    z = np.empty(lead + (d,)) if return_state else None
    rc = _load().oracle_noncausal_phi(_ptr(q), _ptr(k), _ptr(v), _ptr(y), BH, N, d, dv,
                                      float(eps), PHI_KINDS[phi], _ptr(S), _ptr(z),
                                      nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_noncausal failed")
    return (y, S, z) if return_state else y


def quadratic(q, k, v, causal: bool = True, eps: float = 1e-6, nthreads: int | None = None,
              phi: str = "elu1"):
    q, k, v, lead, BH, N, d, dv = _split(q, k, v)
    y = np.empty(lead + (N, dv))
    rc = _load().oracle_quadratic_phi(_ptr(q), _ptr(k), _ptr(v), _ptr(y), BH, N, d, dv,
                                      float(eps), 1 if causal else 0, PHI_KINDS[phi],
                                      nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_quadratic failed")
    return y


def causal_chunked(q, k, v, chunk: int, eps: float = 1e-6, S_in=None, z_in=None,
                   return_state: bool = False, nthreads: int | None = None):
    q, k, v, lead, BH, N, d, dv = _split(q, k, v)
    y = np.empty(lead + (N, dv))
    S_in = None if S_in is None else _f64(S_in).reshape(BH, d, dv)
    z_in = None if z_in is None else _f64(z_in).reshape(BH, d)
    S = np.empty(lead + (d, dv)) if return_state else None
    z = np.empty(lead + (d,)) if return_state else None
    rc = _load().oracle_causal_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(y), BH, N, d, dv,
                                       float(eps), int(chunk), _ptr(S_in), _ptr(z_in), _ptr(S),
                                       _ptr(z), nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_causal_chunked failed")
    return (y, S, z) if return_state else y


def decode_step(q, k, v, S, z, eps: float = 1e-6, nthreads: int | None = None):
    """One decode step.  q, k: [..., d]; v: [..., dv]; S: [..., d, dv]; z: [..., d].

    Returns (y, S_new, z_new); the inputs are not modified.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    S = _f64(S).copy()
    z = _f64(z).copy()
    lead = q.shape[:-1]
    d, dv = q.shape[-1], v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    if S.shape != lead + (d, dv) or z.shape != lead + (d,):
        raise ValueError("state shape mismatch")
    y = np.empty(lead + (dv,))
    rc = _load().oracle_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(y), _ptr(S), _ptr(z),
                                    BH, d, dv, float(eps), nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_decode_step failed")
    return y, S, z


def _head_gammas(gamma, lead, BH):
    g = _f64(gamma).reshape(-1)
    if g.size != BH:
        if len(lead) >= 1 and g.size == lead[-1]:
            g = np.broadcast_to(g, lead).reshape(-1)
        else:
            raise ValueError(f"gamma has {g.size} values for {BH} heads")
    return np.ascontiguousarray(g, dtype=np.float64)


def causal_backward(q, k, v, dy, eps: float = 1e-6, S_in=None, z_in=None,
                    return_state_grad: bool = False, nthreads: int | None = None, gamma=None):
    """Gradients of L = sum_t dy_t . y_t, y the causal output of (q, k, v)
    (with the per-head decay ``gamma`` when given, as ``causal_recurrent_decay``).

    Returns (dq, dk, dv), plus (dS_in, dz_in) when ``return_state_grad``.
    """
    q, k, v, lead, BH, N, d, dv = _split(q, k, v)
    g = None if gamma is None else _head_gammas(gamma, lead, BH)
    dy = _f64(dy)
    if dy.shape != v.shape:
        raise ValueError(f"dy{dy.shape} must match v{v.shape}")
    gq, gk, gv = np.empty(q.shape), np.empty(k.shape), np.empty(v.shape)
    S_in = None if S_in is None else _f64(S_in).reshape(BH, d, dv)
    z_in = None if z_in is None else _f64(z_in).reshape(BH, d)
    gS = np.empty(lead + (d, dv)) if return_state_grad else None
    gz = np.empty(lead + (d,)) if return_state_grad else None
    rc = _load().oracle_causal_backward_decay(_ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(gq),
                                              _ptr(gk), _ptr(gv), BH, N, d, dv, float(eps),
                                              _ptr(g), _ptr(S_in), _ptr(z_in), _ptr(gS), _ptr(gz),
                                              nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_causal_backward failed")
    return (gq, gk, gv, gS, gz) if return_state_grad else (gq, gk, gv)


def causal_recurrent_decay(q, k, v, gamma, eps: float = 1e-6, S_in=None, z_in=None,
                           return_state: bool = False, nthreads: int | None = None):
    """Recurrent form with decay.  ``gamma`` has one value per head: shape [H]
    for q of shape [B, H, N, d] (broadcast over B), or one value per head of
    the flattened leading shape."""
    q, k, v, lead, BH, N, d, dv = _split(q, k, v)
    g = _head_gammas(gamma, lead, BH)
    y = np.empty(lead + (N, dv))
    S_in = None if S_in is None else _f64(S_in).reshape(BH, d, dv)
    z_in = None if z_in is None else _f64(z_in).reshape(BH, d)
    S = np.empty(lead + (d, dv)) if return_state else None
    z = np.empty(lead + (d,)) if return_state else None
    rc = _load().oracle_causal_recurrent_decay(_ptr(q), _ptr(k), _ptr(v), _ptr(y), BH, N, d, dv,
                                               float(eps), _ptr(g), _ptr(S_in), _ptr(z_in),
                                               _ptr(S), _ptr(z), nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_causal_recurrent_decay failed")
    return (y, S, z) if return_state else y


def causal_gated(q, k, v, gate=None, phi: str = "elu1", eps: float = 1e-6, S_in=None,
                 z_in=None, return_state: bool = False, nthreads: int | None = None):
    """Recurrent form with a per-token gate and a choice of feature map.

    ``gate``: None, shape [..., N] (one gate per token: S_t = g_t S_{t-1} +
    phi(k_t) v_t^T) or [..., N, d] (one per token and feature row of S); the
    leading dims are those of q.  ``phi``: "elu1" or "identity"."""
    q, k, v, lead, BH, N, d, dv = _split(q, k, v)
    g, gd = None, 1
    if gate is not None:
        g = _f64(gate)
        if g.shape == lead + (N,):
            gd = 1
        elif g.shape == lead + (N, d):
            gd = d
        else:
            raise ValueError(f"gate{g.shape} must be {lead + (N,)} or {lead + (N, d)}")
        g = np.ascontiguousarray(g.reshape(BH, N, gd))
    y = np.empty(lead + (N, dv))
    S_in = None if S_in is None else _f64(S_in).reshape(BH, d, dv)
    z_in = None if z_in is None else _f64(z_in).reshape(BH, d)
    S = np.empty(lead + (d, dv)) if return_state else None
    z = np.empty(lead + (d,)) if return_state else None
    rc = _load().oracle_causal_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(y), BH, N, d, dv,
                                     float(eps), PHI_KINDS[phi], _ptr(g), gd, _ptr(S_in),
                                     _ptr(z_in), _ptr(S), _ptr(z), nthreads or default_threads())
    if rc:
        raise RuntimeError("oracle_causal_gated failed")
    return (y, S, z) if return_state else y


def random_features(x, W) -> np.ndarray:
    """exp(W x - ||x||^2 / 2) / sqrt(m) for every row x of ``x`` ([..., d]);
    W: [m, d].  Returns [..., m]."""
    x, W = _f64(x), _f64(W)
    d = x.shape[-1]
    if W.ndim != 2 or W.shape[1] != d:
        raise ValueError(f"W{W.shape} must be [m, {d}]")
    m = W.shape[0]
    rows = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    out = np.empty(x.shape[:-1] + (m,))
    rc = _load().oracle_random_features(_ptr(x), _ptr(W), _ptr(out), rows, d, m)
    if rc:
        raise RuntimeError("oracle_random_features failed")
    return out
