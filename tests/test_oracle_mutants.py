"""Plant plausible mistakes in the oracle (CPU only) and check a pin catches each.

Each mutant is a textual edit of a copy of ``oracle/linattn_oracle.c``,
compiled to a temporary library and swapped in for the real one.  The pins
run here are the hand-derived golden cases, the numpy brute force and the
chunked-vs-recurrent agreement from ``test_oracle.py``, and, for the
gradients, central differences of the forward (``backward_pins.py``).
"""
import ctypes
import json
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests import backward_pins

HERE = os.path.dirname(__file__)
SRC = os.path.join(os.path.dirname(HERE), "oracle", "linattn_oracle.c")

MUTANTS = {
    "phi_drops_plus_one": ("x > 0.0 ? x + 1.0 : exp(x)", "x > 0.0 ? x : exp(x)"),
    "phi_exp_branch_minus_one": ("x > 0.0 ? x + 1.0 : exp(x)", "x > 0.0 ? x + 1.0 : exp(x) - 1.0"),
    "eps_added_not_clamped": ("return den < eps ? eps : den;", "return den + eps;"),
    "recurrent_wrong_v_index": ("S[(long)a * dv + b] += fk[a] * v[(long)t * dv + b];",
                                "S[(long)a * dv + b] += fk[a] * v[(long)t * dv + 0];"),
    "recurrent_z_counts_tokens": ("            z[a] += fk[a];\n        }\n        for (int a = 0; a < d; ++a) fq[a]",
                                  "            z[a] += 1.0;\n        }\n        for (int a = 0; a < d; ++a) fq[a]"),
    "chunked_strict_mask": ("for (int j = 0; j <= i; ++j) {", "for (int j = 0; j < i; ++j) {"),
    "quadratic_exclusive": ("const int jmax = J->causal ? i : N - 1;", "const int jmax = J->causal ? i - 1 : N - 1;"),
    "noncausal_transposed_state": ("for (int a = 0; a < d; ++a) num += f[a] * S[(long)a * dv + b];",
                                   "for (int a = 0; a < d; ++a) num += f[a] * S[(long)b * dv + a];"),
    # gradients of the causal form
    "bwd_den_term_dropped": ("e[t] = den >= J->eps ? -dyy / D : 0.0;", "e[t] = 0.0;"),
    "bwd_clamp_passes_gradient": ("e[t] = den >= J->eps ? -dyy / D : 0.0;", "e[t] = -dyy / D;"),
    "bwd_dphi_is_one": ("return x > 0.0 ? 1.0 : exp(x);", "return x > 0.0 ? 1.0 : 1.0;"),
    "bwd_g_not_divided": ("g[(long)t * dv + b] = dy[(long)t * dv + b] / D;",
                          "g[(long)t * dv + b] = dy[(long)t * dv + b];"),
    "bwd_zh_dropped_from_dk": ("double s = z[a];", "double s = 0.0;"),
    "bwd_dv_uses_phi_q": ("s += S[(long)a * dv + b] * fk[a];", "s += S[(long)a * dv + b] * fq[a];"),
    "bwd_state_grad_not_reset": ("memset(S, 0, sizeof(double) * d * dv);", ";"),
    # decay
    "decay_skips_z": ("                z[a] *= g;\n", ""),
    "decay_squared_on_S": ("for (int b = 0; b < dv; ++b) S[(long)a * dv + b] *= g;",
                           "for (int b = 0; b < dv; ++b) S[(long)a * dv + b] *= g * g;"),
    "bwd_decay_state_grad_unscaled": ("J->dS_in[(long)h * d * dv + i] = gam * S[i];",
                                      "J->dS_in[(long)h * d * dv + i] = S[i];"),
    # gate and feature maps
    "gate_skips_z": ("                const double g = gt[J->gate_dim == 1 ? 0 : a];\n                for (int b = 0; b < dv; ++b) S[(long)a * dv + b] *= g;\n                z[a] *= g;",
                     "                const double g = gt[J->gate_dim == 1 ? 0 : a];\n                for (int b = 0; b < dv; ++b) S[(long)a * dv + b] *= g;"),
    "gate_first_feature_only": ("const double g = gt[J->gate_dim == 1 ? 0 : a];", "const double g = gt[0];"),
    "gate_previous_token": ("const double *gt = J->gate + ((long)h * N + t) * J->gate_dim;",
                            "const double *gt = J->gate + ((long)h * N + (t > 0 ? t - 1 : 0)) * J->gate_dim;"),
    "identity_map_is_elu": ("return kind == 1 ? x : phi(x);", "return phi(x);"),
    "random_features_no_norm_term": ("scale * exp(wx - 0.5 * nrm)", "scale * exp(wx)"),
    "random_features_scale_1_over_m": ("1.0 / sqrt((double)m)", "1.0 / (double)m"),
    "bwd_decay_skips_reverse_z": ("                z[a] *= gam;\n            }\n        for (int a = 0; a < d; ++a) {\n            for (int b = 0; b < dv; ++b) S[(long)a * dv + b] += fq[a]",
                                  "            }\n        for (int a = 0; a < d; ++a) {\n            for (int b = 0; b < dv; ++b) S[(long)a * dv + b] += fq[a]"),
}


def _phi_np(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _brute(q, k, v, causal):
    fq, fk = _phi_np(q), _phi_np(k)
    N = q.shape[0]
    y = np.zeros((N, v.shape[1]))
    for i in range(N):
        j = i + 1 if causal else N
        w = fk[:j] @ fq[i]
        y[i] = (w @ v[:j]) / max(w.sum(), 1e-6)
    return y


def _pins_pass() -> bool:
    """True if every pin passes with the currently loaded oracle."""
    with open(os.path.join(HERE, "golden", "hand_examples.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q, k, v = (np.array(c[x], dtype=np.float64) for x in ("q", "k", "v"))
        want = np.array(c["y"])
        if c["mode"] == "causal":
            outs = [oracle.causal_recurrent(q, k, v, eps=c["eps"]),
                    oracle.quadratic(q, k, v, True, eps=c["eps"]),
                    oracle.causal_chunked(q, k, v, 2, eps=c["eps"])]
        else:
            outs = [oracle.noncausal(q, k, v, eps=c["eps"]),
                    oracle.quadratic(q, k, v, False, eps=c["eps"])]
        for y in outs:
            if not np.allclose(y, want, rtol=1e-12, atol=1e-300):
                return False
    r = np.random.default_rng(5)
    q, k, v = (r.standard_normal((40, n)) for n in (4, 4, 3))
    if not np.allclose(oracle.causal_recurrent(q, k, v), _brute(q, k, v, True), rtol=1e-11):
        return False
    if not np.allclose(oracle.noncausal(q, k, v), _brute(q, k, v, False), rtol=1e-11):
        return False
    if not np.allclose(oracle.quadratic(q, k, v, True), _brute(q, k, v, True), rtol=1e-11):
        return False
    if not np.allclose(oracle.causal_chunked(q, k, v, 7), oracle.causal_recurrent(q, k, v),
                       rtol=1e-11):
        return False
    # gradients: central differences of the forward, with an initial state
    # and a clamp that is active for some tokens only
    if not (backward_pins.fd_pin_passes(seed=3) and backward_pins.fd_pin_passes(seed=4)):
        return False
    if not backward_pins.fd_decay_pin_passes(seed=5):
        return False
    # decay: the pairwise form with gamma^(t-j) weights
    from tests.test_oracle_decay import brute_decay
    for gam in (0.5, 0.9):
        if not np.allclose(oracle.causal_recurrent_decay(q, k, v, [gam]),
                           brute_decay(q, k, v, gam), rtol=1e-11):
            return False
    # gates and feature maps: hand examples, the closed form with products of
    # gates (both gate shapes, both maps), the random features' closed form
    from tests import gated_pins
    with open(os.path.join(HERE, "golden", "gated_examples.json")) as f:
        for c in json.load(f)["cases"]:
            y = oracle.causal_gated(*(np.array(c[x], dtype=np.float64) for x in ("q", "k", "v")),
                                    gate=np.array(c["gate"]), phi=c["phi"], eps=c["eps"])
            if not np.allclose(y, np.array(c["y"]), rtol=1e-12):
                return False
    r = np.random.default_rng(6)
    qg, kg = (np.abs(r.standard_normal((25, 3))) + 0.1 for _ in range(2))
    vg = r.standard_normal((25, 2))
    for kind in ("elu1", "identity"):
        for shape in ((25,), (25, 3)):
            g = r.uniform(0.1, 1.0, shape)
            if not np.allclose(oracle.causal_gated(qg, kg, vg, gate=g, phi=kind),
                               gated_pins.brute_gated(qg, kg, vg, g, kind), rtol=1e-11):
                return False
    W = r.standard_normal((16, 3))
    if not np.allclose(oracle.random_features(qg, W), gated_pins.random_features_np(qg, W),
                       rtol=1e-12):
        return False
    return True


def test_unmutated_oracle_passes_pins():
    assert _pins_pass()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new, 1)
    c = tmp_path / "mut.c"
    so = tmp_path / "libmut.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", str(c), "-o",
                    str(so), "-lm"], check=True)
    saved = oracle._lib
    oracle._lib = oracle._bind(ctypes.CDLL(str(so)))
    try:
        assert not _pins_pass(), f"mutant {name} survived every pin"
    finally:
        oracle._lib = saved
