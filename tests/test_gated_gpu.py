"""GPU parity of the gated recurrence and the feature-map swaps against the
fp64 oracle ("Linear Attention/es", "Variantes y extensiones": gated linear
attention; "Mapas de características": identity and random-feature maps).

la_decode_step_gated and la_forward_noncausal_phi with the identity map run in
float32 on the CUDA cores for both input dtypes (bf16 inputs are exact in
float32), so the float32 bound, 1e-4 of RMS, applies to them, and to
la_forward_causal_gated wherever it runs on the CUDA cores.  With bf16 inputs,
d and dv in {64, 128}, one gate per token and elu + 1, la_forward_causal_gated
runs on the tensor cores (tests/test_gated_tc_gpu.py), and the bf16 bound,
2e-2 of RMS, applies.  The
identity map's denominator can cross zero; those cases draw q and k around
+1.5 so that it stays away from the clamp, except the clamp case itself.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_rnn_sequence_gb300 import linattn as la
from linear_rnn_sequence_gb300.workloads import (WORKLOADS, head_decays, make_gated_inputs,
                                                 random_gated, random_projection, random_qkv)
from metrics import TOL_BF16, TOL_F32, rel_max_err

pytestmark = pytest.mark.gpu


def gated_tol(dt, d, dv, gate_dim, phi, gated=True):
    """The bound of the path la_forward_causal_gated takes for these arguments."""
    tc = (dt == torch.bfloat16 and d in (64, 128) and dv in (64, 128) and gate_dim == 1
          and phi == "elu1" and gated)
    return TOL_BF16 if tc else TOL_F32


def _check(got, want, tol=TOL_F32, what=""):
    for name, g, w in zip(("y", "S", "z"), got, want):
        err = rel_max_err(g, w)
        assert err <= tol, f"{what} {name}: {err:.3e}"


CASES = [
    # B, H, N, d, dv, dtype
    (1, 2, 300, 32, 32, torch.float32),
    (2, 2, 517, 64, 64, torch.bfloat16),
    (1, 3, 257, 128, 128, torch.float32),
    (1, 2, 1000, 64, 128, torch.bfloat16),
    (1, 2, 129, 128, 64, torch.float32),
]


def _ids(c):
    B, H, N, d, dv, dt = c
    return f"B{B}H{H}N{N}d{d}dv{dv}{'bf16' if dt == torch.bfloat16 else 'f32'}"


@pytest.mark.parametrize("phi", ["elu1", "identity"])
@pytest.mark.parametrize("gate_dim", ["none", "token", "feature"])
@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_causal_gated_matches_oracle(case, gate_dim, phi, cuda_device):
    B, H, N, d, dv, dt = case
    gd = {"none": 1, "token": 1, "feature": d}[gate_dim]
    shift = 1.5 if phi == "identity" else 0.0
    q, k, v, g = random_gated(B, H, N, d, dv, gd, dtype=dt, scale=d ** -0.5 if phi == "elu1" else 0.5,
                              seed=N + d, shift=shift)
    if gate_dim == "none":
        g = None
    gen = torch.Generator().manual_seed(N)
    S_in = torch.randn(B, H, d, dv, generator=gen) * 0.5
    z_in = torch.rand(B, H, d, generator=gen) * 5 + 1
    dev = lambda t: None if t is None else t.to(cuda_device)
    y, S, z = la.forward_causal_gated(dev(q), dev(k), dev(v), gate=dev(g), phi=phi,
                                      S_in=dev(S_in), z_in=dev(z_in), return_state=True)
    torch.cuda.synchronize()
    want = oracle.causal_gated(q, k, v, gate=g, phi=phi, S_in=S_in, z_in=z_in, return_state=True)
    _check((y, S, z), want, tol=gated_tol(dt, d, dv, gd, phi, g is not None),
           what=f"{gate_dim} {phi}")


def test_gated_with_constant_gates_equals_decay(cuda_device):
    """Gates equal to a head's gamma at every token reproduce the per-head decay."""
    B, H, N, d, dv = 1, 4, 700, 64, 64
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.float32, scale=0.125, seed=3)
    gam = torch.tensor([0.3, 0.7, 0.95, 1.0])
    g = gam[None, :, None].expand(B, H, N).contiguous()
    y = la.forward_causal_gated(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                gate=g.to(cuda_device))
    torch.cuda.synchronize()
    assert rel_max_err(y, oracle.causal_recurrent_decay(q, k, v, gam)) <= TOL_F32


def test_closed_gate_restarts_the_state(cuda_device):
    q, k, v, g = random_gated(1, 2, 200, 64, 64, 1, dtype=torch.bfloat16, scale=0.125, seed=4)
    g[:, :, [0, 50, 127, 128, 199]] = 0.0
    y = la.forward_causal_gated(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                gate=g.to(cuda_device))
    torch.cuda.synchronize()
    for t in (50, 127, 128, 199):
        assert torch.allclose(y[:, :, t].cpu(), v[:, :, t].float(), rtol=1e-5, atol=1e-6)
    assert rel_max_err(y, oracle.causal_gated(q, k, v, gate=g)) <= TOL_F32


def test_identity_map_clamp(cuda_device):
    """phi(x) = x with inputs of both signs: some denominators are negative or
    near zero and the clamp max(den, eps) decides them, on both sides alike."""
    q, k, v = random_qkv(1, 2, 150, 32, 32, dtype=torch.float32, scale=1.0, seed=5)
    eps = 0.5
    y = la.forward_causal_gated(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                phi="identity", eps=eps)
    torch.cuda.synchronize()
    want = oracle.causal_gated(q, k, v, phi="identity", eps=eps)
    assert rel_max_err(y, want) <= TOL_F32


@pytest.mark.parametrize("gate_dim", [1, 64])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_gated_decode_steps(gate_dim, dt, cuda_device):
    B, H, Np, d, dv = 2, 3, 60, 64, 64
    q, k, v, g = random_gated(B, H, Np, d, dv, gate_dim, dtype=dt, scale=0.3, seed=6)
    _, So, zo = oracle.causal_gated(q, k, v, gate=g, return_state=True)
    S = torch.tensor(So, dtype=torch.float32, device=cuda_device)
    z = torch.tensor(zo, dtype=torch.float32, device=cuda_device)
    gen = torch.Generator().manual_seed(7)
    for t in range(8):
        qs, ks, vs = ((torch.randn(B, H, n, generator=gen) * 0.3).to(dt) for n in (d, d, dv))
        gs = 1.0 - torch.rand((B, H) if gate_dim == 1 else (B, H, d), generator=gen) * 0.3
        y = la.decode_step_gated(qs.to(cuda_device), ks.to(cuda_device), vs.to(cuda_device), S, z,
                                 gate=gs.to(cuda_device))
        yo, So, zo = oracle.causal_gated(qs[:, :, None], ks[:, :, None], vs[:, :, None],
                                         gate=gs[:, :, None], S_in=So, z_in=zo, return_state=True)
        torch.cuda.synchronize()
        assert rel_max_err(y, yo[:, :, 0]) <= TOL_F32, f"step {t}"
    assert rel_max_err(S, So) <= TOL_F32 and rel_max_err(z, zo) <= TOL_F32


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_identity_decode_steps(dt, cuda_device):
    B, H, d, dv = 2, 2, 32, 64
    gen = torch.Generator().manual_seed(8)
    So = np.abs(np.random.default_rng(1).standard_normal((B, H, d, dv)))
    zo = np.random.default_rng(2).uniform(5, 10, (B, H, d))
    S = torch.tensor(So, dtype=torch.float32, device=cuda_device)
    z = torch.tensor(zo, dtype=torch.float32, device=cuda_device)
    for t in range(4):
        qs, ks = ((torch.rand(B, H, d, generator=gen) + 0.5).to(dt) for _ in range(2))
        vs = torch.randn(B, H, dv, generator=gen).to(dt)
        y = la.decode_step_gated(qs.to(cuda_device), ks.to(cuda_device), vs.to(cuda_device), S, z,
                                 phi="identity")
        yo, So, zo = oracle.causal_gated(qs[:, :, None], ks[:, :, None], vs[:, :, None],
                                         phi="identity", S_in=So, z_in=zo, return_state=True)
        torch.cuda.synchronize()
        assert rel_max_err(y, yo[:, :, 0]) <= TOL_F32


@pytest.mark.parametrize("B,H,N,d,dv,dt", [(1, 3, 1000, 64, 64, torch.bfloat16),
                                           (2, 2, 333, 128, 32, torch.float32)])
def test_noncausal_identity_map(B, H, N, d, dv, dt, cuda_device):
    q, k, v = random_qkv(B, H, N, d, dv, dtype=dt, scale=0.5, seed=N, shift=1.5)
    y, S, z = la.forward_noncausal_phi(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                       phi="identity", return_state=True)
    torch.cuda.synchronize()
    _check((y, S, z), oracle.noncausal(q, k, v, phi="identity", return_state=True))
    # elu + 1 through the same entry point is la_forward_noncausal
    y1 = la.forward_noncausal_phi(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                  phi="elu1")
    torch.cuda.synchronize()
    assert rel_max_err(y1, oracle.noncausal(q, k, v)) <= (TOL_F32 if dt == torch.float32 else 2e-2)


@pytest.mark.parametrize("m,d,dt", [(64, 64, torch.bfloat16), (128, 32, torch.float32),
                                    (32, 128, torch.float32), (200, 16, torch.float32)])
def test_random_features_match_oracle(m, d, dt, cuda_device):
    x = (torch.randn(3, 2, 77, d, generator=torch.Generator().manual_seed(m)) * d ** -0.5).to(dt)
    W = random_projection(m, d, seed=d)
    f = la.random_features(x.to(cuda_device), W.to(cuda_device))
    torch.cuda.synchronize()
    want = oracle.random_features(x, W)
    assert f.shape == want.shape
    np.testing.assert_allclose(f.cpu().double().numpy(), want, rtol=1e-5, atol=0)


def test_random_feature_attention_end_to_end(cuda_device):
    """Random features of q and k, then the identity-map causal attention on
    them: the kernels' result matches the oracle's on the oracle's features."""
    B, H, N, d, dv, m = 1, 2, 400, 64, 64, 128
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.float32, scale=0.125, seed=9)
    W = random_projection(m, d, seed=10)
    fq = la.random_features(q.to(cuda_device), W.to(cuda_device))
    fk = la.random_features(k.to(cuda_device), W.to(cuda_device))
    y = la.forward_causal_gated(fq, fk, v.to(cuda_device), phi="identity")
    torch.cuda.synchronize()
    Fq, Fk = oracle.random_features(q, W), oracle.random_features(k, W)
    assert rel_max_err(y, oracle.causal_gated(Fq, Fk, v, phi="identity")) <= TOL_F32


def test_gated_workload_sampled_heads(cuda_device):
    """The gated training-shape workload in the launch configuration the
    benchmark times (its gates lie in [3/4, 1): every head on the tensor
    cores); whole heads checked (heads are independent)."""
    w = WORKLOADS["causal_gated_bf16_b8h16n8192d128"]
    q, k, v, g = make_gated_inputs(w)
    y = la.forward_causal_gated(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                gate=g.to(cuda_device))
    torch.cuda.synchronize()
    flat = lambda t: t.reshape(w.BH, w.N, *t.shape[3:])
    for h in (0, 77, 127):
        want = oracle.causal_gated(flat(q)[h], flat(k)[h], flat(v)[h], gate=flat(g)[h])
        assert rel_max_err(flat(y)[h], want) <= TOL_BF16, f"head {h}"   # tensor cores


def test_gated_empty_sequence_copies_state(cuda_device):
    q = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device=cuda_device)
    S_in = torch.randn(1, 2, 64, 64, device=cuda_device)
    z_in = torch.rand(1, 2, 64, device=cuda_device)
    y, S, z = la.forward_causal_gated(q, q, q, S_in=S_in, z_in=z_in, return_state=True)
    torch.cuda.synchronize()
    assert y.shape == (1, 2, 0, 64) and torch.equal(S, S_in) and torch.equal(z, z_in)
