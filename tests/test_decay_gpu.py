"""GPU parity of the decay entry points against the fp64 oracle.

la_forward_causal_decay and la_decode_step_decay (RetNet's update,
"Linear Attention/es", "Variantes y extensiones") on seeded inputs: every
(d, dv) pair, both input dtypes, ragged tails, per-head gamma, initial and
final state; the limits gamma = 1 (the plain form) and gamma = 0 (y = v);
decode steps continuing a decayed prefill; sampled heads of the full-size
workloads.

Two kernels compute the decayed forward.  bf16 inputs with d, dv in
{64, 128} and gamma in [2^-1/2, 1] take the tensor-core kernel (bf16 psi
operands, fp32 accumulation: the bf16 bound, as for the plain causal form);
every other head takes the fp32 CUDA-core kernel (the float32 bound for both
input dtypes).  The decode step is fp32 for both dtypes.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_rnn_sequence_gb300 import linattn as la
from linear_rnn_sequence_gb300.workloads import (WORKLOADS, head_decays, make_qkv,
                                                 next_decode_inputs, decode_step_generator,
                                                 random_qkv)
from metrics import TOL_BF16, TOL_F32, rel_max_err

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, N, d, dv, dtype, scale
    (1, 2, 256, 32, 32, torch.float32, 1.0),
    (1, 3, 333, 64, 64, torch.float32, 1.0),
    (2, 2, 517, 128, 128, torch.float32, 0.2),
    (1, 2, 1000, 64, 128, torch.float32, 0.5),
    (2, 3, 1031, 64, 64, torch.bfloat16, 0.125),
    (1, 4, 777, 128, 128, torch.bfloat16, 0.0884),
    (1, 2, 129, 128, 32, torch.bfloat16, 1.0),
    (1, 2, 385, 32, 128, torch.bfloat16, 1.0),
]


def tol_decay(dt, d, dv, gamma) -> float:
    """The bound of the kernel that computes a head with this decay."""
    tc = (dt == torch.bfloat16 and d in (64, 128) and dv in (64, 128)
          and 2 ** -0.5 <= float(gamma) <= 1.0)
    return TOL_BF16 if tc else TOL_F32


def _ids(c):
    B, H, N, d, dv, dt, s = c
    return f"B{B}H{H}N{N}d{d}dv{dv}{'bf16' if dt == torch.bfloat16 else 'f32'}"


@pytest.mark.parametrize("with_state", [False, True])
@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_causal_decay_matches_oracle(case, with_state, cuda_device):
    B, H, N, d, dv, dt, s = case
    q, k, v = random_qkv(B, H, N, d, dv, dtype=dt, scale=s, seed=N + 9)
    gam = head_decays(H)
    S_in = z_in = None
    if with_state:
        qp, kp, vp = random_qkv(B, H, 40, d, dv, dtype=dt, scale=0.5, seed=N)
        _, S_in, z_in = oracle.causal_recurrent_decay(qp, kp, vp, gam, return_state=True)
    dev = lambda t: None if t is None else torch.as_tensor(t, dtype=torch.float32).to(cuda_device)
    y, S, z = la.forward_causal_decay(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                      gam.to(cuda_device), S_in=dev(S_in), z_in=dev(z_in),
                                      return_state=True)
    torch.cuda.synchronize()
    yo, So, zo = oracle.causal_recurrent_decay(q, k, v, gam, S_in=S_in, z_in=z_in,
                                               return_state=True)
    tol = max(tol_decay(dt, d, dv, g) for g in gam)
    for name, g, w in (("y", y, yo), ("S", S, So), ("z", z, zo)):
        err = rel_max_err(g, w)
        assert err <= tol, f"{name}: {err:.3e}"


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (64, 128)])
def test_causal_decay_routes_each_head(d, dv, cuda_device):
    """One call with decays on both sides of 2^-1/2 (and the limits 0, 1):
    each head matches the oracle within its own kernel's bound, with an
    initial and a final state and a ragged last block."""
    B, H, N = 2, 8, 389
    gam = torch.tensor([0.0, 0.3, 0.7071, 0.70711, 0.75, 0.9, 0.999, 1.0])
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.bfloat16, scale=d ** -0.5, seed=d + dv)
    qp, kp, vp = random_qkv(B, H, 50, d, dv, dtype=torch.bfloat16, scale=0.3, seed=3)
    _, S_in, z_in = oracle.causal_recurrent_decay(qp, kp, vp, gam, return_state=True)
    dev = lambda t: torch.as_tensor(t, dtype=torch.float32).to(cuda_device)
    y, S, z = la.forward_causal_decay(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                      gam.to(cuda_device), S_in=dev(S_in), z_in=dev(z_in),
                                      return_state=True, check_status=True)
    torch.cuda.synchronize()
    yo, So, zo = oracle.causal_recurrent_decay(q, k, v, gam, S_in=S_in, z_in=z_in,
                                               return_state=True)
    for h in range(H):
        tol = tol_decay(torch.bfloat16, d, dv, gam[h])
        for name, g, w in (("y", y[:, h], yo[:, h]), ("S", S[:, h], So[:, h]),
                           ("z", z[:, h], zo[:, h])):
            err = rel_max_err(g, w)
            assert err <= tol, f"head {h} (gamma {float(gam[h])}) {name}: {err:.3e}"


def test_causal_decay_long_sequence_state(cuda_device):
    """33 blocks with an initial state: the tensor-core kernel restarts its
    state scale every block (gamma 0.72), every few blocks (0.9, 0.97) or
    never (0.9995); y on whole heads, and the final S and z, against the
    oracle."""
    B, H, N, d, dv = 1, 4, 4099, 64, 128
    gam = torch.tensor([0.72, 0.9, 0.97, 0.9995])
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.bfloat16, scale=d ** -0.5, seed=41)
    qp, kp, vp = random_qkv(B, H, 64, d, dv, dtype=torch.bfloat16, scale=0.3, seed=42)
    _, S_in, z_in = oracle.causal_recurrent_decay(qp, kp, vp, gam, return_state=True)
    dev = lambda t: torch.as_tensor(t, dtype=torch.float32).to(cuda_device)
    y, S, z = la.forward_causal_decay(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                      gam.to(cuda_device), S_in=dev(S_in), z_in=dev(z_in),
                                      return_state=True, check_status=True)
    torch.cuda.synchronize()
    yo, So, zo = oracle.causal_recurrent_decay(q, k, v, gam, S_in=S_in, z_in=z_in,
                                               return_state=True)
    for h in range(H):
        for name, g, w in (("y", y[:, h], yo[:, h]), ("S", S[:, h], So[:, h]),
                           ("z", z[:, h], zo[:, h])):
            err = rel_max_err(g, w)
            assert err <= TOL_BF16, f"head {h} (gamma {float(gam[h])}) {name}: {err:.3e}"


@pytest.mark.parametrize("B,H,N,d,dv,gammas", [
    (1, 2, 20000, 64, 64, (0.72, 0.99)),            # 157 segments of one block each
    (1, 3, 5000, 128, 64, (0.9, 0.999, 1.0)),
    (2, 2, 3333, 64, 128, (0.97, 0.9995)),
])
def test_causal_decay_split_sequence(B, H, N, d, dv, gammas, cuda_device):
    """Few heads: the sequence is cut into segments, whose decayed states
    and decayed prefixes seed the chunk kernel.  Whole heads against the
    oracle, with an initial and a final state."""
    gam = torch.tensor(gammas)
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.bfloat16, scale=d ** -0.5, seed=N)
    qp, kp, vp = random_qkv(B, H, 64, d, dv, dtype=torch.bfloat16, scale=0.3, seed=7)
    _, S_in, z_in = oracle.causal_recurrent_decay(qp, kp, vp, gam, return_state=True)
    dev = lambda t: torch.as_tensor(t, dtype=torch.float32).to(cuda_device)
    assert la.causal_workspace_bytes(B, H, N, d, dv) > 256   # segment states: split
    y, S, z = la.forward_causal_decay(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                      gam.to(cuda_device), S_in=dev(S_in), z_in=dev(z_in),
                                      return_state=True, check_status=True)
    torch.cuda.synchronize()
    yo, So, zo = oracle.causal_recurrent_decay(q, k, v, gam, S_in=S_in, z_in=z_in,
                                               return_state=True)
    for h in range(H):
        for name, g, w in (("y", y[:, h], yo[:, h]), ("S", S[:, h], So[:, h]),
                           ("z", z[:, h], zo[:, h])):
            err = rel_max_err(g, w)
            assert err <= TOL_BF16, f"head {h} (gamma {float(gam[h])}) {name}: {err:.3e}"


def test_causal_decay_long_workload_sampled_heads(cuda_device):
    """Full-size long-context shape with decay (B1 H32 N131072 d64, split into
    segments): whole heads against the oracle."""
    w = WORKLOADS["causal_decay_bf16_b1h32n131072d64"]
    q, k, v = make_qkv(w, device=cuda_device, gen_device=cuda_device)
    gam = head_decays(w.H)
    y = la.forward_causal_decay(q, k, v, gam.to(cuda_device), check_status=True)
    torch.cuda.synchronize()
    for h in (0, 13, 31):
        yo = oracle.causal_recurrent_decay(q[0, h][None].cpu(), k[0, h][None].cpu(),
                                           v[0, h][None].cpu(), gam[h:h + 1])
        assert rel_max_err(y[0, h], yo[0]) <= tol_decay(w.dtype, w.d, w.dv, gam[h])


def test_causal_decay_gamma_one_is_the_plain_kernel(cuda_device):
    """gamma = 1 on the tensor cores: every key weight is 1 and every
    rescaling factor is 1 exactly, so the output and final state equal the
    plain causal kernel's bit for bit (96 heads: neither call splits the
    sequence)."""
    B, H, N, d, dv = 4, 24, 300, 64, 128
    q, k, v = (t.to(cuda_device) for t in random_qkv(B, H, N, d, dv, dtype=torch.bfloat16,
                                                     scale=0.125, seed=12))
    y1, S1, z1 = la.forward_causal_decay(q, k, v, torch.ones(H, device=cuda_device),
                                         return_state=True)
    y0, S0, z0 = la.forward_causal(q, k, v, return_state=True)
    torch.cuda.synchronize()
    assert torch.equal(y1, y0) and torch.equal(S1, S0) and torch.equal(z1, z0)


def test_decay_limits(cuda_device):
    """gamma = 1 is the plain causal form; gamma = 0 returns v."""
    q, k, v = random_qkv(2, 3, 300, 64, 64, dtype=torch.bfloat16, scale=0.125, seed=2)
    qd, kd, vd = (t.to(cuda_device) for t in (q, k, v))
    y1 = la.forward_causal_decay(qd, kd, vd, torch.ones(3, device=cuda_device))
    y0 = la.forward_causal_decay(qd, kd, vd, torch.zeros(3, device=cuda_device))
    torch.cuda.synchronize()
    # gamma = 1: tensor cores (bf16 bound); gamma = 0: CUDA cores, exact
    assert rel_max_err(y1, oracle.causal_recurrent(q, k, v)) <= TOL_BF16
    assert rel_max_err(y0, v.double().numpy()) <= 1e-6


@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 256, 257])
def test_causal_decay_edge_lengths(N, cuda_device):
    """Block edges on the tensor cores: a single token, a block exactly full,
    one token into the next block; with an initial and a final state."""
    B, H, d, dv = 1, 3, 64, 128
    gam = torch.tensor([0.75, 0.97, 1.0])
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.bfloat16, scale=0.3, seed=50 + N)
    qp, kp, vp = random_qkv(B, H, 20, d, dv, dtype=torch.bfloat16, scale=0.3, seed=9)
    _, S_in, z_in = oracle.causal_recurrent_decay(qp, kp, vp, gam, return_state=True)
    dev = lambda t: torch.as_tensor(t, dtype=torch.float32).to(cuda_device)
    y, S, z = la.forward_causal_decay(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                      gam.to(cuda_device), S_in=dev(S_in), z_in=dev(z_in),
                                      return_state=True, check_status=True)
    torch.cuda.synchronize()
    yo, So, zo = oracle.causal_recurrent_decay(q, k, v, gam, S_in=S_in, z_in=z_in,
                                               return_state=True)
    for name, g, w in (("y", y, yo), ("S", S, So), ("z", z, zo)):
        err = rel_max_err(g, w)
        assert err <= TOL_BF16, f"{name}: {err:.3e}"


def test_decay_empty_sequence_copies_state(cuda_device):
    S_in = torch.randn(1, 2, 64, 64, device=cuda_device)
    z_in = torch.rand(1, 2, 64, device=cuda_device) + 1
    q = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device=cuda_device)
    y, S, z = la.forward_causal_decay(q, q, q, head_decays(2).to(cuda_device), S_in=S_in,
                                      z_in=z_in, return_state=True)
    torch.cuda.synchronize()
    assert torch.equal(S, S_in) and torch.equal(z, z_in)


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d,dv", [(32, 32), (64, 128), (128, 128), (128, 64)])
def test_decode_decay_steps_match_oracle(dt, d, dv, cuda_device):
    B, H, Np, steps = 2, 3, 100, 20
    gam = head_decays(H)
    q, k, v = random_qkv(B, H, Np, d, dv, dtype=dt, scale=0.5, seed=7)
    _, So, zo = oracle.causal_recurrent_decay(q, k, v, gam, return_state=True)
    S = torch.tensor(So, dtype=torch.float32, device=cuda_device)
    z = torch.tensor(zo, dtype=torch.float32, device=cuda_device)
    Sref, zref = So, zo
    g = torch.Generator().manual_seed(11)
    for _ in range(steps):
        qs, ks, vs = ((torch.randn(B, H, n, generator=g) * 0.3).to(dt) for n in (d, d, dv))
        y = la.decode_step_decay(qs.to(cuda_device), ks.to(cuda_device), vs.to(cuda_device), S, z,
                                 gam.to(cuda_device))
        yo, Sref, zref = oracle.causal_recurrent_decay(qs[:, :, None], ks[:, :, None],
                                                       vs[:, :, None], gam, S_in=Sref, z_in=zref,
                                                       return_state=True)
        torch.cuda.synchronize()
        assert rel_max_err(y, yo[:, :, 0]) <= TOL_F32
    assert rel_max_err(S, Sref) <= TOL_F32
    assert rel_max_err(z, zref) <= TOL_F32


def test_causal_decay_workload_sampled_heads(cuda_device):
    """Full-size prefill shape; whole heads checked against the oracle."""
    w = WORKLOADS["causal_decay_bf16_b8h16n8192d128"]
    q, k, v = make_qkv(w)
    gam = head_decays(w.H)
    y = la.forward_causal_decay(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                gam.to(cuda_device))
    torch.cuda.synchronize()
    for b, h in ((0, 0), (3, 7), (7, 15)):
        yo = oracle.causal_recurrent_decay(q[b, h][None], k[b, h][None], v[b, h][None],
                                           gam[h:h + 1])
        assert rel_max_err(y[b, h], yo[0]) <= tol_decay(w.dtype, w.d, w.dv, gam[h])


def test_decode_decay_workload_steps(cuda_device):
    """Decode shape B256 H32 d128: 1024-token decayed prefill (tensor cores),
    then 16 fp32 steps, each step's output and the final state checked on
    sampled heads (the bf16 bound: the state comes from the prefill)."""
    w = WORKLOADS["decode_decay_bf16_b256h32d128"]
    q, k, v = make_qkv(w, device=cuda_device, gen_device=cuda_device)
    gam = head_decays(w.H).to(cuda_device)
    _, S, z = la.forward_causal_decay(q, k, v, gam, return_state=True)
    heads = [(0, 0), (100, 17), (255, 31)]
    sel = lambda t: torch.stack([t[b, h] for b, h in heads]).cpu()
    g32 = head_decays(w.H)
    gsel = torch.stack([g32[h] for _, h in heads])
    _, Sref, zref = oracle.causal_recurrent_decay(sel(q), sel(k), sel(v), gsel, return_state=True)
    gen = decode_step_generator(w, gen_device=cuda_device)
    for _ in range(16):
        qs, ks, vs = next_decode_inputs(w, gen)
        y = la.decode_step_decay(qs, ks, vs, S, z, gam)
        yo, Sref, zref = oracle.causal_recurrent_decay(sel(qs)[:, None], sel(ks)[:, None],
                                                       sel(vs)[:, None], gsel, S_in=Sref,
                                                       z_in=zref, return_state=True)
        torch.cuda.synchronize()
        assert rel_max_err(sel(y), yo[:, 0]) <= TOL_BF16
    assert rel_max_err(sel(S), Sref) <= TOL_BF16


def test_decay_outputs_stay_in_bounds(cuda_device):
    """Canary-padded y, S, z for the decayed forward and decode step."""
    B, H, N, d, dv = 1, 2, 130, 64, 64
    q, k, v = (t.to(cuda_device) for t in random_qkv(B, H, N, d, dv, dtype=torch.bfloat16,
                                                     scale=0.2, seed=5))
    gam = head_decays(H).to(cuda_device)
    pad = 4096
    ybuf = torch.full((B * H * N * dv + pad,), 12345.0, device=cuda_device)
    Sbuf = torch.full((B * H * d * dv + pad,), 12345.0, device=cuda_device)
    zbuf = torch.full((B * H * d + pad,), 12345.0, device=cuda_device)
    y = ybuf[: B * H * N * dv].view(B, H, N, dv)
    S = Sbuf[: B * H * d * dv].view(B, H, d, dv)
    z = zbuf[: B * H * d].view(B, H, d)
    la.forward_causal_decay(q, k, v, gam, out=y, S_out=S, z_out=z, return_state=True)
    yd = ybuf[: B * H * dv].view(B, H, dv)
    la.decode_step_decay(q[:, :, 0].contiguous(), k[:, :, 0].contiguous(),
                         v[:, :, 0].contiguous(), S, z, gam, out=yd)
    torch.cuda.synchronize()
    for buf in (ybuf, Sbuf, zbuf):
        assert (buf[-pad:] == 12345.0).all()
