"""GPU parity of the causal gradients (la_backward_causal) against the fp64 oracle.

Element by element on seeded inputs, for every (d, dv) pair, both input
dtypes, ragged tails and sequences split into many segments, with and
without an initial state; then the degenerate cases and sampled heads of the
training-shape workload.  The kernels compute in fp32 throughout (bf16 inputs
are exact in fp32), so both dtypes share one bound, TOL_BWD; the largest
error is in dL/dq, where two terms of similar size cancel.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_rnn_sequence_gb300 import linattn as la
from linear_rnn_sequence_gb300.workloads import (WORKLOADS, make_backward_inputs, random_qkv,
                                                 random_qkv_dy)
from metrics import TOL_BWD, rel_max_err

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, N, d, dv, dtype, scale
    (1, 2, 256, 32, 32, torch.float32, 1.0),
    (1, 3, 333, 64, 64, torch.float32, 1.0),
    (2, 2, 517, 128, 128, torch.float32, 0.2),
    (1, 2, 1000, 64, 128, torch.float32, 0.5),
    (1, 2, 700, 128, 64, torch.float32, 0.5),
    (2, 3, 1031, 64, 64, torch.bfloat16, 0.125),
    (1, 4, 777, 128, 128, torch.bfloat16, 0.0884),
    (1, 2, 129, 128, 32, torch.bfloat16, 1.0),
    (1, 2, 385, 32, 128, torch.bfloat16, 1.0),
    (1, 1, 4000, 128, 128, torch.bfloat16, 0.0884),
]


def _ids(c):
    B, H, N, d, dv, dt, s = c
    return f"B{B}H{H}N{N}d{d}dv{dv}{'bf16' if dt == torch.bfloat16 else 'f32'}"


def _state(B, H, d, dv, dt, seed):
    """A realistic initial state: the oracle's final state after a 50-token prefill."""
    q, k, v = random_qkv(B, H, 50, d, dv, dtype=dt, scale=0.5, seed=seed)
    _, S, z = oracle.causal_recurrent(q, k, v, return_state=True)
    return S, z


def _check(got, want):
    for name, g, w in zip(("dq", "dk", "dv", "dS_in", "dz_in"), got, want):
        if w is None:
            continue
        err = rel_max_err(g, w)
        assert err <= TOL_BWD, f"{name}: {err:.3e}"


@pytest.mark.parametrize("with_state", [False, True])
@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_backward_matches_oracle(case, with_state, cuda_device):
    B, H, N, d, dv, dt, s = case
    q, k, v, dy = random_qkv_dy(B, H, N, d, dv, dtype=dt, scale=s, seed=N + 5)
    S_in = z_in = None
    if with_state:
        S_in, z_in = _state(B, H, d, dv, dt, seed=N)
    dev = [t.to(cuda_device) for t in (q, k, v, dy)]
    Sd = None if S_in is None else torch.tensor(S_in, dtype=torch.float32, device=cuda_device)
    zd = None if z_in is None else torch.tensor(z_in, dtype=torch.float32, device=cuda_device)
    got = la.backward_causal(*dev, S_in=Sd, z_in=zd, return_state_grad=True)
    torch.cuda.synchronize()
    want = oracle.causal_backward(q, k, v, dy, S_in=S_in, z_in=z_in, return_state_grad=True)
    _check(got, want)


def test_backward_single_token(cuda_device):
    """N = 1 from a zero state: dv = dy, dq = dk = 0."""
    q, k, v, dy = random_qkv_dy(2, 3, 1, 64, 64, dtype=torch.bfloat16, seed=3)
    dq, dk, dvv = la.backward_causal(*(t.to(cuda_device) for t in (q, k, v, dy)))
    torch.cuda.synchronize()
    assert torch.allclose(dvv.cpu(), dy, rtol=1e-6, atol=1e-7)
    assert dq.abs().max().item() < 1e-5 and dk.abs().max().item() < 1e-5


def test_backward_fully_clamped(cuda_device):
    """eps above every denominator: the clamp blocks the den path everywhere."""
    q, k, v, dy = random_qkv_dy(1, 2, 300, 64, 64, dtype=torch.float32, scale=0.5, seed=9)
    got = la.backward_causal(*(t.to(cuda_device) for t in (q, k, v, dy)), eps=1e6)
    torch.cuda.synchronize()
    _check(got, oracle.causal_backward(q, k, v, dy, eps=1e6))


def test_backward_empty_sequence(cuda_device):
    q = torch.zeros(1, 2, 0, 64, dtype=torch.bfloat16, device=cuda_device)
    dy = torch.zeros(1, 2, 0, 64, dtype=torch.float32, device=cuda_device)
    gq, gk, gv, gS, gz = la.backward_causal(q, q, q, dy, return_state_grad=True)
    torch.cuda.synchronize()
    assert gq.shape == (1, 2, 0, 64) and not gS.any() and not gz.any()


@pytest.mark.parametrize("name,heads", [("causal_backward_bf16_b8h16n8192d128", (0, 77, 127))])
def test_backward_workload_sampled_heads(name, heads, cuda_device):
    """Full-size training shape, in the launch configuration the benchmark times;
    the oracle checks whole heads (heads are independent)."""
    w = WORKLOADS[name]
    q, k, v, dy = make_backward_inputs(w)
    dq, dk, dvv = la.backward_causal(*(t.to(cuda_device) for t in (q, k, v, dy)))
    torch.cuda.synchronize()
    flat = lambda t: t.reshape(w.BH, w.N, t.shape[-1])
    for h in heads:
        want = oracle.causal_backward(flat(q)[h], flat(k)[h], flat(v)[h], flat(dy)[h])
        _check([flat(dq)[h], flat(dk)[h], flat(dvv)[h]], want)


def test_backward_long_sequence_sampled_heads(cuda_device):
    """B1 H32 N131072 d64: the sequence is split into segments joined by the
    prefix and suffix scans; whole heads are checked against the oracle."""
    w = WORKLOADS["causal_bf16_b1h32n131072d64"]
    q, k, v, dy = make_backward_inputs(w.with_(mode="backward"))
    dq, dk, dvv = la.backward_causal(*(t.to(cuda_device) for t in (q, k, v, dy)))
    torch.cuda.synchronize()
    flat = lambda t: t.reshape(w.BH, w.N, t.shape[-1])
    for h in (0, 31):
        want = oracle.causal_backward(flat(q)[h], flat(k)[h], flat(v)[h], flat(dy)[h])
        _check([flat(dq)[h], flat(dk)[h], flat(dvv)[h]], want)


DECAY_CASES = [
    (1, 2, 256, 32, 32, torch.float32, 1.0),
    (2, 2, 517, 128, 128, torch.float32, 0.2),
    (1, 3, 1031, 64, 64, torch.bfloat16, 0.125),
    (1, 2, 385, 32, 128, torch.bfloat16, 1.0),
    (1, 1, 4000, 128, 128, torch.bfloat16, 0.0884),
]


@pytest.mark.parametrize("with_state", [False, True])
@pytest.mark.parametrize("case", DECAY_CASES, ids=_ids)
def test_backward_decay_matches_oracle(case, with_state, cuda_device):
    """Gradients of the decayed forward, per-head gamma; split sequences too."""
    from linear_rnn_sequence_gb300.workloads import head_decays
    B, H, N, d, dv, dt, s = case
    q, k, v, dy = random_qkv_dy(B, H, N, d, dv, dtype=dt, scale=s, seed=N + 17)
    gam = head_decays(H)
    S_in = z_in = None
    if with_state:
        qp, kp, vp = random_qkv(B, H, 50, d, dv, dtype=dt, scale=0.5, seed=N)
        _, S_in, z_in = oracle.causal_recurrent_decay(qp, kp, vp, gam, return_state=True)
    dev = lambda t: None if t is None else torch.as_tensor(t, dtype=torch.float32).to(cuda_device)
    got = la.backward_causal(*(t.to(cuda_device) for t in (q, k, v, dy)), S_in=dev(S_in),
                             z_in=dev(z_in), return_state_grad=True, gamma=gam.to(cuda_device))
    torch.cuda.synchronize()
    want = oracle.causal_backward(q, k, v, dy, S_in=S_in, z_in=z_in, return_state_grad=True,
                                  gamma=gam)
    _check(got, want)


def test_backward_decay_long_sequence_sampled_heads(cuda_device):
    """B1 H32 N131072 d64 with decays: split into segments, decayed scans."""
    from linear_rnn_sequence_gb300.workloads import head_decays
    w = WORKLOADS["causal_bf16_b1h32n131072d64"]
    q, k, v, dy = make_backward_inputs(w.with_(mode="backward"))
    gam = head_decays(w.H)
    dq, dk, dvv = la.backward_causal(*(t.to(cuda_device) for t in (q, k, v, dy)),
                                     gamma=gam.to(cuda_device))
    torch.cuda.synchronize()
    flat = lambda t: t.reshape(w.BH, w.N, t.shape[-1])
    for h in (0, 31):
        want = oracle.causal_backward(flat(q)[h], flat(k)[h], flat(v)[h], flat(dy)[h],
                                      gamma=gam[h:h + 1])
        _check([flat(dq)[h], flat(dk)[h], flat(dvv)[h]], want)


@pytest.mark.parametrize("decay", [False, True])
def test_backward_outputs_stay_in_bounds_and_are_deterministic(decay, cuda_device):
    """Canary-padded gradient buffers (a split, ragged sequence with an initial
    state): nothing is written past any output, and two runs agree bitwise."""
    from linear_rnn_sequence_gb300.workloads import head_decays
    B, H, N, d, dv = 1, 2, 1000, 64, 128
    q, k, v, dy = (t.to(cuda_device) for t in random_qkv_dy(B, H, N, d, dv,
                                                            dtype=torch.bfloat16, scale=0.2,
                                                            seed=21))
    S_in = torch.randn(B, H, d, dv, device=cuda_device)
    z_in = torch.rand(B, H, d, device=cuda_device) + 1.0
    gam = head_decays(H).to(cuda_device) if decay else None
    pad = 4096
    sizes = (B * H * N * d, B * H * N * d, B * H * N * dv, B * H * d * dv, B * H * d)
    bufs = [torch.full((n + pad,), 12345.0, device=cuda_device) for n in sizes]
    views = [b[:n] for b, n in zip(bufs, sizes)]
    gq, gk, gv = (views[0].view(B, H, N, d), views[1].view(B, H, N, d),
                  views[2].view(B, H, N, dv))
    ws = la.alloc_workspace(la.causal_backward_workspace_bytes(B, H, N, d, dv), cuda_device)
    out = la.backward_causal(q, k, v, dy, S_in=S_in, z_in=z_in, return_state_grad=True,
                             out=(gq, gk, gv), workspace=ws, gamma=gam)
    torch.cuda.synchronize()
    for b in bufs[:3]:
        assert (b[-pad:] == 12345.0).all()
    again = la.backward_causal(q, k, v, dy, S_in=S_in, z_in=z_in, return_state_grad=True,
                               workspace=ws, gamma=gam)
    torch.cuda.synchronize()
    for x, y in zip(out, again):
        assert torch.equal(x, y)


@pytest.mark.parametrize("gammas", [(0.0, 0.1, 0.2, 0.24), (0.25, 0.5, 0.9, 1.0)])
def test_backward_decay_both_state_paths(gammas, cuda_device):
    """gamma < 1/4 multiplies the state per element; gamma >= 1/4 carries it
    rescaled within each chunk.  Both, including the limits 0 and 1, on a
    split sequence with an initial state."""
    B, H, N, d, dv = 1, 4, 2000, 64, 64
    q, k, v, dy = random_qkv_dy(B, H, N, d, dv, dtype=torch.float32, scale=0.5, seed=31)
    gam = torch.tensor(gammas, dtype=torch.float32)
    qp, kp, vp = random_qkv(B, H, 30, d, dv, dtype=torch.float32, scale=0.5, seed=32)
    _, S_in, z_in = oracle.causal_recurrent_decay(qp, kp, vp, gam, return_state=True)
    dev = lambda t: torch.as_tensor(t, dtype=torch.float32).to(cuda_device)
    got = la.backward_causal(*(t.to(cuda_device) for t in (q, k, v, dy)), S_in=dev(S_in),
                             z_in=dev(z_in), return_state_grad=True, gamma=gam.to(cuda_device))
    y = la.forward_causal_decay(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                gam.to(cuda_device), S_in=dev(S_in), z_in=dev(z_in))
    torch.cuda.synchronize()
    want = oracle.causal_backward(q, k, v, dy, S_in=S_in, z_in=z_in, return_state_grad=True,
                                  gamma=gam)
    _check(got, want)
    assert rel_max_err(y, oracle.causal_recurrent_decay(q, k, v, gam, S_in=S_in,
                                                        z_in=z_in)) <= TOL_BWD


def test_backward_with_partly_active_clamp(cuda_device):
    """eps between the denominators (away from all of them): tokens below it
    pass no gradient through the denominator."""
    from tests import backward_pins as bp
    B, H, N, d, dv = 1, 2, 300, 32, 32
    q, k, v, dy = random_qkv_dy(B, H, N, d, dv, dtype=torch.float32, scale=1.0, seed=33)
    dd = np.sort(bp.dens(q.double().numpy(), k.double().numpy()).reshape(-1))
    gaps = np.diff(dd)
    i = int(np.argmax(gaps[: len(gaps) // 2]))   # a wide gap among the smaller dens
    eps = float((dd[i] + dd[i + 1]) / 2)
    assert 0 < i and gaps[i] > 1e-3 * dd[i]
    got = la.backward_causal(*(t.to(cuda_device) for t in (q, k, v, dy)), eps=eps)
    torch.cuda.synchronize()
    _check(got, oracle.causal_backward(q, k, v, dy, eps=eps))
