"""GPU parity of the gated causal form on the tensor cores against the fp64
oracle ("Linear Attention/es", "Variantes y extensiones": gated linear
attention, read as S_t = g_t S_{t-1} + phi(k_t) v_t^T with z alike).

With bf16 inputs, d and dv in {64, 128}, one gate per token and elu + 1,
la_forward_causal_gated runs the decayed chunk kernel with the decay taken
from per-block tables of gate products.  A head goes there when all its gates
lie in [2^-1/2, 1] (the device decides from the values); the other heads run
on the CUDA cores in fp32.  Tensor-core heads are held to the bf16 bound, 2e-2
of RMS, CUDA-core heads to 1e-4.
"""
import numpy as np
import pytest
import torch

import oracle
from linear_rnn_sequence_gb300 import linattn as la
from linear_rnn_sequence_gb300.workloads import random_gated
from metrics import TOL_BF16, TOL_F32, rel_max_err

pytestmark = pytest.mark.gpu


def _phi(x):
    x = np.asarray(x, np.float64)
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def gated_dens(q, k, g):
    """fp64 denominators phi(q_t) . z_t of the gated form (one gate per token),
    only to place eps between them."""
    fq, fk, gg = _phi(q.double().numpy()), _phi(k.double().numpy()), g.double().numpy()
    B, H, N, d = fq.shape
    out = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            z = np.zeros(d)
            for t in range(N):
                z = gg[b, h, t] * z + fk[b, h, t]
                out[b, h, t] = fq[b, h, t] @ z
    return out


def _run(q, k, v, g, dev, eps=1e-6, S_in=None, z_in=None):
    d = lambda t: None if t is None else t.to(dev)
    out = la.forward_causal_gated(d(q), d(k), d(v), gate=d(g), eps=eps, S_in=d(S_in),
                                  z_in=d(z_in), return_state=True, check_status=True)
    torch.cuda.synchronize()
    return out


def _check(got, want, tol, what=""):
    for name, a, b in zip(("y", "S", "z"), got, want):
        err = rel_max_err(a, b)
        assert err <= tol, f"{what} {name}: {err:.3e}"


@pytest.mark.parametrize("N", [1, 127, 128, 129, 300, 1000])
@pytest.mark.parametrize("d,dv", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_gated_tc_shapes(d, dv, N, cuda_device):
    B, H = 1, 3
    q, k, v, g = random_gated(B, H, N, d, dv, 1, dtype=torch.bfloat16, scale=d ** -0.5,
                              seed=N + d + dv)
    gen = torch.Generator().manual_seed(N)
    S_in = torch.randn(B, H, d, dv, generator=gen) * 0.5
    z_in = torch.rand(B, H, d, generator=gen) * 5 + 1
    got = _run(q, k, v, g, cuda_device, S_in=S_in, z_in=z_in)
    want = oracle.causal_gated(q, k, v, gate=g, S_in=S_in, z_in=z_in, return_state=True)
    _check(got, want, TOL_BF16, f"d{d} dv{dv} N{N}")


# Few heads and long sequences: the sequence is split into segments (a state
# pass over the segments with their products of gates, a prefix scan, then the
# chunk kernel from each segment's prefix).
@pytest.mark.parametrize("B,H,N,d,dv", [(1, 2, 20000, 64, 64), (1, 3, 5000, 128, 128),
                                        (2, 2, 3000, 64, 128)])
def test_gated_tc_split_sequences(B, H, N, d, dv, cuda_device):
    q, k, v, g = random_gated(B, H, N, d, dv, 1, dtype=torch.bfloat16, scale=d ** -0.5, seed=N + d)
    gen = torch.Generator().manual_seed(N + 1)
    S_in = torch.randn(B, H, d, dv, generator=gen) * 0.5
    z_in = torch.rand(B, H, d, generator=gen) * 5 + 1
    got = _run(q, k, v, g, cuda_device, S_in=S_in, z_in=z_in)
    want = oracle.causal_gated(q, k, v, gate=g, S_in=S_in, z_in=z_in, return_state=True)
    _check(got, want, TOL_BF16, f"B{B} H{H} N{N} d{d} dv{dv}")


def test_gated_tc_constant_gates_are_the_decay(cuda_device):
    """Gates equal to a per-head gamma at every token give the decayed form."""
    B, H, N, d, dv = 2, 4, 700, 64, 64
    q, k, v, _ = random_gated(B, H, N, d, dv, 1, dtype=torch.bfloat16, scale=0.125, seed=11)
    gam = torch.tensor([0.72, 0.9, 0.999, 1.0])
    g = gam[None, :, None].expand(B, H, N).contiguous()
    y = _run(q, k, v, g, cuda_device)[0]
    assert rel_max_err(y, oracle.causal_recurrent_decay(q, k, v, gam)) <= TOL_BF16


def test_gated_tc_heads_on_both_paths_in_place(cuda_device):
    """One call with heads on both paths (a gate below 2^-1/2, a closed gate, a
    NaN-free gate above 1 is not drawn), and S_in, z_in the same buffers as
    S_out, z_out: each path reads its heads' initial state before it writes."""
    B, H, N, d, dv = 1, 4, 500, 64, 64
    q, k, v, g = random_gated(B, H, N, d, dv, 1, dtype=torch.bfloat16, scale=0.125, seed=12)
    g[0, 1, 250] = 0.5    # below the tensor-core range
    g[0, 3, 100] = 0.0    # a closed gate
    gen = torch.Generator().manual_seed(13)
    S0 = torch.randn(B, H, d, dv, generator=gen) * 0.5
    z0 = torch.rand(B, H, d, generator=gen) * 5 + 1
    yo, So, zo = oracle.causal_gated(q, k, v, gate=g, S_in=S0, z_in=z0, return_state=True)
    S = S0.to(cuda_device)
    z = z0.to(cuda_device)
    y = la.forward_causal_gated(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                gate=g.to(cuda_device), S_in=S, z_in=z, S_out=S, z_out=z,
                                check_status=True)
    torch.cuda.synchronize()
    for h, tol in ((0, TOL_BF16), (1, TOL_F32), (2, TOL_BF16), (3, TOL_F32)):
        for name, a, b in (("y", y[:, h], yo[:, h]), ("S", S[:, h], So[:, h]),
                           ("z", z[:, h], zo[:, h])):
            err = rel_max_err(a, b)
            assert err <= tol, f"head {h} {name}: {err:.3e}"


@pytest.mark.parametrize("clamp", ["all", "median"])
def test_gated_tc_clamp(clamp, cuda_device):
    """eps above every denominator (y = num / eps) or at their median: the
    kernel's clamp, rescaled per row by the block's gate products, binds."""
    B, H, N, d, dv = 1, 2, 400, 64, 64
    q, k, v, g = random_gated(B, H, N, d, dv, 1, dtype=torch.bfloat16, scale=0.125, seed=14)
    dens = gated_dens(q, k, g)
    eps = float(dens.max() * 4) if clamp == "all" else float(np.median(dens))
    got = _run(q, k, v, g, cuda_device, eps=eps)
    want = oracle.causal_gated(q, k, v, gate=g, eps=eps, return_state=True)
    _check(got, want, TOL_BF16, clamp)


# The final state of strongly shifted inputs carries the bf16 rounding of the
# key features as a cancelling sum (as for the other tensor-core paths); y and
# z stay within the bf16 bound.
TOL_STATE_SHIFTED = 4e-2


@pytest.mark.parametrize("scale,shift", [(1.0, -4.0), (3.0, 0.0)])
def test_gated_tc_input_range(scale, shift, cuda_device):
    B, H, N, d, dv = 1, 4, 600, 128, 128
    q, k, v, g = random_gated(B, H, N, d, dv, 1, dtype=torch.bfloat16, scale=scale, seed=15,
                              shift=shift)
    y, S, z = _run(q, k, v, g, cuda_device)
    yo, So, zo = oracle.causal_gated(q, k, v, gate=g, return_state=True)
    assert rel_max_err(y, yo) <= TOL_BF16
    assert rel_max_err(z, zo) <= TOL_BF16
    assert rel_max_err(S, So) <= (TOL_STATE_SHIFTED if shift else TOL_BF16)


def test_gated_tc_is_deterministic(cuda_device):
    B, H, N, d, dv = 1, 2, 777, 128, 128
    q, k, v, g = (t.to(cuda_device) for t in random_gated(B, H, N, d, dv, 1, dtype=torch.bfloat16,
                                                          scale=0.09, seed=16))
    y1 = la.forward_causal_gated(q, k, v, gate=g)
    y2 = la.forward_causal_gated(q, k, v, gate=g)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_gated_tc_dropped_copy_times_out_and_context_survives(cuda_device):
    """The fault hook on the gated tensor-core path: a copy that never arrives
    runs out its bounded wait, the call reports LA_ERR_TIMEOUT, and the next
    call is clean."""
    B, H, N, d, dv = 1, 4, 600, 64, 64
    q, k, v, g = random_gated(B, H, N, d, dv, 1, dtype=torch.bfloat16, scale=0.125, seed=17)
    qd, kd, vd, gd = (t.to(cuda_device) for t in (q, k, v, g))
    try:
        la.set_fault(drop_load_item=1, wait_limit_ns=5_000_000)
        with pytest.raises(la.LinAttnError) as ei:
            la.forward_causal_gated(qd, kd, vd, gate=gd, check_status=True)
        assert ei.value.status == la.LA_ERR_TIMEOUT
    finally:
        la.set_fault(-1, 0)
    y = la.forward_causal_gated(qd, kd, vd, gate=gd, check_status=True)
    torch.cuda.synchronize()
    assert rel_max_err(y, oracle.causal_gated(q, k, v, gate=g)) <= TOL_BF16


def test_gated_workspace_size_and_rejection(cuda_device):
    B, H, N, d, dv = 1, 2, 300, 64, 64
    need = la.causal_gated_workspace_bytes(B, H, N, d, dv, torch.bfloat16, "elu1", 1)
    nb = (N + 127) // 128
    assert need >= 256 + B * H * nb * 1056
    assert la.causal_gated_workspace_bytes(B, H, N, d, dv, torch.float32, "elu1", 1) == 256
    assert la.causal_gated_workspace_bytes(B, H, N, d, dv, torch.bfloat16, "elu1", d) == 256
    q, k, v, g = (t.to(cuda_device) for t in random_gated(B, H, N, d, dv, 1, dtype=torch.bfloat16,
                                                          scale=0.125, seed=18))
    small = torch.empty(need - 256, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(la.LinAttnError) as ei:
        la.forward_causal_gated(q, k, v, gate=g, workspace=small)
    assert ei.value.status == la.LA_ERR_WORKSPACE
