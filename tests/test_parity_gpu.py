"""GPU parity against the fp64 oracle, element by element, through the C ABI.

Sizes here are small enough for the oracle to finish in seconds while still
spanning several blocks and a ragged tail; the full-size workloads are in
test_parity_full_gpu.py.  Metric: max |GPU - oracle| / RMS(oracle).
"""
import numpy as np
import pytest
import torch

import oracle
from linear_rnn_sequence_gb300 import linattn as la
from linear_rnn_sequence_gb300.workloads import random_qkv
from metrics import TOL_BF16, TOL_F32, rel_max_err, tol_for

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
]


def _ids(c):
    B, H, N, d, dv, dt, s = c
    return f"B{B}H{H}N{N}d{d}dv{dv}{'bf16' if dt == torch.bfloat16 else 'f32'}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_causal_matches_oracle(case, cuda_device):
    B, H, N, d, dv, dt, s = case
    q, k, v = random_qkv(B, H, N, d, dv, dtype=dt, scale=s, seed=N)
    y, S, z = la.forward_causal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                return_state=True, check_status=True)
    torch.cuda.synchronize()
    yo, So, zo = oracle.causal_recurrent(q, k, v, return_state=True)
    tol = tol_for(dt)
    assert rel_max_err(y, yo) <= tol
    assert rel_max_err(S, So) <= tol
    assert rel_max_err(z, zo) <= tol


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_noncausal_matches_oracle(case, cuda_device):
    B, H, N, d, dv, dt, s = case
    q, k, v = random_qkv(B, H, N, d, dv, dtype=dt, scale=s, seed=N + 1)
    y, S, z = la.forward_noncausal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                   return_state=True, check_status=True)
    torch.cuda.synchronize()
    yo, So, zo = oracle.noncausal(q, k, v, return_state=True)
    tol = tol_for(dt)
    assert rel_max_err(y, yo) <= tol
    assert rel_max_err(S, So) <= tol
    assert rel_max_err(z, zo) <= tol


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("d,dv", [(32, 32), (64, 128), (128, 128), (128, 64)])
def test_decode_steps_match_oracle(dt, d, dv, cuda_device):
    B, H, Np, steps = 2, 3, 100, 20
    q, k, v = random_qkv(B, H, Np, d, dv, dtype=dt, scale=0.5, seed=7)
    _, So, zo = oracle.causal_recurrent(q, k, v, return_state=True)
    S = torch.tensor(So, dtype=torch.float32, device=cuda_device)
    z = torch.tensor(zo, dtype=torch.float32, device=cuda_device)
    Sref, zref = So.copy(), zo.copy()
    g = torch.Generator().manual_seed(11)
    for t in range(steps):
        qs = (torch.randn(B, H, d, generator=g) * 0.3).to(dt)
        ks = (torch.randn(B, H, d, generator=g) * 0.3).to(dt)
        vs = (torch.randn(B, H, dv, generator=g) * 0.3).to(dt)
        y = la.decode_step(qs.to(cuda_device), ks.to(cuda_device), vs.to(cuda_device), S, z)
        yo, Sref, zref = oracle.decode_step(qs, ks, vs, Sref, zref)
        torch.cuda.synchronize()
        assert rel_max_err(y, yo) <= tol_for(dt), f"step {t}"
    assert rel_max_err(S, Sref) <= tol_for(dt)
    assert rel_max_err(z, zref) <= tol_for(dt)


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_causal_initial_state_and_split(dt, cuda_device):
    """prefill(N1) -> S, z; causal(N2, S_in) equals the tail of causal(N1+N2)."""
    B, H, N1, N2, d, dv = 1, 3, 301, 259, 64, 64
    q, k, v = random_qkv(B, H, N1 + N2, d, dv, dtype=dt, scale=0.3, seed=21)
    qd, kd, vd = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device)
    y_full, S_full, z_full = la.forward_causal(qd, kd, vd, return_state=True, check_status=True)
    _, S1, z1 = la.forward_causal(qd[:, :, :N1].contiguous(), kd[:, :, :N1].contiguous(),
                                  vd[:, :, :N1].contiguous(), return_state=True)
    y2, S2, z2 = la.forward_causal(qd[:, :, N1:].contiguous(), kd[:, :, N1:].contiguous(),
                                   vd[:, :, N1:].contiguous(), S_in=S1, z_in=z1,
                                   return_state=True)
    torch.cuda.synchronize()
    yo, So, zo = oracle.causal_recurrent(q, k, v, return_state=True)
    tol = tol_for(dt)
    assert rel_max_err(y2, yo[:, :, N1:]) <= tol
    assert rel_max_err(S2, So) <= tol and rel_max_err(z2, zo) <= tol
    assert rel_max_err(S_full, So) <= tol


def test_prefill_then_decode_equals_causal(cuda_device):
    B, H, Np, M, d, dv = 1, 2, 200, 8, 128, 128
    q, k, v = random_qkv(B, H, Np + M, d, dv, dtype=torch.bfloat16, scale=0.09, seed=31)
    qd, kd, vd = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device)
    _, S, z = la.forward_causal(qd[:, :, :Np].contiguous(), kd[:, :, :Np].contiguous(),
                                vd[:, :, :Np].contiguous(), return_state=True)
    ys = [la.decode_step(qd[:, :, t].contiguous(), kd[:, :, t].contiguous(),
                         vd[:, :, t].contiguous(), S, z) for t in range(Np, Np + M)]
    torch.cuda.synchronize()
    yo, So, zo = oracle.causal_recurrent(q, k, v, return_state=True)
    got = torch.stack(ys, dim=2)
    assert rel_max_err(got, yo[:, :, Np:]) <= TOL_BF16
    assert rel_max_err(S, So) <= TOL_BF16


@pytest.mark.parametrize("N", [0, 1, 2, 63, 64, 65, 127, 128, 129])
def test_causal_edge_lengths(N, cuda_device):
    B, H, d, dv = 1, 2, 128, 128
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.bfloat16, scale=0.3, seed=41 + N)
    S_in = torch.randn(B, H, d, dv, generator=torch.Generator().manual_seed(N)) * 0.1
    z_in = torch.rand(B, H, d, generator=torch.Generator().manual_seed(N + 1)) * 3 + 1
    y, S, z = la.forward_causal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                S_in=S_in.to(cuda_device), z_in=z_in.to(cuda_device),
                                return_state=True, check_status=True)
    torch.cuda.synchronize()
    yo, So, zo = oracle.causal_recurrent(q, k, v, S_in=S_in, z_in=z_in, return_state=True)
    assert y.shape == (B, H, N, dv)
    if N:
        assert rel_max_err(y, yo) <= TOL_BF16
    assert rel_max_err(S, So) <= TOL_BF16 and rel_max_err(z, zo) <= TOL_BF16


def test_first_token_returns_v1(cuda_device):
    """y_1 = w_11 v_1 / w_11 = v_1 (one token from a zero state).  The
    tensor-core path forms the numerator from the weight split into bf16 hi +
    lo, which carries w to 2^-18 of itself, and the denominator from w in
    fp32, so each element of y_1 is v_1 to within 2^-17 of |v_1|."""
    q, k, v = random_qkv(2, 4, 1, 64, 64, dtype=torch.bfloat16, scale=1.0, seed=3)
    y = la.forward_causal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device))
    torch.cuda.synchronize()
    vd = v.double()
    assert torch.all((y.cpu().double() - vd).abs() <= 2.0 ** -17 * vd.abs())


def test_outputs_stay_in_bounds(cuda_device):
    """Canary-padded buffers: nothing is written past y, S or z."""
    B, H, N, d, dv = 1, 2, 130, 64, 64
    q, k, v = (t.to(cuda_device) for t in random_qkv(B, H, N, d, dv, dtype=torch.bfloat16,
                                                     scale=0.2, seed=5))
    pad = 4096
    ybuf = torch.full((B * H * N * dv + pad,), 12345.0, device=cuda_device)
    Sbuf = torch.full((B * H * d * dv + pad,), 12345.0, device=cuda_device)
    zbuf = torch.full((B * H * d + pad,), 12345.0, device=cuda_device)
    y = ybuf[: B * H * N * dv].view(B, H, N, dv)
    S = Sbuf[: B * H * d * dv].view(B, H, d, dv)
    z = zbuf[: B * H * d].view(B, H, d)
    la.forward_causal(q, k, v, out=y, S_out=S, z_out=z, return_state=True, check_status=True)
    la.forward_noncausal(q, k, v, out=y, S_out=S, z_out=z, return_state=True)
    torch.cuda.synchronize()
    for buf in (ybuf, Sbuf, zbuf):
        assert (buf[-pad:] == 12345.0).all()


def test_runs_are_bitwise_deterministic(cuda_device):
    q, k, v = (t.to(cuda_device) for t in random_qkv(2, 4, 1500, 128, 128,
                                                     dtype=torch.bfloat16, scale=0.09, seed=9))
    a = la.forward_causal(q, k, v, return_state=True, check_status=True)
    b = la.forward_causal(q, k, v, return_state=True, check_status=True)
    c = la.forward_noncausal(q, k, v, return_state=True, check_status=True)
    d = la.forward_noncausal(q, k, v, return_state=True, check_status=True)
    torch.cuda.synchronize()
    for x, y in zip(a + c, b + d):
        assert torch.equal(x, y)


def test_misaligned_pointer_is_rejected(cuda_device):
    q, k, v = (t.to(cuda_device) for t in random_qkv(1, 1, 64, 64, 64, dtype=torch.bfloat16))
    flat = torch.empty(64 * 64 + 8, dtype=torch.bfloat16, device=cuda_device)
    qm = flat[1:1 + 64 * 64].view(1, 1, 64, 64)   # 2-byte offset
    with pytest.raises(la.LinAttnError) as ei:
        la.forward_causal(qm, k, v)
    assert ei.value.status == la.LA_ERR_INVALID_ARG


def test_workspace_too_small_is_rejected(cuda_device):
    q, k, v = (t.to(cuda_device) for t in random_qkv(1, 2, 4096, 64, 64, dtype=torch.bfloat16))
    need = la.noncausal_workspace_bytes(1, 2, 4096, 64, 64)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(la.LinAttnError) as ei:
        la.forward_noncausal(q, k, v, workspace=ws)
    assert ei.value.status == la.LA_ERR_WORKSPACE


# The tensor-core non-causal path (bf16, d and dv in {64, 128}): every shape,
# ragged tails, one-block and many-segment splits (few heads, long sequences).
@pytest.mark.parametrize("B,H,N,d,dv", [
    (1, 1, 1, 64, 64), (1, 2, 2, 128, 128), (1, 2, 127, 64, 128), (1, 2, 128, 128, 64),
    (1, 2, 129, 64, 64), (2, 3, 1000, 64, 128), (1, 3, 2049, 128, 64),
    (1, 1, 20000, 64, 64), (1, 2, 9001, 128, 128),
])
def test_noncausal_tc_shapes(B, H, N, d, dv, cuda_device):
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.bfloat16, scale=d ** -0.5, seed=N + d)
    y, S, z = la.forward_noncausal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                   return_state=True, check_status=True)
    torch.cuda.synchronize()
    yo, So, zo = oracle.noncausal(q, k, v, return_state=True)
    e = (rel_max_err(y, yo), rel_max_err(S, So), rel_max_err(z, zo))
    print(f"noncausal tc B{B}H{H}N{N}d{d}dv{dv}: y {e[0]:.2e} S {e[1]:.2e} z {e[2]:.2e}")
    assert max(e) <= TOL_BF16


@pytest.mark.parametrize("B,H,N,d,dv,dt,pinned", [
    (2, 8, 700, 128, 128, torch.bfloat16, True),     # 16 heads in 8 groups
    (1, 3, 257, 64, 64, torch.bfloat16, False),      # pageable memory, fewer heads than groups
    (1, 5, 300, 64, 32, torch.float32, True),        # CUDA-core path
])
def test_causal_host_buffers_match_oracle(B, H, N, d, dv, dt, pinned, cuda_device):
    q, k, v = random_qkv(B, H, N, d, dv, dtype=dt, scale=d ** -0.5, seed=N + H)
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    y, S, z = la.forward_causal_host(q, k, v, return_state=True, device=cuda_device)
    assert not y.is_cuda and y.shape == (B, H, N, dv)
    yo, So, zo = oracle.causal_recurrent(q, k, v, return_state=True)
    tol = tol_for(dt)
    assert rel_max_err(y, yo) <= tol
    assert rel_max_err(S, So) <= tol and rel_max_err(z, zo) <= tol
    # same numbers as the device-pointer entry point, up to summation order
    yd = la.forward_causal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device)).cpu()
    assert rel_max_err(y, yd.double().numpy()) <= tol


def test_causal_host_buffer_too_small_is_rejected(cuda_device):
    q, k, v = random_qkv(1, 2, 256, 64, 64, dtype=torch.bfloat16)
    need = la.causal_host_buffer_bytes(1, 2, 256, 64, 64)
    buf = torch.empty(need - 256, dtype=torch.uint8, device=cuda_device)
    with pytest.raises(la.LinAttnError) as ei:
        la.forward_causal_host(q, k, v, dev_buf=buf, device=cuda_device)
    assert ei.value.status == la.LA_ERR_WORKSPACE


# The tensor-core causal path for every (d, dv) pair, ragged tails, one-block
# sequences, the sequence split (few heads, long sequences) and one CTA per
# head for 64 to 128 heads, with and without an initial state.
@pytest.mark.parametrize("B,H,N,d,dv,with_state", [
    (1, 1, 1, 64, 64, False), (1, 2, 127, 64, 128, True), (1, 2, 129, 128, 64, False),
    (2, 3, 1000, 64, 128, False), (1, 3, 2049, 128, 64, True), (1, 1, 20000, 64, 64, True),
    (1, 2, 9001, 128, 128, False), (96, 1, 300, 64, 128, False),
    (1, 96, 600, 64, 64, True), (1, 128, 1031, 128, 128, False), (4, 25, 2049, 64, 128, True),
    (2, 64, 777, 128, 64, True),
])
def test_causal_tc_shapes(B, H, N, d, dv, with_state, cuda_device):
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.bfloat16, scale=d ** -0.5, seed=N + dv)
    S_in = z_in = None
    if with_state:
        g = torch.Generator().manual_seed(N)
        S_in = torch.randn(B, H, d, dv, generator=g) * 0.5
        z_in = torch.rand(B, H, d, generator=g) * 5 + 1
    y, S, z = la.forward_causal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                S_in=None if S_in is None else S_in.to(cuda_device),
                                z_in=None if z_in is None else z_in.to(cuda_device),
                                return_state=True, check_status=True)
    torch.cuda.synchronize()
    yo, So, zo = oracle.causal_recurrent(q, k, v, S_in=S_in, z_in=z_in, return_state=True)
    e = (rel_max_err(y, yo), rel_max_err(S, So), rel_max_err(z, zo))
    print(f"causal tc B{B}H{H}N{N}d{d}dv{dv} state={with_state}: y {e[0]:.2e} S {e[1]:.2e} z {e[2]:.2e}")
    assert max(e) <= TOL_BF16
