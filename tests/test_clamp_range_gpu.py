"""GPU parity where the denominator clamp binds, and for inputs outside the
well-centred range, on every forward entry point.

The pages clamp the denominator from below (``clamp_min(eps)`` in the worked
PyTorch examples of "Linear Transformer (Transformers are RNNs)", read as
max(den, eps)).  With the workloads' inputs den is far above eps = 1e-6, so
here eps is set above every denominator (fully clamped: y = num / eps) or at
the median of them (partly clamped), on both tensor-core paths (whole heads
and sequences split into segments), the decayed tensor-core kernel (whose
clamp is rescaled per row), the CUDA-core kernels and decode, and the GPU is
compared with the oracle element by element.

The range tests draw q and k far from zero: N(-4, 1), where every feature
phi = e^x is far below 1, and N(0, 9).  The bf16 tensor-core kernels split
each token's features as c + (phi - c) with a per-token constant c, so the
bf16 bound (2e-2 of RMS) holds there too; float32 inputs take the CUDA-core
kernels and meet 1e-4 even for N(-8, 1).
"""
import numpy as np
import pytest
import torch

import oracle
from linear_rnn_sequence_gb300 import linattn as la
from linear_rnn_sequence_gb300.workloads import random_qkv
from metrics import TOL_BF16, TOL_F32, rel_max_err, tol_for

pytestmark = pytest.mark.gpu


def _phi(x):
    x = np.asarray(x, np.float64)
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def causal_dens(q, k, gamma=None):
    """fp64 denominators phi(q_t) . z_t of the causal form (z_t with a decay
    per head when gamma is given), only to place eps between them."""
    fq, fk = _phi(q.double().numpy()), _phi(k.double().numpy())
    B, H, N, d = fq.shape
    out = np.empty((B, H, N))
    for h in range(H):
        g = 1.0 if gamma is None else float(gamma[h])
        for b in range(B):
            z = np.zeros(d)
            for t in range(N):
                z = g * z + fk[b, h, t]
                out[b, h, t] = fq[b, h, t] @ z
    return out


def _dev(t, dev):
    return None if t is None else torch.as_tensor(t, dtype=torch.float32).to(dev)


def _check(got, want, tol, what=""):
    for name, g, w in zip(("y", "S", "z"), got, want):
        err = rel_max_err(g, w)
        assert err <= tol, f"{what} {name}: {err:.3e}"


# (name, B, H, N, d, dv, dtype): which kernels run is noted per case
CAUSAL_CASES = [
    ("tc_whole_heads", 2, 48, 300, 64, 64, torch.bfloat16),      # 96 heads: one item per head
    ("tc_split", 1, 2, 2000, 64, 128, torch.bfloat16),           # segments + prefix scan
    ("tc_whole_heads_d128", 1, 96, 200, 128, 128, torch.bfloat16),
    ("cuda_cores_f32", 1, 2, 700, 64, 64, torch.float32),
    ("cuda_cores_bf16_d32", 1, 2, 333, 32, 32, torch.bfloat16),
]


@pytest.mark.parametrize("clamp", ["full", "partly"])
@pytest.mark.parametrize("case", CAUSAL_CASES, ids=lambda c: c[0])
def test_causal_clamp(case, clamp, cuda_device):
    name, B, H, N, d, dv, dt = case
    q, k, v = random_qkv(B, H, N, d, dv, dtype=dt, scale=d ** -0.5, seed=N + H)
    eps = 1e9 if clamp == "full" else float(np.median(causal_dens(q, k)))
    y, S, z = la.forward_causal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device), eps=eps,
                                return_state=True, check_status=True)
    torch.cuda.synchronize()
    want = oracle.causal_recurrent(q, k, v, eps=eps, return_state=True)
    _check((y, S, z), want, tol_for(dt), f"{name} eps={eps:.4g}")


NONCAUSAL_CASES = [
    ("tc", 1, 3, 1000, 64, 64, torch.bfloat16),
    ("tc_d128", 2, 2, 777, 128, 128, torch.bfloat16),
    ("cuda_cores_f32", 1, 2, 500, 128, 64, torch.float32),
]


@pytest.mark.parametrize("clamp", ["full", "partly"])
@pytest.mark.parametrize("case", NONCAUSAL_CASES, ids=lambda c: c[0])
def test_noncausal_clamp(case, clamp, cuda_device):
    name, B, H, N, d, dv, dt = case
    q, k, v = random_qkv(B, H, N, d, dv, dtype=dt, scale=d ** -0.5, seed=N + 2)
    if clamp == "full":
        eps = 1e9
    else:
        fq, fk = _phi(q.double().numpy()), _phi(k.double().numpy())
        eps = float(np.median(np.einsum("bhnd,bhd->bhn", fq, fk.sum(2))))
    y, S, z = la.forward_noncausal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                   eps=eps, return_state=True, check_status=True)
    torch.cuda.synchronize()
    want = oracle.noncausal(q, k, v, eps=eps, return_state=True)
    _check((y, S, z), want, tol_for(dt), f"{name} eps={eps:.4g}")


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_decode_clamp(dt, cuda_device):
    """Decode steps from a prefilled state with eps above some (partly) and
    then all (fully) of the step denominators."""
    B, H, Np, d, dv = 2, 3, 64, 128, 128
    q, k, v = random_qkv(B, H, Np, d, dv, dtype=dt, scale=0.3, seed=5)
    _, So, zo = oracle.causal_recurrent(q, k, v, return_state=True)
    g = torch.Generator().manual_seed(6)
    for eps in (float(np.median(_phi(q[:, :, -1].double().numpy()) @ np.ones(d)) * Np), 1e9):
        S = torch.tensor(So, dtype=torch.float32, device=cuda_device)
        z = torch.tensor(zo, dtype=torch.float32, device=cuda_device)
        Sr, zr = So.copy(), zo.copy()
        for t in range(6):
            qs, ks, vs = ((torch.randn(B, H, n, generator=g) * 0.5).to(dt) for n in (d, d, dv))
            y = la.decode_step(qs.to(cuda_device), ks.to(cuda_device), vs.to(cuda_device), S, z,
                               eps=eps)
            yo, Sr, zr = oracle.decode_step(qs, ks, vs, Sr, zr, eps=eps)
            torch.cuda.synchronize()
            assert rel_max_err(y, yo) <= tol_for(dt), f"eps {eps:.4g} step {t}"
        assert rel_max_err(S, Sr) <= tol_for(dt) and rel_max_err(z, zr) <= tol_for(dt)


# decayed forward: heads on the tensor cores (gamma in [2^-1/2, 1]: the clamp
# becomes max(den', eps gamma^-(i+1)) per row there) and on the CUDA cores
DECAY_CASES = [
    ("tc_whole_heads", 2, 48, 300, 64, 64, (0.72, 0.9, 0.99, 1.0)),
    ("tc_split", 1, 4, 2000, 64, 64, (0.75, 0.9, 0.999, 1.0)),
    ("tc_whole_heads_d128", 1, 96, 260, 128, 128, (0.71, 0.8, 0.97, 0.9999)),
    ("cuda_cores", 1, 4, 500, 64, 128, (0.0, 0.3, 0.5, 0.7)),
]


@pytest.mark.parametrize("clamp", ["full", "partly"])
@pytest.mark.parametrize("case", DECAY_CASES, ids=lambda c: c[0])
def test_causal_decay_clamp(case, clamp, cuda_device):
    name, B, H, N, d, dv, gl = case
    gam = torch.tensor([gl[h % len(gl)] for h in range(H)], dtype=torch.float32)
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.bfloat16, scale=d ** -0.5, seed=N + 7)
    eps = 1e9 if clamp == "full" else float(np.median(causal_dens(q, k, gam)))
    y, S, z = la.forward_causal_decay(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                      gam.to(cuda_device), eps=eps, return_state=True,
                                      check_status=True)
    torch.cuda.synchronize()
    want = oracle.causal_recurrent_decay(q, k, v, gam, eps=eps, return_state=True)
    tol = TOL_F32 if name == "cuda_cores" else TOL_BF16
    _check((y, S, z), want, tol, f"{name} eps={eps:.4g}")


def test_decode_decay_clamp(cuda_device):
    B, H, Np, d, dv = 2, 4, 80, 64, 64
    gam = torch.tensor([0.0, 0.5, 0.9, 1.0])
    q, k, v = random_qkv(B, H, Np, d, dv, dtype=torch.bfloat16, scale=0.3, seed=8)
    _, So, zo = oracle.causal_recurrent_decay(q, k, v, gam, return_state=True)
    g = torch.Generator().manual_seed(9)
    for eps in (30.0, 1e9):
        S = torch.tensor(So, dtype=torch.float32, device=cuda_device)
        z = torch.tensor(zo, dtype=torch.float32, device=cuda_device)
        Sr, zr = So.copy(), zo.copy()
        for t in range(5):
            qs, ks, vs = ((torch.randn(B, H, n, generator=g) * 0.5).to(torch.bfloat16)
                          for n in (d, d, dv))
            y = la.decode_step_decay(qs.to(cuda_device), ks.to(cuda_device), vs.to(cuda_device),
                                     S, z, gam.to(cuda_device), eps=eps)
            # the oracle's decode is the recurrent form on one token from (Sr, zr)
            yo, Sr, zr = oracle.causal_recurrent_decay(qs[:, :, None], ks[:, :, None],
                                                       vs[:, :, None], gam, eps=eps, S_in=Sr,
                                                       z_in=zr, return_state=True)
            torch.cuda.synchronize()
            assert rel_max_err(y, yo[:, :, 0]) <= TOL_F32, f"eps {eps} step {t}"


# ---------------------------------------------------------------- input range
RANGE_DISTS = [("shifted_-4", 1.0, -4.0), ("scale_3", 3.0, 0.0)]

# The final state S of strongly shifted inputs: S = sum_j phi(k_j) v_j^T with
# lognormal phi(k) and random-sign v is a cancelling sum in which every key
# feature carries its bf16 rounding (2^-9 of |phi - c'|).  Rounding only the
# key features to bf16, with everything else exact, already moves the
# largest element of S by 1.5e-2 to 2e-2 of RMS(S) at 96 heads of N(-4, 1)
# draws, for any choice of c' (including 0); the kernels add their fp32 sums
# to that.  y and z stay within the bf16 bound.  float32 inputs (the CUDA-core
# kernels) are the route to a state within 1e-4 for such inputs.
TOL_STATE_SHIFTED = 4e-2


def _check_range(got, want, dist):
    tol_s = TOL_STATE_SHIFTED if dist.startswith("shifted") else TOL_BF16
    for name, g, w, tol in zip(("y", "S", "z"), got, want, (TOL_BF16, tol_s, TOL_BF16)):
        err = rel_max_err(g, w)
        assert err <= tol, f"{dist} {name}: {err:.3e}"


@pytest.mark.parametrize("dist", RANGE_DISTS, ids=lambda c: c[0])
@pytest.mark.parametrize("shape", [(2, 48, 300, 64, 64), (1, 2, 2000, 64, 128),
                                   (1, 96, 260, 128, 128)],
                         ids=["whole_heads", "split", "whole_heads_d128"])
def test_causal_tc_input_range(shape, dist, cuda_device):
    B, H, N, d, dv = shape
    _, scale, shift = dist
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.bfloat16, scale=scale, shift=shift,
                         seed=N + 11)
    y, S, z = la.forward_causal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                return_state=True, check_status=True)
    torch.cuda.synchronize()
    _check_range((y, S, z), oracle.causal_recurrent(q, k, v, return_state=True), dist[0])


@pytest.mark.parametrize("dist", RANGE_DISTS, ids=lambda c: c[0])
@pytest.mark.parametrize("shape", [(1, 3, 1000, 64, 64), (2, 2, 777, 128, 128)],
                         ids=["d64", "d128"])
def test_noncausal_tc_input_range(shape, dist, cuda_device):
    B, H, N, d, dv = shape
    _, scale, shift = dist
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.bfloat16, scale=scale, shift=shift,
                         seed=N + 12)
    y, S, z = la.forward_noncausal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                   return_state=True, check_status=True)
    torch.cuda.synchronize()
    _check_range((y, S, z), oracle.noncausal(q, k, v, return_state=True), dist[0])


@pytest.mark.parametrize("dist", RANGE_DISTS, ids=lambda c: c[0])
@pytest.mark.parametrize("shape", [(2, 48, 300, 64, 64), (1, 4, 2000, 64, 64)],
                         ids=["whole_heads", "split"])
def test_causal_decay_tc_input_range(shape, dist, cuda_device):
    B, H, N, d, dv = shape
    _, scale, shift = dist
    gl = (0.72, 0.9, 0.99, 1.0)
    gam = torch.tensor([gl[h % 4] for h in range(H)], dtype=torch.float32)
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.bfloat16, scale=scale, shift=shift,
                         seed=N + 13)
    y, S, z = la.forward_causal_decay(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                      gam.to(cuda_device), return_state=True, check_status=True)
    torch.cuda.synchronize()
    _check_range((y, S, z), oracle.causal_recurrent_decay(q, k, v, gam, return_state=True),
                 dist[0])


@pytest.mark.parametrize("dist", [("shifted_-8", 1.0, -8.0), ("heavy", 2.0, -3.0),
                                  ("scale_3", 3.0, 0.0)], ids=lambda c: c[0])
def test_float32_inputs_any_range(dist, cuda_device):
    """float32 inputs run on the fp32 CUDA-core kernels: the 1e-4 bound holds
    for inputs the bf16 scheme is not meant for."""
    _, scale, shift = dist
    q, k, v = random_qkv(1, 3, 600, 64, 64, dtype=torch.float32, scale=scale, shift=shift,
                         seed=14)
    y, S, z = la.forward_causal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                return_state=True)
    yn, Sn, zn = la.forward_noncausal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                      return_state=True)
    torch.cuda.synchronize()
    _check((y, S, z), oracle.causal_recurrent(q, k, v, return_state=True), TOL_F32, "causal")
    _check((yn, Sn, zn), oracle.noncausal(q, k, v, return_state=True), TOL_F32, "noncausal")


# ------------------------------------------------- decayed forward, in place
@pytest.mark.parametrize("shape", [(24, 4, 300, 64, 64), (1, 4, 2000, 64, 128)],
                         ids=["whole_heads", "split"])
def test_causal_decay_in_place_state(shape, cuda_device):
    """S_in aliased by S_out (and z_in by z_out) with heads on both kernels:
    the tensor-core kernel leaves the CUDA-core heads' state untouched, so
    every head continues from its own initial state."""
    B, H, N, d, dv = shape
    gam = torch.tensor([0.0, 0.3, 0.9, 1.0])
    q, k, v = random_qkv(B, H, N, d, dv, dtype=torch.bfloat16, scale=d ** -0.5, seed=N + 15)
    qp, kp, vp = random_qkv(B, H, 40, d, dv, dtype=torch.bfloat16, scale=0.3, seed=16)
    _, S_in, z_in = oracle.causal_recurrent_decay(qp, kp, vp, gam, return_state=True)
    S = _dev(S_in, cuda_device)
    z = _dev(z_in, cuda_device)
    y = la.forward_causal_decay(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                gam.to(cuda_device), S_in=S, z_in=z, S_out=S, z_out=z,
                                return_state=True, check_status=True)[0]
    torch.cuda.synchronize()
    yo, So, zo = oracle.causal_recurrent_decay(q, k, v, gam, S_in=S_in, z_in=z_in,
                                               return_state=True)
    for h in range(H):
        tol = TOL_F32 if float(gam[h]) < 2 ** -0.5 else TOL_BF16
        _check((y[:, h], S[:, h], z[:, h]), (yo[:, h], So[:, h], zo[:, h]), tol, f"head {h}")


# ------------------------------------------------ the kernels' feature function
def _bf16_all_finite():
    bits = np.arange(1 << 16, dtype=np.uint32)
    x = (bits << 16).view(np.float32)
    keep = np.isfinite(x)
    return bits[keep].astype(np.uint16), x[keep].astype(np.float64)


def _ulp_bf16(v):
    """Spacing of bf16 values at |v| (8 significant bits; subnormals 2^-133)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a >= 2.0 ** -126, 2.0 ** (e - 7), 2.0 ** -133)


def _feature_on_gpu(bits, c, dev):
    x = torch.from_numpy(bits.view(np.int16).copy()).to(dev)
    out = torch.empty_like(x)
    st = la.lib().la_debug_feature_bf16(x.data_ptr(), out.data_ptr(), x.numel(), float(c),
                                        la._stream_handle(None, dev))
    assert st == la.LA_OK
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    return got.view(np.float32).astype(np.float64)


def test_feature_function_is_elu_to_one_bf16_unit(cuda_device):
    """With c = 1 the residual the MMAs see is elu(x) = x (x > 0), e^x - 1
    (x <= 0): checked against numpy's expm1 in fp64 for every finite bf16
    input, including |x| < 1e-3, subnormal inputs and inputs whose e^x
    underflows; within one bf16 unit of the exact value."""
    bits, x = _bf16_all_finite()
    got = _feature_on_gpu(bits, 1.0, cuda_device)
    exact = np.where(x > 0, x, np.expm1(np.minimum(x, 0.0)))
    err = np.abs(got - exact)
    bad = err > _ulp_bf16(exact)
    assert not bad.any(), f"{bad.sum()} inputs, e.g. x={x[bad][:4]} got={got[bad][:4]} want={exact[bad][:4]}"
    assert got[x == 0].tolist() == [0.0] * int((x == 0).sum())


@pytest.mark.parametrize("c", [0.5, 0.03125, 0.0])
def test_feature_function_other_constants(c, cuda_device):
    """phi(x) - c for the constants of tokens with strongly negative features:
    within one bf16 unit plus the fp32 rounding of phi before the
    subtraction (and e^x below 2^-126 flushed to zero)."""
    bits, x = _bf16_all_finite()
    got = _feature_on_gpu(bits, c, cuda_device)
    phi = np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))
    exact = phi - c
    bound = _ulp_bf16(exact) + 2.0 ** -22 * phi + 2.0 ** -126
    bad = np.abs(got - exact) > bound
    assert not bad.any(), f"{bad.sum()} inputs, e.g. x={x[bad][:4]} got={got[bad][:4]} want={exact[bad][:4]}"
