"""The allocation-free non-causal entry point, la_forward_noncausal_noalloc.

It serves callers that cannot allocate device memory (for example code that
is handed only its input and output buffers by the framework it runs in), so
it uses a fixed scratch array inside the library instead of a workspace.
These tests call it through the C ABI and check, on two calls in a row, its
outputs against the fp64 oracle (the bound the other parity tests use) and
against la_forward_noncausal with a caller-provided workspace; that sizes
beyond the scratch are rejected; and that a bounded wait that runs out is
reported through la_noalloc_status, after which a clean call is correct
again.  The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import oracle
from linear_rnn_sequence_gb300 import linattn as la
from linear_rnn_sequence_gb300.workloads import WORKLOADS, make_qkv, random_qkv
from metrics import rel_max_err, tol_for

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20   # LA_NOALLOC_SCRATCH_BYTES in include/linattn.h


def _stream(dev):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _call(q, k, v, eps=1e-6):
    B, H, N, d = q.shape
    dv = v.shape[-1]
    y = torch.full((B, H, N, dv), float("nan"), device=q.device)
    S = torch.full((B, H, d, dv), float("nan"), device=q.device)
    z = torch.full((B, H, d), float("nan"), device=q.device)
    code = la.LA_DTYPE_BF16 if q.dtype == torch.bfloat16 else la.LA_DTYPE_F32
    st = la.lib().la_forward_noncausal_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                               y.data_ptr(), B, H, N, d, dv, code, eps,
                                               S.data_ptr(), z.data_ptr(), _stream(q.device))
    assert st == la.LA_OK, la.status_string(st)
    return y, S, z


def _status(dev):
    return la.lib().la_noalloc_status(_stream(dev))


CASES = [
    ("noncausal_bf16_b4h8n4096d64", None),
    ("adhoc_f32", (1, 3, 517, 128, 64, torch.float32, 0.5)),
    ("adhoc_bf16_ragged", (2, 2, 333, 64, 128, torch.bfloat16, 0.2)),
]


def _inputs(case, dev):
    name, spec = case
    if spec is None:
        w = WORKLOADS[name]
        q, k, v = make_qkv(w)
        return q, k, v, w.dtype
    B, H, N, d, dv, dt, s = spec
    q, k, v = random_qkv(B, H, N, d, dv, dtype=dt, scale=s, seed=N)
    return q, k, v, dt


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_noalloc_matches_oracle_twice(case, cuda_device):
    q, k, v, dt = _inputs(case, cuda_device)
    need = la.noncausal_workspace_bytes(*q.shape, v.shape[-1], dt)
    assert need <= SCRATCH_BYTES
    want = oracle.noncausal(q, k, v, return_state=True)
    qd, kd, vd = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device)
    y_ws, S_ws, z_ws = la.forward_noncausal(qd, kd, vd, return_state=True)
    tol = tol_for(dt)
    for _ in range(2):   # the second call reuses the scratch the first one left behind
        got = _call(qd, kd, vd)
        assert _status(cuda_device) == la.LA_OK
        for g, w in zip(got, want):
            assert rel_max_err(g, w) <= tol
        # the same kernels as the workspace entry point, in the same order
        for g, w in zip(got, (y_ws, S_ws, z_ws)):
            assert torch.equal(g, w)


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_device):
    B, H, N, d, dv = 64, 16, 4096, 128, 128   # 1024 heads: their partial states exceed it
    assert la.noncausal_workspace_bytes(B, H, N, d, dv) > SCRATCH_BYTES
    # the size check comes first, so these (never touched) pointers are fine
    q = torch.empty(16, dtype=torch.bfloat16, device=cuda_device)
    st = la.lib().la_forward_noncausal_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(),
                                               q.data_ptr(), B, H, N, d, dv, la.LA_DTYPE_BF16,
                                               1e-6, None, None, None)
    assert st == la.LA_ERR_WORKSPACE


def test_noalloc_reports_a_timed_out_wait(cuda_device):
    """The host-side hook makes one query item's first tile copy never arrive
    (nothing faults or hangs: the wait gives up after 5 ms); the status query
    reports it, and the next clean call matches the oracle again."""
    q, k, v = random_qkv(1, 2, 1000, 64, 64, dtype=torch.bfloat16, scale=0.125, seed=3)
    qd, kd, vd = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device)
    try:
        la.set_fault(drop_load_item=1, wait_limit_ns=5_000_000)
        _call(qd, kd, vd)
        assert _status(cuda_device) == la.LA_ERR_TIMEOUT
    finally:
        la.set_fault(-1, 0)
    got = _call(qd, kd, vd)
    assert _status(cuda_device) == la.LA_OK
    for g, w in zip(got, oracle.noncausal(q, k, v, return_state=True)):
        assert rel_max_err(g, w) <= tol_for(torch.bfloat16)
