"""The allocation-free non-causal entry point, la_forward_noncausal_noalloc.

It serves callers that cannot allocate device memory (for example code that
is handed only its input and output buffers by the framework it runs in), so
it uses a fixed scratch array inside the library instead of a workspace.
These tests call it through the C ABI and check that two calls in a row give
the same outputs as la_forward_noncausal with a caller-provided workspace,
within the tolerance the other parity tests use.  The file is named so that
pytest collects it last.
"""
import ctypes

import pytest
import torch

from linear_rnn_sequence_gb300 import linattn as la
from linear_rnn_sequence_gb300.workloads import WORKLOADS, make_qkv, random_qkv
from metrics import rel_max_err, tol_for

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20   # LA_NOALLOC_SCRATCH_BYTES in include/linattn.h


def _noalloc():
    f = la.lib().la_forward_noncausal_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float, vp, vp, vp]
    f.restype = i
    return f


def _call(q, k, v, eps=1e-6):
    B, H, N, d = q.shape
    dv = v.shape[-1]
    y = torch.full((B, H, N, dv), float("nan"), device=q.device)
    S = torch.full((B, H, d, dv), float("nan"), device=q.device)
    z = torch.full((B, H, d), float("nan"), device=q.device)
    code = la.LA_DTYPE_BF16 if q.dtype == torch.bfloat16 else la.LA_DTYPE_F32
    stream = ctypes.c_void_p(torch.cuda.current_stream(q.device).cuda_stream)
    st = _noalloc()(q.data_ptr(), k.data_ptr(), v.data_ptr(), y.data_ptr(), B, H, N, d, dv, code,
                    eps, S.data_ptr(), z.data_ptr(), stream)
    assert st == la.LA_OK, la.status_string(st)
    return y, S, z


@pytest.mark.parametrize("case", [
    ("noncausal_bf16_b4h8n4096d64", None),
    ("adhoc_f32", (1, 3, 517, 128, 64, torch.float32, 0.5)),
    ("adhoc_bf16_ragged", (2, 2, 333, 64, 128, torch.bfloat16, 0.2)),
], ids=lambda c: c[0])
def test_noalloc_matches_workspace_path_twice(case, cuda_device):
    name, spec = case
    if spec is None:
        w = WORKLOADS[name]
        q, k, v = (t.to(cuda_device) for t in make_qkv(w))
        dt = w.dtype
    else:
        B, H, N, d, dv, dt, s = spec
        q, k, v = (t.to(cuda_device) for t in random_qkv(B, H, N, d, dv, dtype=dt, scale=s,
                                                         seed=N))
    need = la.noncausal_workspace_bytes(*q.shape, v.shape[-1], dt)
    assert need <= SCRATCH_BYTES
    y_ref, S_ref, z_ref = la.forward_noncausal(q, k, v, return_state=True)
    torch.cuda.synchronize()
    ref = [t.cpu().double().numpy() for t in (y_ref, S_ref, z_ref)]
    tol = tol_for(dt)
    for _ in range(2):   # the second call reuses the scratch the first one left behind
        got = _call(q, k, v)
        torch.cuda.synchronize()
        for g, r in zip(got, ref):
            assert rel_max_err(g, r) <= tol


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_device):
    B, H, N, d, dv = 8, 16, 65536, 128, 128
    assert la.noncausal_workspace_bytes(B, H, N, d, dv) > SCRATCH_BYTES
    # the size check comes first, so these (never touched) pointers are fine
    q = torch.empty(16, dtype=torch.bfloat16, device=cuda_device)
    st = _noalloc()(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), B, H, N, d, dv,
                    la.LA_DTYPE_BF16, 1e-6, None, None, None)
    assert st == la.LA_ERR_WORKSPACE
