"""Failure path of the tensor-core kernels, tested without a GPU fault.

The test hook makes one work item's first tile copy never arrive (the copy is
announced on its mbarrier but not issued).  Every wait on that tile runs out
after a short limit, the kernel records LA_ERR_TIMEOUT in the workspace
header and its CTA unwinds.  Nothing traps or hangs, so the context stays
usable: the next call on the same device runs clean and matches the oracle.
"""
import pytest
import torch

import oracle
from linear_rnn_sequence_gb300 import linattn as la
from linear_rnn_sequence_gb300.workloads import random_qkv
from metrics import TOL_BF16, rel_max_err

pytestmark = pytest.mark.gpu

LIMIT_NS = 5_000_000   # 5 ms per bounded wait while the hook is on


@pytest.mark.parametrize("mode,H,N", [
    ("causal", 4, 1000),     # sequence split into segments: state + scan + chunk kernels
    ("causal", 96, 256),     # one CTA per head
    ("noncausal", 4, 1000),
    ("decay", 8, 600),       # decayed form: one CTA per head, then the CUDA-core pass
])
def test_dropped_copy_times_out_and_context_survives(mode, H, N, cuda_device):
    q, k, v = random_qkv(1, H, N, 64, 64, dtype=torch.bfloat16, scale=0.125, seed=H + N)
    qd, kd, vd = q.to(cuda_device), k.to(cuda_device), v.to(cuda_device)
    gam = torch.full((H,), 0.95)
    fn = {"causal": la.forward_causal, "noncausal": la.forward_noncausal,
          "decay": lambda *a, **kw: la.forward_causal_decay(*a, gam.to(cuda_device), **kw)}[mode]
    try:
        la.set_fault(drop_load_item=1, wait_limit_ns=LIMIT_NS)
        with pytest.raises(la.LinAttnError) as ei:
            fn(qd, kd, vd, check_status=True)
        assert ei.value.status == la.LA_ERR_TIMEOUT
    finally:
        la.set_fault(-1, 0)
    y = fn(qd, kd, vd, check_status=True)
    torch.cuda.synchronize()
    ref = {"causal": lambda: oracle.causal_recurrent(q, k, v),
           "noncausal": lambda: oracle.noncausal(q, k, v),
           "decay": lambda: oracle.causal_recurrent_decay(q, k, v, gam)}[mode]()
    assert rel_max_err(y, ref) <= TOL_BF16


def test_hook_off_by_default_and_limit_restored(cuda_device):
    la.set_fault(-1, 0)
    q, k, v = (t.to(cuda_device) for t in random_qkv(1, 2, 300, 128, 128,
                                                     dtype=torch.bfloat16, scale=0.09))
    la.forward_causal(q, k, v, check_status=True)
    la.forward_noncausal(q, k, v, check_status=True)
