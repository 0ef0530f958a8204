"""Full-size workloads against the fp64 oracle, in the launch configuration the
benchmark times.  Where the oracle cannot cover every head in seconds, it runs
on a fixed sample of heads and the GPU output for exactly those heads is
compared element by element (outputs and final state)."""
import numpy as np
import pytest
import torch

import oracle
from linear_rnn_sequence_gb300 import linattn as la
from linear_rnn_sequence_gb300.workloads import (WORKLOADS, decode_step_generator, make_qkv,
                                                 next_decode_inputs)
from metrics import rel_max_err, tol_for

pytestmark = pytest.mark.gpu


def _heads(BH, n):
    if n >= BH:
        return list(range(BH))
    return sorted(set(int(round(x)) for x in np.linspace(0, BH - 1, n)))


def _flat(t):
    return t.reshape(-1, *t.shape[2:])


@pytest.mark.parametrize("name,nsample", [
    ("causal_fp32_b1h2n256d32", 2),
    ("causal_bf16_b8h16n8192d128", 4),
    ("causal_bf16_b1h32n131072d64", 2),
])
def test_causal_workload(name, nsample, cuda_device):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w)
    y, S, z = la.forward_causal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                eps=w.eps, return_state=True, check_status=True)
    torch.cuda.synchronize()
    hs = _heads(w.BH, nsample)
    yo, So, zo = oracle.causal_recurrent(_flat(q)[hs], _flat(k)[hs], _flat(v)[hs], eps=w.eps,
                                         return_state=True)
    tol = tol_for(w.dtype)
    e_y = rel_max_err(_flat(y)[hs], yo)
    e_S = rel_max_err(_flat(S)[hs], So)
    e_z = rel_max_err(_flat(z)[hs], zo)
    print(f"{name}: y {e_y:.3e} S {e_S:.3e} z {e_z:.3e}")
    assert e_y <= tol and e_S <= tol and e_z <= tol


def test_noncausal_workload(cuda_device):
    w = WORKLOADS["noncausal_bf16_b4h8n4096d64"]
    q, k, v = make_qkv(w)
    y, S, z = la.forward_noncausal(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                                   eps=w.eps, return_state=True)
    torch.cuda.synchronize()
    yo, So, zo = oracle.noncausal(q, k, v, eps=w.eps, return_state=True)
    e = (rel_max_err(y, yo), rel_max_err(S, So), rel_max_err(z, zo))
    print("noncausal:", e)
    assert max(e) <= tol_for(w.dtype)


def test_decode_workload(cuda_device):
    """Prefill 1024 tokens per sequence, then every one of the 4096 steps is
    checked on a sample of 16 heads, and the final state at the end."""
    w = WORKLOADS["decode_bf16_b256h32d128"]
    hs = _heads(w.BH, 16)
    idx = torch.tensor(hs, device=cuda_device)
    q, k, v = make_qkv(w, device=cuda_device, gen_device=cuda_device)
    _, S, z = la.forward_causal(q, k, v, eps=w.eps, return_state=True, check_status=True)
    qh, kh, vh = (_flat(t).index_select(0, idx).cpu() for t in (q, k, v))
    del q, k, v
    torch.cuda.synchronize()
    _, So, zo = oracle.causal_recurrent(qh, kh, vh, eps=w.eps, return_state=True)
    assert rel_max_err(_flat(S).index_select(0, idx), So) <= tol_for(w.dtype)

    g = decode_step_generator(w, gen_device=cuda_device)
    T = w.steps
    yh = torch.empty(T, len(hs), w.dv, device=cuda_device)
    ins = [torch.empty(T, len(hs), n, dtype=w.dtype, device=cuda_device) for n in (w.d, w.d, w.dv)]
    ybuf = torch.empty(w.B, w.H, w.dv, device=cuda_device)
    for t in range(T):
        qs, ks, vs = next_decode_inputs(w, g)
        la.decode_step(qs, ks, vs, S, z, eps=w.eps, out=ybuf)
        yh[t] = ybuf.view(-1, w.dv).index_select(0, idx)
        for buf, x in zip(ins, (qs, ks, vs)):
            buf[t] = x.view(-1, x.shape[-1]).index_select(0, idx)
    torch.cuda.synchronize()
    yh = yh.cpu().double().numpy()
    qs_h, ks_h, vs_h = (b.cpu() for b in ins)
    worst = 0.0
    for t in range(T):
        yo, So, zo = oracle.decode_step(qs_h[t], ks_h[t], vs_h[t], So, zo, eps=w.eps)
        e = rel_max_err(yh[t], yo)
        worst = max(worst, e)
        assert e <= tol_for(w.dtype), f"step {t}: {e}"
    eS = rel_max_err(_flat(S).index_select(0, idx), So)
    ez = rel_max_err(_flat(z).index_select(0, idx), zo)
    print(f"decode: worst step {worst:.3e}, final S {eS:.3e}, z {ez:.3e}")
    assert eS <= tol_for(w.dtype) and ez <= tol_for(w.dtype)
