"""The entry points can be captured in a CUDA graph.

Given a workspace, a call enqueues only kernel launches and a memset on the
caller's stream: no allocation, no host synchronisation, no host read of
device data.  A serving loop can therefore capture a layer's call once and
replay it.  These tests capture calls with torch's graph API (which captures
the current stream the binding passes), replay them, and require the same
bits as direct calls: every kernel involved is deterministic.  The direct
calls themselves are compared with the oracle elsewhere.
"""
import pytest
import torch

from linear_rnn_sequence_gb300 import linattn as la
from linear_rnn_sequence_gb300.workloads import random_qkv

pytestmark = pytest.mark.gpu


def _capture(fn):
    """Warm fn up on a side stream (as graph capture requires), then capture it."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


# (B, H, N): whole heads on the tensor cores, and few heads with a long
# sequence (segment states, prefix scan and chunk kernel, three launches)
@pytest.mark.parametrize("B,H,N,d,dv", [(2, 4, 777, 128, 128), (1, 2, 9001, 64, 64)])
def test_causal_call_replays_from_a_graph(B, H, N, d, dv, cuda_device):
    q, k, v = (t.to(cuda_device) for t in random_qkv(B, H, N, d, dv, dtype=torch.bfloat16,
                                                     scale=d ** -0.5, seed=N))
    ws = la.alloc_workspace(la.causal_workspace_bytes(B, H, N, d, dv, torch.bfloat16), cuda_device)
    want = la.forward_causal(q, k, v, workspace=ws)
    torch.cuda.synchronize()
    y = torch.empty_like(want)
    S = torch.empty(B, H, d, dv, device=cuda_device)
    z = torch.empty(B, H, d, device=cuda_device)
    g = _capture(lambda: la.forward_causal(q, k, v, out=y, S_out=S, z_out=z, workspace=ws))
    y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, want)
    _, S_want, z_want = la.forward_causal(q, k, v, workspace=ws, return_state=True)
    torch.cuda.synchronize()
    assert torch.equal(S, S_want) and torch.equal(z, z_want)
    assert la.workspace_header(ws)[0] == la.LA_OK


def test_noncausal_call_replays_from_a_graph(cuda_device):
    """The fused kernel's items meet through memory (a cooperative launch);
    the per-call clearing of its counters is captured with it."""
    B, H, N, d, dv = 2, 4, 3000, 64, 64
    q, k, v = (t.to(cuda_device) for t in random_qkv(B, H, N, d, dv, dtype=torch.bfloat16,
                                                     scale=0.125, seed=5))
    ws = la.alloc_workspace(la.noncausal_workspace_bytes(B, H, N, d, dv), cuda_device)
    want = la.forward_noncausal(q, k, v, workspace=ws)
    torch.cuda.synchronize()
    y = torch.empty_like(want)
    g = _capture(lambda: la.forward_noncausal(q, k, v, out=y, workspace=ws))
    for _ in range(3):   # replays reuse the counters: each must start from zero
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, want)
    assert la.workspace_header(ws)[0] == la.LA_OK


def test_decode_steps_replay_from_a_graph(cuda_device):
    """A decode step updates (S, z) in place, so two replays are two steps."""
    B, H, Np, d, dv = 2, 3, 200, 128, 128
    q, k, v = (t.to(cuda_device) for t in random_qkv(B, H, Np + 2, d, dv, dtype=torch.bfloat16,
                                                     scale=0.3, seed=9))
    _, S0, z0 = la.forward_causal(q[:, :, :Np].contiguous(), k[:, :, :Np].contiguous(),
                                  v[:, :, :Np].contiguous(), return_state=True)
    torch.cuda.synchronize()
    step = [tuple(t[:, :, Np + i].contiguous() for t in (q, k, v)) for i in range(2)]
    # direct: two steps
    S_d, z_d = S0.clone(), z0.clone()
    y_d = [la.decode_step(*step[i], S_d, z_d) for i in range(2)]
    torch.cuda.synchronize()
    # graphed: one captured step on fixed input buffers, replayed twice
    S_g, z_g = S0.clone(), z0.clone()
    qs, ks, vs = (t.clone() for t in step[0])
    y_g = torch.empty(B, H, dv, device=cuda_device)
    S_w, z_w = S_g.clone(), z_g.clone()   # warm-up and capture run on copies
    g = _capture(lambda: la.decode_step(qs, ks, vs, S_w, z_w, out=y_g))
    for i in range(2):
        for dst, src in zip((qs, ks, vs), step[i]):
            dst.copy_(src)
        S_w.copy_(S_g)
        z_w.copy_(z_g)
        g.replay()
        torch.cuda.synchronize()
        S_g.copy_(S_w)
        z_g.copy_(z_w)
        assert torch.equal(y_g, y_d[i]), f"step {i}"
    assert torch.equal(S_g, S_d) and torch.equal(z_g, z_d)
