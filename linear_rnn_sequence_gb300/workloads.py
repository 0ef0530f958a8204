"""Seeded synthetic workloads for kernelized linear attention.

This module only draws random inputs.  It holds none of the method's
arithmetic, so both the CUDA path's tests and the fp64 oracle can use it
without sharing any computation.

Recipe (one ``torch.Generator`` per workload): q, then k, then v are drawn
in that order as iid N(0, 1) float32 tensors of the full ``[B, H, N, d]`` /
``[B, H, N, dv]`` shape, multiplied by ``scale`` in float32, then cast to the
workload's input dtype (bf16 by round-to-nearest-even).  The decode workload
draws its prefill (unscaled) from a generator seeded ``seed`` and its per-step
q, k, v (scaled by 1/sqrt(d)) from a second generator seeded ``seed + 1``,
step after step, q then k then v.  The backward workload draws q, k, v as the
causal one does and then, from the same generator, the upstream gradient dy
as iid N(0, 1) float32 of shape ``[B, H, N, dv]`` (unscaled).  The decay
workloads draw as their plain counterparts and use one fixed decay per head,
gamma_h = 1 - 2^(-5 - 8 h / H): from 1 - 1/32 (a memory of about 32 tokens)
to about 1 - 2^-13, a spread of time scales across the heads.  The gated
workload draws as the causal one and then, from the same generator, one gate
per token (and per feature when asked), g = 1 - 2^-(2 + 11 u) with u ~ U(0, 1)
in float32: gates from 3/4 to 1 - 2^-13, spread evenly in their memory length.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    mode: str            # "causal" | "noncausal" | "decode" | "backward" | "causal_decay" | "decode_decay"
    B: int
    H: int
    N: int               # sequence length (decode: prefill length)
    d: int
    dv: int
    dtype: torch.dtype   # input dtype of q, k, v
    scale: float         # multiplier applied to the N(0,1) draws
    seed: int = 0
    eps: float = 1e-6
    steps: int = 0       # decode steps
    step_scale: float = 1.0

    @property
    def BH(self) -> int:
        return self.B * self.H

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    # fp32 causal, small enough for the oracle in well under a second.
    "causal_fp32_b1h2n256d32": Workload("causal_fp32_b1h2n256d32", "causal", 1, 2, 256, 32, 32,
                                        torch.float32, 1.0),
    # non-causal bf16.
    "noncausal_bf16_b4h8n4096d64": Workload("noncausal_bf16_b4h8n4096d64", "noncausal", 4, 8,
                                            4096, 64, 64, torch.bfloat16, 1.0 / math.sqrt(64)),
    # causal chunkwise, training / prefill shape.
    "causal_bf16_b8h16n8192d128": Workload("causal_bf16_b8h16n8192d128", "causal", 8, 16, 8192,
                                           128, 128, torch.bfloat16, 1.0 / math.sqrt(128)),
    # long-context causal.
    "causal_bf16_b1h32n131072d64": Workload("causal_bf16_b1h32n131072d64", "causal", 1, 32,
                                            131072, 64, 64, torch.bfloat16, 1.0 / math.sqrt(64)),
    # gradients of the causal form at the training shape.
    "causal_backward_bf16_b8h16n8192d128": Workload("causal_backward_bf16_b8h16n8192d128",
                                                    "backward", 8, 16, 8192, 128, 128,
                                                    torch.bfloat16, 1.0 / math.sqrt(128)),
    # causal with a per-head decay, training / prefill shape.
    "causal_decay_bf16_b8h16n8192d128": Workload("causal_decay_bf16_b8h16n8192d128",
                                                 "causal_decay", 8, 16, 8192, 128, 128,
                                                 torch.bfloat16, 1.0 / math.sqrt(128)),
    # long-context causal with a per-head decay (few heads: the sequence is split).
    "causal_decay_bf16_b1h32n131072d64": Workload("causal_decay_bf16_b1h32n131072d64",
                                                  "causal_decay", 1, 32, 131072, 64, 64,
                                                  torch.bfloat16, 1.0 / math.sqrt(64)),
    # recurrent decode with a per-head decay from a 1024-token prefill.
    "decode_decay_bf16_b256h32d128": Workload("decode_decay_bf16_b256h32d128", "decode_decay",
                                              256, 32, 1024, 128, 128, torch.bfloat16, 1.0,
                                              steps=4096, step_scale=1.0 / math.sqrt(128)),
    # gated causal (one gate per token and head), training / prefill shape.
    "causal_gated_bf16_b8h16n8192d128": Workload("causal_gated_bf16_b8h16n8192d128",
                                                 "causal_gated", 8, 16, 8192, 128, 128,
                                                 torch.bfloat16, 1.0 / math.sqrt(128)),
    # recurrent decode from a 1024-token prefill.
    "decode_bf16_b256h32d128": Workload("decode_bf16_b256h32d128", "decode", 256, 32, 1024, 128,
                                        128, torch.bfloat16, 1.0, steps=4096,
                                        step_scale=1.0 / math.sqrt(128)),
}


def _draw(gen: torch.Generator, shape, scale: float, dtype: torch.dtype, device) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=gen.device)
    if scale != 1.0:
        x = x * torch.tensor(scale, dtype=torch.float32, device=x.device)
    return x.to(dtype).to(device)


def make_qkv(w: Workload, device="cpu", gen_device="cpu"):
    """Draw (q, k, v) for a causal / non-causal workload, or the decode prefill.

    ``gen_device`` picks the generator's device; the same seed on a different
    generator device gives different (but equally seeded) numbers, so a test
    must compare against the oracle on the tensors this returns.
    """
    g = torch.Generator(device=gen_device)
    g.manual_seed(w.seed)
    q = _draw(g, (w.B, w.H, w.N, w.d), w.scale, w.dtype, device)
    k = _draw(g, (w.B, w.H, w.N, w.d), w.scale, w.dtype, device)
    v = _draw(g, (w.B, w.H, w.N, w.dv), w.scale, w.dtype, device)
    return q, k, v


def make_backward_inputs(w: Workload, device="cpu", gen_device="cpu"):
    """Draw (q, k, v, dy): q, k, v as ``make_qkv``, then dy from the same generator."""
    g = torch.Generator(device=gen_device)
    g.manual_seed(w.seed)
    q = _draw(g, (w.B, w.H, w.N, w.d), w.scale, w.dtype, device)
    k = _draw(g, (w.B, w.H, w.N, w.d), w.scale, w.dtype, device)
    v = _draw(g, (w.B, w.H, w.N, w.dv), w.scale, w.dtype, device)
    dy = _draw(g, (w.B, w.H, w.N, w.dv), 1.0, torch.float32, device)
    return q, k, v, dy


def head_decays(H: int) -> torch.Tensor:
    """The decay workloads' per-head gamma_h = 1 - 2^(-5 - 8 h / H) (float32, CPU)."""
    h = torch.arange(H, dtype=torch.float64)
    return (1.0 - torch.pow(2.0, -5.0 - 8.0 * h / H)).to(torch.float32)


def decode_step_generator(w: Workload, gen_device="cpu") -> torch.Generator:
    g = torch.Generator(device=gen_device)
    g.manual_seed(w.seed + 1)
    return g


def next_decode_inputs(w: Workload, g: torch.Generator, device=None):
    """Draw one decode step's (q, k, v): [B, H, d], [B, H, d], [B, H, dv]."""
    device = device if device is not None else g.device
    q = _draw(g, (w.B, w.H, w.d), w.step_scale, w.dtype, device)
    k = _draw(g, (w.B, w.H, w.d), w.step_scale, w.dtype, device)
    v = _draw(g, (w.B, w.H, w.dv), w.step_scale, w.dtype, device)
    return q, k, v


def random_qkv(B, H, N, d, dv, dtype=torch.float32, scale=1.0, seed=0, device="cpu",
               shift=0.0):
    """Ad-hoc seeded draw with the same recipe (for edge-case tests).

    With ``shift`` the draws of q and k are moved by that amount in float32
    before the cast (q, k ~ N(shift, scale^2), v ~ N(0, scale^2)), the inputs
    whose features phi are all far below 1 when the shift is strongly negative.
    """
    w = Workload("adhoc", "causal", B, H, N, d, dv, dtype, scale, seed)
    if shift == 0.0:
        return make_qkv(w, device=device)
    q, k, v = make_qkv(w.with_(dtype=torch.float32), device=device)
    sh = torch.tensor(shift, dtype=torch.float32)
    return (q + sh).to(dtype), (k + sh).to(dtype), v.to(dtype)


def random_qkv_dy(B, H, N, d, dv, dtype=torch.float32, scale=1.0, seed=0, device="cpu"):
    """Ad-hoc seeded (q, k, v, dy) draw with the backward recipe."""
    w = Workload("adhoc", "backward", B, H, N, d, dv, dtype, scale, seed)
    return make_backward_inputs(w, device=device)


def _gates(g: torch.Generator, shape, device) -> torch.Tensor:
    u = torch.rand(shape, generator=g, dtype=torch.float32, device=g.device)
    two = torch.tensor(2.0, dtype=torch.float32, device=u.device)
    return (1.0 - torch.pow(two, -(2.0 + 11.0 * u))).to(device)


def make_gated_inputs(w: Workload, gate_dim: int = 1, device="cpu", gen_device="cpu"):
    """Draw (q, k, v, gate): q, k, v as ``make_qkv``, then the gates from the same
    generator, [B, H, N] (gate_dim 1) or [B, H, N, d]."""
    g = torch.Generator(device=gen_device)
    g.manual_seed(w.seed)
    q = _draw(g, (w.B, w.H, w.N, w.d), w.scale, w.dtype, device)
    k = _draw(g, (w.B, w.H, w.N, w.d), w.scale, w.dtype, device)
    v = _draw(g, (w.B, w.H, w.N, w.dv), w.scale, w.dtype, device)
    shape = (w.B, w.H, w.N) if gate_dim == 1 else (w.B, w.H, w.N, w.d)
    return q, k, v, _gates(g, shape, device)


def random_gated(B, H, N, d, dv, gate_dim=1, dtype=torch.float32, scale=1.0, seed=0,
                 device="cpu", shift=0.0):
    """Ad-hoc seeded (q, k, v, gate) draw with the gated recipe (``shift`` as in
    ``random_qkv``)."""
    w = Workload("adhoc", "causal_gated", B, H, N, d, dv, torch.float32, scale, seed)
    q, k, v, gate = make_gated_inputs(w, gate_dim, device=device)
    sh = torch.tensor(shift, dtype=torch.float32)
    return (q + sh).to(dtype), (k + sh).to(dtype), v.to(dtype), gate


def random_projection(m: int, d: int, seed: int = 0) -> torch.Tensor:
    """W [m, d] with iid N(0, 1) rows (float32): the random projections of the
    random-feature map."""
    g = torch.Generator().manual_seed(seed)
    return torch.randn((m, d), generator=g, dtype=torch.float32)
