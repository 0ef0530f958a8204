"""ctypes binding of liblinattn.so (C ABI: include/linattn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C entry points.  Tensors must be contiguous CUDA tensors;
outputs and workspaces are allocated here with torch (the library allocates
nothing).  There is no CPU fallback: a missing or unbuildable library raises.

Names follow the C ABI:

* ``forward_causal``    -> ``la_forward_causal``
* ``forward_noncausal`` -> ``la_forward_noncausal``
* ``decode_step``       -> ``la_decode_step``
* ``forward_causal_gated``, ``decode_step_gated``, ``forward_noncausal_phi``,
  ``random_features`` -> the gated and feature-map entry points
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_TIMEOUT, LA_ERR_WORKSPACE = range(6)
LA_DTYPE_F32, LA_DTYPE_BF16 = 0, 1
PHI = {"elu1": 0, "identity": 1}   # la_phi

_lock = threading.Lock()
_lib = None


class LinAttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB


def lib():
    """Load (building first if the sources are newer) and return the ctypes library."""
    global _lib
    with _lock:
        if _lib is None:
            if _build.is_stale():
                _build.build()
            if not os.path.exists(_build.LIB):
                raise RuntimeError(f"liblinattn.so missing at {_build.LIB}")
            L = ctypes.CDLL(_build.LIB)
            vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            L.la_status_string.argtypes = [i]
            L.la_status_string.restype = ctypes.c_char_p
            L.la_version.argtypes = []
            L.la_version.restype = ctypes.c_char_p
            L.la_causal_workspace_bytes.argtypes = [i, i, i, i, i, i]
            L.la_causal_workspace_bytes.restype = sz
            L.la_noncausal_workspace_bytes.argtypes = [i, i, i, i, i, i]
            L.la_noncausal_workspace_bytes.restype = sz
            L.la_forward_causal.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, vp, vp, vp, vp,
                                            vp, sz, vp]
            L.la_forward_causal.restype = i
            L.la_forward_noncausal.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, vp, vp, vp,
                                               sz, vp]
            L.la_forward_noncausal.restype = i
            L.la_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
            L.la_decode_step.restype = i
            L.la_causal_host_buffer_bytes.argtypes = [i, i, i, i, i, i]
            L.la_causal_host_buffer_bytes.restype = sz
            L.la_forward_causal_host.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, vp, vp, vp,
                                                 sz, vp]
            L.la_forward_causal_host.restype = i
            L.la_forward_causal_decay.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, vp, vp, vp,
                                                  vp, vp, vp, sz, vp]
            L.la_forward_causal_decay.restype = i
            L.la_decode_step_decay.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, vp]
            L.la_decode_step_decay.restype = i
            L.la_causal_backward_workspace_bytes.argtypes = [i, i, i, i, i, i]
            L.la_causal_backward_workspace_bytes.restype = sz
            L.la_backward_causal.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f,
                                             vp, vp, vp, vp, vp, sz, vp]
            L.la_backward_causal.restype = i
            L.la_backward_causal_decay.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                                   f, vp, vp, vp, vp, vp, vp, sz, vp]
            L.la_backward_causal_decay.restype = i
            L.la_workspace_status.argtypes = [vp, sz, vp]
            L.la_workspace_status.restype = i
            L.la_debug_set_fault.argtypes = [i, ctypes.c_longlong]
            L.la_debug_set_fault.restype = None
            L.la_debug_feature_bf16.argtypes = [vp, vp, ctypes.c_longlong, f, vp]
            L.la_debug_feature_bf16.restype = i
            L.la_forward_noncausal_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, vp,
                                                       vp, vp]
            L.la_forward_noncausal_noalloc.restype = i
            L.la_noalloc_status.argtypes = [vp]
            L.la_noalloc_status.restype = i
            L.la_forward_causal_gated.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, i,
                                                  vp, vp, vp, vp, vp, sz, vp]
            L.la_forward_causal_gated.restype = i
            L.la_causal_gated_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
            L.la_causal_gated_workspace_bytes.restype = sz
            L.la_decode_step_gated.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i,
                                               vp]
            L.la_decode_step_gated.restype = i
            L.la_noncausal_phi_workspace_bytes.argtypes = [i, i, i, i, i, i, i]
            L.la_noncausal_phi_workspace_bytes.restype = sz
            L.la_forward_noncausal_phi.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, vp,
                                                   vp, sz, vp]
            L.la_forward_noncausal_phi.restype = i
            L.la_random_features.argtypes = [vp, vp, ctypes.c_longlong, i, i, i, vp, vp]
            L.la_random_features.restype = i
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().la_status_string(int(status)).decode()


def version() -> str:
    return lib().la_version().decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return LA_DTYPE_BF16
    if t.dtype == torch.float32:
        return LA_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}; use bfloat16 or float32")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream, device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _check_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must be CUDA tensors (no CPU fallback)")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _raise(st: int, where: str):
    if st != LA_OK:
        raise LinAttnError(st, where)


def causal_workspace_bytes(B, H, N, d, dv, dtype=torch.bfloat16) -> int:
    code = LA_DTYPE_BF16 if dtype == torch.bfloat16 else LA_DTYPE_F32
    return int(lib().la_causal_workspace_bytes(B, H, N, d, dv, code))


def noncausal_workspace_bytes(B, H, N, d, dv, dtype=torch.bfloat16) -> int:
    code = LA_DTYPE_BF16 if dtype == torch.bfloat16 else LA_DTYPE_F32
    return int(lib().la_noncausal_workspace_bytes(B, H, N, d, dv, code))


def alloc_workspace(nbytes: int, device) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    # torch's caching allocator returns blocks aligned to at least 512 bytes
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def forward_causal(q, k, v, eps: float = 1e-6, S_in=None, z_in=None, return_state=False,
                   out=None, S_out=None, z_out=None, workspace=None, stream=None,
                   check_status=False):
    """Causal elu+1 linear attention.  q, k: [B,H,N,d]; v: [B,H,N,dv] (bf16 or fp32).

    Returns y [B,H,N,dv] float32 (and the final (S, z) when ``return_state``).
    With ``check_status`` the call synchronises and raises if a kernel recorded
    a run-time error (a bounded wait that ran out) in the workspace.
    """
    _check_cuda(q, k, v, S_in, z_in, out, S_out, z_out, workspace)
    B, H, N, d = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v shapes / dtypes disagree")
    y = out if out is not None else torch.empty((B, H, N, dv), dtype=torch.float32, device=q.device)
    if return_state and S_out is None:
        S_out = torch.empty((B, H, d, dv), dtype=torch.float32, device=q.device)
        z_out = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    need = int(lib().la_causal_workspace_bytes(B, H, N, d, dv, dt))
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().la_forward_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(y), B, H, N, d, dv, dt,
                                 float(eps), _ptr(S_in), _ptr(z_in), _ptr(S_out), _ptr(z_out),
                                 _ptr(workspace), wbytes, _stream_handle(stream, q.device))
    _raise(st, "la_forward_causal")
    if check_status and workspace is not None:
        err, where = workspace_header(workspace)
        if err != LA_OK:
            raise LinAttnError(err, f"la_forward_causal (run time, wait site {where})")
    return (y, S_out, z_out) if return_state else y


def forward_causal_decay(q, k, v, gamma, eps: float = 1e-6, S_in=None, z_in=None,
                         return_state=False, out=None, S_out=None, z_out=None, workspace=None,
                         stream=None, check_status=False):
    """Causal attention with a per-head decay ``gamma`` (float32 CUDA tensor [H]).

    q, k: [B,H,N,d]; v: [B,H,N,dv].  Returns y [B,H,N,dv] float32 (and the
    final (S, z) when ``return_state``).  The workspace and ``check_status``
    are as in ``forward_causal``.
    """
    _check_cuda(q, k, v, gamma, S_in, z_in, out, S_out, z_out, workspace)
    B, H, N, d = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v shapes / dtypes disagree")
    if gamma.shape != (H,) or gamma.dtype != torch.float32:
        raise ValueError("gamma must be a float32 tensor of shape [H]")
    y = out if out is not None else torch.empty((B, H, N, dv), dtype=torch.float32, device=q.device)
    if return_state and S_out is None:
        S_out = torch.empty((B, H, d, dv), dtype=torch.float32, device=q.device)
        z_out = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    need = int(lib().la_causal_workspace_bytes(B, H, N, d, dv, dt))
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().la_forward_causal_decay(_ptr(q), _ptr(k), _ptr(v), _ptr(y), B, H, N, d, dv, dt,
                                       float(eps), _ptr(gamma), _ptr(S_in), _ptr(z_in),
                                       _ptr(S_out), _ptr(z_out), _ptr(workspace), wbytes,
                                       _stream_handle(stream, q.device))
    _raise(st, "la_forward_causal_decay")
    if check_status and workspace is not None:
        err, where = workspace_header(workspace)
        if err != LA_OK:
            raise LinAttnError(err, f"la_forward_causal_decay (run time, wait site {where})")
    return (y, S_out, z_out) if return_state else y


def decode_step_decay(q, k, v, S, z, gamma, eps: float = 1e-6, out=None, stream=None):
    """One decode step with decay; S and z are updated in place.  Returns y."""
    _check_cuda(q, k, v, S, z, gamma, out)
    B, H, d = q.shape
    dv = v.shape[-1]
    if gamma.shape != (H,) or gamma.dtype != torch.float32:
        raise ValueError("gamma must be a float32 tensor of shape [H]")
    y = out if out is not None else torch.empty((B, H, dv), dtype=torch.float32, device=q.device)
    st = lib().la_decode_step_decay(_ptr(q), _ptr(k), _ptr(v), _ptr(y), _ptr(S), _ptr(z), B, H,
                                    d, dv, _dtype_code(q), float(eps), _ptr(gamma),
                                    _stream_handle(stream, q.device))
    _raise(st, "la_decode_step_decay")
    return y


def causal_backward_workspace_bytes(B, H, N, d, dv, dtype=torch.bfloat16) -> int:
    code = LA_DTYPE_BF16 if dtype == torch.bfloat16 else LA_DTYPE_F32
    return int(lib().la_causal_backward_workspace_bytes(B, H, N, d, dv, code))


def backward_causal(q, k, v, dy, eps: float = 1e-6, S_in=None, z_in=None,
                    return_state_grad=False, out=None, workspace=None, stream=None, gamma=None):
    """Gradients of the causal forward for the upstream gradient ``dy``.

    q, k: [B,H,N,d]; v: [B,H,N,dv] (bf16 or fp32); dy: [B,H,N,dv] float32.
    With ``gamma`` (float32 CUDA tensor [H]) the gradients are those of the
    decayed forward (``forward_causal_decay``).
    Returns (dq, dk, dv) float32, plus (dS_in, dz_in) when ``return_state_grad``.
    ``out`` may be a preallocated (dq, dk, dv) triple.
    """
    _check_cuda(q, k, v, dy, S_in, z_in, workspace, gamma)
    B, H, N, d = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v shapes / dtypes disagree")
    if dy.shape != v.shape or dy.dtype != torch.float32:
        raise ValueError("dy must be float32 with the shape of v")
    if out is None:
        out = (torch.empty((B, H, N, d), dtype=torch.float32, device=q.device),
               torch.empty((B, H, N, d), dtype=torch.float32, device=q.device),
               torch.empty((B, H, N, dv), dtype=torch.float32, device=q.device))
    gq, gk, gv = out
    _check_cuda(gq, gk, gv)
    gS = gz = None
    if return_state_grad:
        gS = torch.empty((B, H, d, dv), dtype=torch.float32, device=q.device)
        gz = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    need = int(lib().la_causal_backward_workspace_bytes(B, H, N, d, dv, dt))
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if gamma is None:
        st = lib().la_backward_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(gq), _ptr(gk),
                                      _ptr(gv), B, H, N, d, dv, dt, float(eps), _ptr(S_in),
                                      _ptr(z_in), _ptr(gS), _ptr(gz), _ptr(workspace), wbytes,
                                      _stream_handle(stream, q.device))
        _raise(st, "la_backward_causal")
    else:
        if gamma.shape != (H,) or gamma.dtype != torch.float32:
            raise ValueError("gamma must be a float32 tensor of shape [H]")
        st = lib().la_backward_causal_decay(_ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(gq),
                                            _ptr(gk), _ptr(gv), B, H, N, d, dv, dt, float(eps),
                                            _ptr(gamma), _ptr(S_in), _ptr(z_in), _ptr(gS),
                                            _ptr(gz), _ptr(workspace), wbytes,
                                            _stream_handle(stream, q.device))
        _raise(st, "la_backward_causal_decay")
    return (gq, gk, gv, gS, gz) if return_state_grad else (gq, gk, gv)


def causal_host_buffer_bytes(B, H, N, d, dv, dtype=torch.bfloat16) -> int:
    code = LA_DTYPE_BF16 if dtype == torch.bfloat16 else LA_DTYPE_F32
    return int(lib().la_causal_host_buffer_bytes(B, H, N, d, dv, code))


def forward_causal_host(q, k, v, eps: float = 1e-6, return_state=False, out=None, S_out=None,
                        z_out=None, dev_buf=None, device=None, stream=None):
    """Causal forward on host (CPU) tensors through la_forward_causal_host.

    q, k: [B,H,N,d]; v: [B,H,N,dv] CPU tensors (bf16 or fp32; page-locked
    memory makes the copies overlap).  Returns y [B,H,N,dv] float32 on the CPU
    (and the final (S, z) when ``return_state``).  ``dev_buf`` is the device
    staging memory (allocated on ``device`` when not given).
    """
    for t in (q, k, v, out, S_out, z_out):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise ValueError("forward_causal_host takes contiguous CPU tensors")
    B, H, N, d = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v shapes / dtypes disagree")
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    y = out if out is not None else torch.empty((B, H, N, dv), dtype=torch.float32)
    if return_state and S_out is None:
        S_out = torch.empty((B, H, d, dv), dtype=torch.float32)
        z_out = torch.empty((B, H, d), dtype=torch.float32)
    if dev_buf is None:
        dev_buf = alloc_workspace(int(lib().la_causal_host_buffer_bytes(B, H, N, d, dv, dt)), dev)
    nbytes = 0 if dev_buf is None else dev_buf.numel() * dev_buf.element_size()
    st = lib().la_forward_causal_host(_ptr(q), _ptr(k), _ptr(v), _ptr(y), B, H, N, d, dv, dt,
                                      float(eps), _ptr(S_out), _ptr(z_out), _ptr(dev_buf), nbytes,
                                      _stream_handle(stream, dev))
    _raise(st, "la_forward_causal_host")
    return (y, S_out, z_out) if return_state else y


def forward_noncausal(q, k, v, eps: float = 1e-6, return_state=False, out=None, S_out=None,
                      z_out=None, workspace=None, stream=None, check_status=False):
    """Non-causal elu+1 linear attention.  Returns y [B,H,N,dv] float32 (+ S, z).

    ``check_status`` as for :func:`forward_causal`.
    """
    _check_cuda(q, k, v, out, S_out, z_out, workspace)
    B, H, N, d = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v shapes / dtypes disagree")
    y = out if out is not None else torch.empty((B, H, N, dv), dtype=torch.float32, device=q.device)
    if return_state and S_out is None:
        S_out = torch.empty((B, H, d, dv), dtype=torch.float32, device=q.device)
        z_out = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    need = int(lib().la_noncausal_workspace_bytes(B, H, N, d, dv, dt))
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().la_forward_noncausal(_ptr(q), _ptr(k), _ptr(v), _ptr(y), B, H, N, d, dv, dt,
                                    float(eps), _ptr(S_out), _ptr(z_out), _ptr(workspace), wbytes,
                                    _stream_handle(stream, q.device))
    _raise(st, "la_forward_noncausal")
    if check_status and workspace is not None:
        err, where = workspace_header(workspace)
        if err != LA_OK:
            raise LinAttnError(err, f"la_forward_noncausal (run time, wait site {where})")
    return (y, S_out, z_out) if return_state else y


def decode_step(q, k, v, S, z, eps: float = 1e-6, out=None, stream=None):
    """One decode step in place on (S, z).  q, k: [B,H,d]; v: [B,H,dv]; returns y [B,H,dv] fp32."""
    _check_cuda(q, k, v, S, z, out)
    B, H, d = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    if S.dtype != torch.float32 or z.dtype != torch.float32:
        raise TypeError("state must be float32")
    if S.shape != (B, H, d, dv) or z.shape != (B, H, d):
        raise ValueError("state shape mismatch")
    y = out if out is not None else torch.empty((B, H, dv), dtype=torch.float32, device=q.device)
    st = lib().la_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(y), _ptr(S), _ptr(z), B, H, d, dv,
                              dt, float(eps), _stream_handle(stream, q.device))
    _raise(st, "la_decode_step")
    return y


def workspace_status(workspace, stream=None) -> int:
    """Synchronise and return the run-time status recorded in ``workspace``."""
    if workspace is None:
        return LA_OK
    return int(lib().la_workspace_status(_ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         _stream_handle(stream, workspace.device)))


def workspace_header(workspace) -> tuple[int, int]:
    """(error word, diagnostic word) recorded in a workspace header (synchronises)."""
    torch.cuda.synchronize(workspace.device)
    h = workspace[:8].cpu().view(torch.int32)
    return int(h[0]), int(h[1])


def set_fault(drop_load_item: int = -1, wait_limit_ns: int = 0) -> None:
    """Test hook: see la_debug_set_fault in include/linattn.h."""
    lib().la_debug_set_fault(int(drop_load_item), int(wait_limit_ns))

def _gate_dim(gate, lead, d):
    """gate_dim of a gate tensor whose leading shape is ``lead`` (1 or d)."""
    if gate is None:
        return 1
    if gate.dtype != torch.float32:
        raise TypeError("gate must be float32")
    if tuple(gate.shape) == tuple(lead):
        return 1
    if tuple(gate.shape) == tuple(lead) + (d,):
        return d
    raise ValueError(f"gate shape {tuple(gate.shape)} must be {tuple(lead)} or {tuple(lead) + (d,)}")


def causal_gated_workspace_bytes(B, H, N, d, dv, dtype=torch.bfloat16, phi="elu1",
                                 gate_dim=1) -> int:
    code = LA_DTYPE_BF16 if dtype == torch.bfloat16 else LA_DTYPE_F32
    return int(lib().la_causal_gated_workspace_bytes(B, H, N, d, dv, code, PHI[phi], gate_dim))


def forward_causal_gated(q, k, v, gate=None, phi="elu1", eps: float = 1e-6, S_in=None,
                         z_in=None, return_state=False, out=None, S_out=None, z_out=None,
                         workspace=None, stream=None, check_status=False):
    """Gated causal attention.  gate: None, [B,H,N] or [B,H,N,d] float32; phi:
    "elu1" or "identity".  bf16 inputs with d, dv in {64, 128}, one gate per
    token and elu + 1 run on the tensor cores (heads whose gates all lie in
    [2^-1/2, 1]); everything else in fp32 on the CUDA cores.  Returns y (and the
    final (S, z)); ``check_status`` as for :func:`forward_causal`."""
    _check_cuda(q, k, v, gate, S_in, z_in, out, S_out, z_out, workspace)
    B, H, N, d = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    if k.shape != q.shape or v.shape[:3] != q.shape[:3] or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v shapes / dtypes disagree")
    gd = _gate_dim(gate, (B, H, N), d)
    y = out if out is not None else torch.empty((B, H, N, dv), dtype=torch.float32, device=q.device)
    if return_state and S_out is None:
        S_out = torch.empty((B, H, d, dv), dtype=torch.float32, device=q.device)
        z_out = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    need = (causal_gated_workspace_bytes(B, H, N, d, dv, q.dtype, phi, gd) if gate is not None
            else 256)
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    st = lib().la_forward_causal_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(y), B, H, N, d, dv, dt,
                                       float(eps), PHI[phi], _ptr(gate), gd, _ptr(S_in),
                                       _ptr(z_in), _ptr(S_out), _ptr(z_out), _ptr(workspace),
                                       workspace.numel() if workspace is not None else 0,
                                       _stream_handle(stream, q.device))
    _raise(st, "la_forward_causal_gated")
    if check_status and workspace is not None:
        err, where = workspace_header(workspace)
        if err != LA_OK:
            raise LinAttnError(err, f"la_forward_causal_gated (run time, wait site {where})")
    return (y, S_out, z_out) if return_state else y


def decode_step_gated(q, k, v, S, z, gate=None, phi="elu1", eps: float = 1e-6, out=None,
                      stream=None):
    """One gated decode step in place on (S, z); gate None, [B,H] or [B,H,d]."""
    _check_cuda(q, k, v, S, z, gate, out)
    B, H, d = q.shape
    dv = v.shape[-1]
    gd = _gate_dim(gate, (B, H), d)
    y = out if out is not None else torch.empty((B, H, dv), dtype=torch.float32, device=q.device)
    st = lib().la_decode_step_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(y), _ptr(S), _ptr(z), B, H,
                                    d, dv, _dtype_code(q), float(eps), PHI[phi], _ptr(gate), gd,
                                    _stream_handle(stream, q.device))
    _raise(st, "la_decode_step_gated")
    return y


def forward_noncausal_phi(q, k, v, phi="identity", eps: float = 1e-6, return_state=False,
                          out=None, workspace=None, stream=None):
    """Non-causal attention with the feature map ``phi`` ("elu1" or "identity")."""
    _check_cuda(q, k, v, out, workspace)
    B, H, N, d = q.shape
    dv = v.shape[-1]
    dt = _dtype_code(q)
    y = out if out is not None else torch.empty((B, H, N, dv), dtype=torch.float32, device=q.device)
    S_out = z_out = None
    if return_state:
        S_out = torch.empty((B, H, d, dv), dtype=torch.float32, device=q.device)
        z_out = torch.empty((B, H, d), dtype=torch.float32, device=q.device)
    need = int(lib().la_noncausal_phi_workspace_bytes(B, H, N, d, dv, dt, PHI[phi]))
    if workspace is None:
        workspace = alloc_workspace(need, q.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib().la_forward_noncausal_phi(_ptr(q), _ptr(k), _ptr(v), _ptr(y), B, H, N, d, dv, dt,
                                        float(eps), PHI[phi], _ptr(S_out), _ptr(z_out),
                                        _ptr(workspace), wbytes, _stream_handle(stream, q.device))
    _raise(st, "la_forward_noncausal_phi")
    return (y, S_out, z_out) if return_state else y


def random_features(x, W, out=None, stream=None):
    """exp(W x - ||x||^2 / 2) / sqrt(m) for every row of x ([..., d], bf16 or fp32);
    W: float32 [m, d] CUDA tensor.  Returns float32 [..., m]."""
    _check_cuda(x, W, out)
    d = x.shape[-1]
    if W.dtype != torch.float32 or W.dim() != 2 or W.shape[1] != d:
        raise ValueError("W must be float32 [m, d]")
    m = W.shape[0]
    rows = x.numel() // d
    y = out if out is not None else torch.empty(tuple(x.shape[:-1]) + (m,), dtype=torch.float32,
                                                device=x.device)
    st = lib().la_random_features(_ptr(x), _ptr(y), rows, d, m, _dtype_code(x), _ptr(W),
                                  _stream_handle(stream, x.device))
    _raise(st, "la_random_features")
    return y
