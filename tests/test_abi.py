"""C-ABI checks that need no GPU: the library builds for sm_103a, loads, and
exports every entry point include/linattn.h declares; host-side argument
validation rejects bad calls before anything is launched."""
import ctypes
import os
import re
import subprocess

import pytest

from linear_rnn_sequence_gb300 import _build
from linear_rnn_sequence_gb300 import linattn as la

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "linattn.h")


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"LA_API\s+[\w\s\*]*?\b(la_\w+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("la_forward_causal", "la_forward_noncausal", "la_decode_step",
              "la_causal_workspace_bytes", "la_noncausal_workspace_bytes", "la_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    L = la.lib()
    for n in declared_functions():
        assert hasattr(L, n), f"{n} not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\bT (la_\w+)", out))
    assert set(declared_functions()) <= exported


def test_build_targets_sm103a_only():
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_header_compiles_as_c():
    src = '#include "linattn.h"\nint main(void){ return (int)LA_OK; }\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                        "-x", "c", "-", "-o", "/dev/null"], input=src, text=True,
                       capture_output=True)
    assert r.returncode == 0, r.stderr


def test_status_strings_and_version():
    assert la.status_string(la.LA_OK) == "LA_OK"
    assert la.status_string(la.LA_ERR_TIMEOUT) == "LA_ERR_TIMEOUT"
    assert la.status_string(99) == "LA_ERR_UNKNOWN"
    assert "sm_103a" in la.version()


def test_workspace_sizes():
    L = la.lib()
    assert L.la_noncausal_workspace_bytes(4, 8, 4096, 64, 64, 1) > 256
    assert L.la_noncausal_workspace_bytes(4, 8, 0, 64, 64, 1) == 0
    assert L.la_noncausal_workspace_bytes(4, 8, 16, 48, 64, 1) == 0
    assert L.la_causal_workspace_bytes(1, 1, 10, 48, 64, 1) == 0


# Fake, 256-byte aligned "device" addresses: every call below must be rejected
# by the host-side checks, so nothing is ever dereferenced or launched.
P = ctypes.c_void_p(1 << 20)
P2 = ctypes.c_void_p((1 << 20) + (1 << 28))
P3 = ctypes.c_void_p((1 << 20) + (2 << 28))
Y = ctypes.c_void_p((1 << 20) + (3 << 28))


def _causal(**kw):
    a = dict(q=P, k=P2, v=P3, y=Y, B=1, H=1, N=8, d=64, dv=64, dt=1, eps=1e-6, S_in=None,
             z_in=None, S_out=None, z_out=None, ws=None, wsb=0, stream=None)
    a.update(kw)
    return la.lib().la_forward_causal(a["q"], a["k"], a["v"], a["y"], a["B"], a["H"], a["N"],
                                      a["d"], a["dv"], a["dt"], a["eps"], a["S_in"], a["z_in"],
                                      a["S_out"], a["z_out"], a["ws"], a["wsb"], a["stream"])


@pytest.mark.parametrize("kw,expected", [
    (dict(q=None), la.LA_ERR_INVALID_ARG),
    (dict(y=None), la.LA_ERR_INVALID_ARG),
    (dict(q=ctypes.c_void_p((1 << 20) + 4)), la.LA_ERR_INVALID_ARG),   # misaligned
    (dict(d=48), la.LA_ERR_UNSUPPORTED),
    (dict(dv=256), la.LA_ERR_UNSUPPORTED),
    (dict(dt=7), la.LA_ERR_UNSUPPORTED),
    (dict(eps=0.0), la.LA_ERR_INVALID_ARG),
    (dict(eps=-1.0), la.LA_ERR_INVALID_ARG),
    (dict(eps=float("nan")), la.LA_ERR_INVALID_ARG),
    (dict(eps=float("inf")), la.LA_ERR_INVALID_ARG),
    (dict(B=0), la.LA_ERR_INVALID_ARG),
    (dict(N=-1), la.LA_ERR_INVALID_ARG),
    (dict(S_in=P), la.LA_ERR_INVALID_ARG),             # S_in without z_in
    (dict(z_out=P), la.LA_ERR_INVALID_ARG),            # z_out without S_out
    (dict(y=ctypes.c_void_p((1 << 20) + 64)), la.LA_ERR_INVALID_ARG),  # y overlaps q
    (dict(B=1 << 14, H=1 << 10, N=1 << 10), la.LA_ERR_INVALID_ARG),    # too large
])
def test_causal_rejects_bad_arguments(kw, expected):
    assert _causal(**kw) == expected


def test_noncausal_needs_workspace_and_tokens():
    L = la.lib()
    st = L.la_forward_noncausal(P, P2, P3, Y, 1, 1, 8, 64, 64, 1, 1e-6, None, None, None, 0, None)
    assert st == la.LA_ERR_WORKSPACE
    st = L.la_forward_noncausal(P, P2, P3, Y, 1, 1, 0, 64, 64, 1, 1e-6, None, None, P, 1 << 20,
                                None)
    assert st == la.LA_ERR_INVALID_ARG
    # misaligned workspace
    need = L.la_noncausal_workspace_bytes(1, 1, 8, 64, 64, 1)
    st = L.la_forward_noncausal(P, P2, P3, Y, 1, 1, 8, 64, 64, 1, 1e-6, None, None,
                                ctypes.c_void_p((3 << 20) + 16), need, None)
    assert st == la.LA_ERR_WORKSPACE


def test_decode_requires_state():
    L = la.lib()
    st = L.la_decode_step(P, P2, P3, Y, None, None, 1, 1, 64, 64, 1, 1e-6, None)
    assert st == la.LA_ERR_INVALID_ARG
    # y overlapping the state
    st = L.la_decode_step(P, P2, P3, Y, Y, P, 1, 1, 64, 64, 1, 1e-6, None)
    assert st == la.LA_ERR_INVALID_ARG


def test_host_entry_point_rejects_bad_arguments():
    L = la.lib()
    h = ctypes.c_void_p(1 << 20)
    # null inputs, mismatched state pointers, bad eps, unsupported sizes: no copy is issued
    assert L.la_forward_causal_host(None, h, h, h, 1, 1, 8, 64, 64, 1, 1e-6, None, None, P, 1 << 30,
                                    None) == la.LA_ERR_INVALID_ARG
    assert L.la_forward_causal_host(h, h, h, Y, 1, 1, 8, 64, 64, 1, 1e-6, h, None, P, 1 << 30,
                                    None) == la.LA_ERR_INVALID_ARG
    assert L.la_forward_causal_host(h, h, h, Y, 1, 1, 8, 64, 64, 1, 0.0, None, None, P, 1 << 30,
                                    None) == la.LA_ERR_INVALID_ARG
    assert L.la_forward_causal_host(h, h, h, Y, 1, 1, 8, 48, 64, 1, 1e-6, None, None, P, 1 << 30,
                                    None) == la.LA_ERR_UNSUPPORTED
    # y overlapping q in host memory
    assert L.la_forward_causal_host(h, P2, P3, ctypes.c_void_p((1 << 20) + 64), 1, 1, 8, 64, 64, 1,
                                    1e-6, None, None, P, 1 << 30, None) == la.LA_ERR_INVALID_ARG
    assert L.la_causal_host_buffer_bytes(1, 1, 0, 64, 64, 1) == 0
    assert L.la_causal_host_buffer_bytes(2, 8, 1000, 64, 64, 1) > 0


def test_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 4, 32)
    with pytest.raises(ValueError):
        la.forward_causal(q, q, q)


def test_backward_rejects_bad_arguments():
    L = la.lib()
    need = L.la_causal_backward_workspace_bytes(1, 1, 8, 64, 64, 1)
    assert need > 256
    assert L.la_causal_backward_workspace_bytes(1, 1, 0, 64, 64, 1) == 0
    assert L.la_causal_backward_workspace_bytes(1, 1, 8, 48, 64, 1) == 0
    p = [ctypes.c_void_p((i + 1) << 24) for i in range(12)]   # far apart, 16-byte aligned
    q, k, v, dy, gq, gk, gv, S, z, gS, gz, ws = p

    def call(**kw):
        a = dict(q=q, k=k, v=v, dy=dy, gq=gq, gk=gk, gv=gv, B=1, H=1, N=8, d=64, dv=64, dt=1,
                 eps=1e-6, S=None, z=None, gS=None, gz=None, ws=ws, wsb=need)
        a.update(kw)
        return L.la_backward_causal(a["q"], a["k"], a["v"], a["dy"], a["gq"], a["gk"], a["gv"],
                                    a["B"], a["H"], a["N"], a["d"], a["dv"], a["dt"], a["eps"],
                                    a["S"], a["z"], a["gS"], a["gz"], a["ws"], a["wsb"], None)

    assert call(dy=None) == la.LA_ERR_INVALID_ARG
    assert call(eps=0.0) == la.LA_ERR_INVALID_ARG
    assert call(d=48) == la.LA_ERR_UNSUPPORTED
    assert call(dt=7) == la.LA_ERR_UNSUPPORTED
    assert call(gq=ctypes.c_void_p(q.value + 256)) == la.LA_ERR_INVALID_ARG    # dq over q
    assert call(gk=ctypes.c_void_p(ws.value + 512)) == la.LA_ERR_INVALID_ARG   # dk over the workspace
    assert call(gv=ctypes.c_void_p(gq.value + 16)) == la.LA_ERR_INVALID_ARG    # two outputs overlap
    assert call(gS=gS) == la.LA_ERR_INVALID_ARG                                # dS without dz
    assert call(S=S) == la.LA_ERR_INVALID_ARG                                  # S_in without z_in
    assert call(gq=ctypes.c_void_p(gq.value + 4)) == la.LA_ERR_INVALID_ARG     # misaligned
    assert call(wsb=need - 1) == la.LA_ERR_WORKSPACE
    assert call(ws=ctypes.c_void_p(ws.value + 16)) == la.LA_ERR_WORKSPACE      # not 256-aligned


def test_decay_entry_points_reject_bad_arguments():
    L = la.lib()
    p = [ctypes.c_void_p((i + 1) << 24) for i in range(8)]
    q, k, v, y, S, z, g, ws = p
    need = L.la_causal_workspace_bytes(1, 2, 8, 64, 64, 1)
    assert need >= 256   # bf16, d = dv = 64: the tensor-core kernel's status header

    def fwd(d=64, eps=1e-6, gam=g, S_in=None, ws_=ws, wsb=need):
        return L.la_forward_causal_decay(q, k, v, y, 1, 2, 8, d, 64, 1, eps, gam, S_in, None,
                                         None, None, ws_, wsb, None)
    assert fwd(gam=None) == la.LA_ERR_INVALID_ARG                  # no gamma
    assert fwd(d=48) == la.LA_ERR_UNSUPPORTED
    assert fwd(eps=0.0) == la.LA_ERR_INVALID_ARG
    assert fwd(S_in=S) == la.LA_ERR_INVALID_ARG                    # S_in alone
    assert fwd(ws_=None, wsb=0) == la.LA_ERR_WORKSPACE
    assert fwd(wsb=need - 1) == la.LA_ERR_WORKSPACE
    assert fwd(ws_=ctypes.c_void_p(ws.value + 16)) == la.LA_ERR_WORKSPACE   # not 256-aligned
    # float32 inputs take the CUDA-core kernel alone: no workspace
    assert L.la_causal_workspace_bytes(1, 2, 8, 64, 64, 0) == 0
    assert L.la_decode_step_decay(q, k, v, y, S, z, 1, 2, 64, 64, 1, 1e-6, None,
                                  None) == la.LA_ERR_INVALID_ARG
    assert L.la_decode_step_decay(q, k, v, y, None, z, 1, 2, 64, 64, 1, 1e-6, g,
                                  None) == la.LA_ERR_INVALID_ARG
    assert L.la_decode_step_decay(q, k, v, y, S, ctypes.c_void_p(S.value + 64), 1, 2, 64, 64, 1,
                                  1e-6, g, None) == la.LA_ERR_INVALID_ARG        # S overlaps z
    assert L.la_decode_step_decay(q, k, v, y, S, z, 1, 2, 64, 64, 1, 1e-6,
                                  ctypes.c_void_p(g.value + 2), None) == la.LA_ERR_INVALID_ARG


def test_backward_decay_rejects_bad_arguments():
    L = la.lib()
    need = L.la_causal_backward_workspace_bytes(1, 2, 8, 64, 64, 1)
    p = [ctypes.c_void_p((i + 1) << 24) for i in range(10)]
    q, k, v, dy, gq, gk, gv, g, ws, _ = p
    call = lambda gamma: L.la_backward_causal_decay(q, k, v, dy, gq, gk, gv, 1, 2, 8, 64, 64, 1,
                                                    1e-6, gamma, None, None, None, None, ws,
                                                    need, None)
    assert call(None) == la.LA_ERR_INVALID_ARG
    assert call(ctypes.c_void_p(g.value + 1)) == la.LA_ERR_INVALID_ARG      # misaligned
    assert call(ctypes.c_void_p(gq.value + 64)) == la.LA_ERR_INVALID_ARG    # gamma inside dq
