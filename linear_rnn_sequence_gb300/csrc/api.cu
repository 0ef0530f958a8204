// api.cu -- the extern "C" entry points of liblinattn.so (declared in
// include/linattn.h): argument checks on the host, then dispatch to the
// kernels.  Nothing here computes attention; every step runs in the kernels.
#include <cmath>
#include <cstring>

#include "la_internal.h"

namespace la {

DebugFault &debug_fault() {
    static DebugFault f;
    return f;
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dim_ok(int x) { return x == 32 || x == 64 || x == 128; }

// [p, p+n) and [q, q+m) overlap?
bool overlap(const void *p, size_t n, const void *q, size_t m) {
    if (!p || !q || n == 0 || m == 0) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + m && b < a + n;
}

size_t esize(la_dtype dt) { return dt == LA_DTYPE_BF16 ? 2 : 4; }

la_status check_common(const void *q, const void *k, const void *v, const float *y, int B, int H,
                       long N, int d, int dv, la_dtype dt, float eps) {
    if (dt != LA_DTYPE_F32 && dt != LA_DTYPE_BF16) return LA_ERR_UNSUPPORTED;
    if (B < 1 || H < 1 || N < 0) return LA_ERR_INVALID_ARG;
    if (!dim_ok(d) || !dim_ok(dv)) return LA_ERR_UNSUPPORTED;
    if (!(eps > 0.f) || !std::isfinite(eps)) return LA_ERR_INVALID_ARG;
    const long long elems = (long long)B * H * (N > 0 ? N : 1) * (d > dv ? d : dv);
    if (elems >= (1LL << 31)) return LA_ERR_INVALID_ARG;
    const size_t es = esize(dt), T = (size_t)B * H * (N > 0 ? N : 0);
    if (T == 0) return LA_OK;  // no tokens: q, k, v, y are never touched (may be null)
    if (!q || !k || !v || !y) return LA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(y)) return LA_ERR_INVALID_ARG;
    const size_t ybytes = T * dv * 4;
    if (overlap(y, ybytes, q, T * d * es) || overlap(y, ybytes, k, T * d * es) ||
        overlap(y, ybytes, v, T * dv * es))
        return LA_ERR_INVALID_ARG;
    return LA_OK;
}

la_status check_state(const float *S, const float *z, bool required) {
    if ((S == nullptr) != (z == nullptr)) return LA_ERR_INVALID_ARG;
    if (required && !S) return LA_ERR_INVALID_ARG;
    if (S && (!aligned16(S) || !aligned16(z))) return LA_ERR_INVALID_ARG;
    return LA_OK;
}

la_status check_ws(void *ws, size_t have, size_t need) {
    if (need == 0) return LA_OK;
    if (!ws || have < need) return LA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return LA_ERR_WORKSPACE;
    return LA_OK;
}

la_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

size_t causal_ws(int B, int H, int N, int d, int dv, la_dtype dt) {
    FwdArgs a{};
    a.B = B; a.H = H; a.N = N; a.d = d; a.dv = dv; a.dt = dt;
    if (B < 1 || H < 1 || N < 0 || !dim_ok(d) || !dim_ok(dv)) return 0;
    if (causal_tc_supported(a)) return causal_tc_workspace(B * H, N, d, dv);
    return 0;
}

}  // namespace
}  // namespace la

using namespace la;

extern "C" {

const char *la_status_string(la_status s) {
    switch (s) {
    case LA_OK: return "LA_OK";
    case LA_ERR_INVALID_ARG: return "LA_ERR_INVALID_ARG";
    case LA_ERR_UNSUPPORTED: return "LA_ERR_UNSUPPORTED";
    case LA_ERR_CUDA: return "LA_ERR_CUDA";
    case LA_ERR_TIMEOUT: return "LA_ERR_TIMEOUT";
    case LA_ERR_WORKSPACE: return "LA_ERR_WORKSPACE";
    }
    return "LA_ERR_UNKNOWN";
}

const char *la_version(void) { return "linattn 0.1 sm_103a"; }

size_t la_causal_workspace_bytes(int B, int H, int N, int d, int dv, la_dtype dt) {
    return causal_ws(B, H, N, d, dv, dt);
}

size_t la_noncausal_workspace_bytes(int B, int H, int N, int d, int dv, la_dtype dt) {
    if (B < 1 || H < 1 || N < 1 || !dim_ok(d) || !dim_ok(dv)) return 0;
    FwdArgs a{};
    a.B = B; a.H = H; a.N = N; a.d = d; a.dv = dv; a.dt = dt;
    if (noncausal_tc_supported(a)) return noncausal_tc_workspace(B * H, N, d, dv);
    return noncausal_simt_workspace(B * H, N, d, dv);
}

la_status la_forward_causal(const void *q, const void *k, const void *v, float *y, int B, int H,
                            int N, int d, int dv, la_dtype dt, float eps, const float *S_in,
                            const float *z_in, float *S_out, float *z_out, void *workspace,
                            size_t workspace_bytes, void *stream) {
    la_status st = check_common(q, k, v, y, B, H, N, d, dv, dt, eps);
    if (st != LA_OK) return st;
    if ((st = check_state(S_in, z_in, false)) != LA_OK) return st;
    if ((st = check_state(S_out, z_out, false)) != LA_OK) return st;
    const size_t T = (size_t)B * H * N, sb = (size_t)B * H * d * dv * 4, zb = (size_t)B * H * d * 4;
    if (overlap(y, T * dv * 4, S_in, sb) || overlap(y, T * dv * 4, z_in, zb) ||
        overlap(y, T * dv * 4, S_out, sb) || overlap(y, T * dv * 4, z_out, zb))
        return LA_ERR_INVALID_ARG;
    const size_t need = causal_ws(B, H, N, d, dv, dt);
    if ((st = check_ws(workspace, workspace_bytes, need)) != LA_OK) return st;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (need > 0) {  // a fresh run-time status for every call that uses the workspace
        cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(WsHeader), s);
        if (e != cudaSuccess) return LA_ERR_CUDA;
    }
    if (N == 0) {  // no tokens: the final state is the initial state
        if (S_out) {
            cudaError_t e = cudaSuccess;
            if (!S_in) e = cudaMemsetAsync(S_out, 0, sb, s);
            else if (S_in != S_out)
                e = cudaMemcpyAsync(S_out, S_in, sb, cudaMemcpyDeviceToDevice, s);
            if (e == cudaSuccess) {
                if (!z_in) e = cudaMemsetAsync(z_out, 0, zb, s);
                else if (z_in != z_out)
                    e = cudaMemcpyAsync(z_out, z_in, zb, cudaMemcpyDeviceToDevice, s);
            }
            return from_cuda(e);
        }
        return LA_OK;
    }
    FwdArgs a{q, k, v, y, B, H, N, d, dv, dt, eps, S_in, z_in, S_out, z_out,
              workspace, workspace_bytes, s};
    if (causal_tc_supported(a)) return from_cuda(launch_causal_tc(a));
    return from_cuda(launch_causal_simt(a));
}

la_status la_forward_noncausal(const void *q, const void *k, const void *v, float *y, int B,
                               int H, int N, int d, int dv, la_dtype dt, float eps, float *S_out,
                               float *z_out, void *workspace, size_t workspace_bytes,
                               void *stream) {
    la_status st = check_common(q, k, v, y, B, H, N, d, dv, dt, eps);
    if (st != LA_OK) return st;
    if (N < 1) return LA_ERR_INVALID_ARG;
    if ((st = check_state(S_out, z_out, false)) != LA_OK) return st;
    const size_t T = (size_t)B * H * N, sb = (size_t)B * H * d * dv * 4, zb = (size_t)B * H * d * 4;
    if (overlap(y, T * dv * 4, S_out, sb) || overlap(y, T * dv * 4, z_out, zb))
        return LA_ERR_INVALID_ARG;
    const size_t need = la_noncausal_workspace_bytes(B, H, N, d, dv, dt);
    if ((st = check_ws(workspace, workspace_bytes, need)) != LA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    FwdArgs a{q, k, v, y, B, H, N, d, dv, dt, eps, nullptr, nullptr, S_out, z_out,
              workspace, workspace_bytes, s};
    const bool tc = noncausal_tc_supported(a);
    // a fresh run-time status (and, on the tensor-core path, fresh per-head
    // counters) for every call
    if (cudaMemsetAsync(workspace, 0, tc ? noncausal_tc_clear_bytes(B * H) : sizeof(WsHeader), s) !=
        cudaSuccess)
        return LA_ERR_CUDA;
    if (tc) return from_cuda(launch_noncausal_tc(a));
    return from_cuda(launch_noncausal_simt(a));
}

la_status la_decode_step(const void *q, const void *k, const void *v, float *y, float *S,
                         float *z, int B, int H, int d, int dv, la_dtype dt, float eps,
                         void *stream) {
    la_status st = check_common(q, k, v, y, B, H, 1, d, dv, dt, eps);
    if (st != LA_OK) return st;
    if ((st = check_state(S, z, true)) != LA_OK) return st;
    const size_t yb = (size_t)B * H * dv * 4, sb = (size_t)B * H * d * dv * 4,
                 zb = (size_t)B * H * d * 4;
    if (overlap(y, yb, S, sb) || overlap(y, yb, z, zb) || overlap(S, sb, z, zb))
        return LA_ERR_INVALID_ARG;
    DecodeArgs a{q, k, v, y, S, z, B, H, d, dv, dt, eps, static_cast<cudaStream_t>(stream)};
    return from_cuda(launch_decode_simt(a));
}

la_status la_forward_causal_decay(const void *q, const void *k, const void *v, float *y, int B,
                                  int H, int N, int d, int dv, la_dtype dt, float eps,
                                  const float *gamma, const float *S_in, const float *z_in,
                                  float *S_out, float *z_out, void *workspace,
                                  size_t workspace_bytes, void *stream) {
    la_status st = check_common(q, k, v, y, B, H, N, d, dv, dt, eps);
    if (st != LA_OK) return st;
    if (!gamma || (reinterpret_cast<uintptr_t>(gamma) & 3u) != 0) return LA_ERR_INVALID_ARG;
    if ((st = check_state(S_in, z_in, false)) != LA_OK) return st;
    if ((st = check_state(S_out, z_out, false)) != LA_OK) return st;
    const size_t T = (size_t)B * H * N, sb = (size_t)B * H * d * dv * 4, zb = (size_t)B * H * d * 4;
    if (overlap(y, T * dv * 4, S_in, sb) || overlap(y, T * dv * 4, z_in, zb) ||
        overlap(y, T * dv * 4, S_out, sb) || overlap(y, T * dv * 4, z_out, zb) ||
        overlap(y, T * dv * 4, gamma, (size_t)H * 4))
        return LA_ERR_INVALID_ARG;
    const size_t need = causal_ws(B, H, N, d, dv, dt);
    if ((st = check_ws(workspace, workspace_bytes, need)) != LA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (need > 0) {  // a fresh run-time status for every call that uses the workspace
        if (cudaMemsetAsync(workspace, 0, sizeof(WsHeader), s) != cudaSuccess) return LA_ERR_CUDA;
    }
    if (N == 0) {  // no tokens: the final state is the initial state
        if (S_out) {
            cudaError_t e = cudaSuccess;
            if (!S_in) e = cudaMemsetAsync(S_out, 0, sb, s);
            else if (S_in != S_out)
                e = cudaMemcpyAsync(S_out, S_in, sb, cudaMemcpyDeviceToDevice, s);
            if (e == cudaSuccess) {
                if (!z_in) e = cudaMemsetAsync(z_out, 0, zb, s);
                else if (z_in != z_out)
                    e = cudaMemcpyAsync(z_out, z_in, zb, cudaMemcpyDeviceToDevice, s);
            }
            return from_cuda(e);
        }
        return LA_OK;
    }
    FwdArgs a{q, k, v, y, B, H, N, d, dv, dt, eps, S_in, z_in, S_out, z_out,
              workspace, workspace_bytes, s};
    a.gamma = gamma;
    // heads with decay_on_tensor_cores(gamma) on the tensor cores, then the
    // rest on the CUDA cores (the second kernel's CTAs for the first kind
    // return at once); no host read of gamma is needed to split them
    if (causal_tc_supported(a)) {
        const cudaError_t e = launch_causal_tc(a);
        if (e != cudaSuccess) return from_cuda(e);
        a.skip_tc_heads = true;
    }
    return from_cuda(launch_causal_simt(a));
}

la_status la_decode_step_decay(const void *q, const void *k, const void *v, float *y, float *S,
                               float *z, int B, int H, int d, int dv, la_dtype dt, float eps,
                               const float *gamma, void *stream) {
    la_status st = check_common(q, k, v, y, B, H, 1, d, dv, dt, eps);
    if (st != LA_OK) return st;
    if (!gamma || (reinterpret_cast<uintptr_t>(gamma) & 3u) != 0) return LA_ERR_INVALID_ARG;
    if ((st = check_state(S, z, true)) != LA_OK) return st;
    const size_t yb = (size_t)B * H * dv * 4, sb = (size_t)B * H * d * dv * 4,
                 zb = (size_t)B * H * d * 4;
    if (overlap(y, yb, S, sb) || overlap(y, yb, z, zb) || overlap(S, sb, z, zb) ||
        overlap(gamma, (size_t)H * 4, S, sb) || overlap(gamma, (size_t)H * 4, z, zb) ||
        overlap(gamma, (size_t)H * 4, y, yb))
        return LA_ERR_INVALID_ARG;
    DecodeArgs a{q, k, v, y, S, z, B, H, d, dv, dt, eps, static_cast<cudaStream_t>(stream)};
    a.gamma = gamma;
    return from_cuda(launch_decode_simt(a));
}

size_t la_causal_gated_workspace_bytes(int B, int H, int N, int d, int dv, la_dtype dt,
                                       la_phi phi, int gate_dim) {
    if (B < 1 || H < 1 || N < 0 || !dim_ok(d) || !dim_ok(dv)) return 0;
    if (dt != LA_DTYPE_F32 && dt != LA_DTYPE_BF16) return 0;
    if (gate_dim != 1 && gate_dim != d) return 0;
    FwdArgs a{};
    a.B = B; a.H = H; a.N = N; a.d = d; a.dv = dv; a.dt = dt;
    a.phi = (int)phi;
    a.gate = reinterpret_cast<const float *>(&a);   // a gate is given (its address is not used)
    a.gate_dim = gate_dim;
    if (N > 0 && gated_tc_supported(a)) return gated_tc_workspace(B * H, N, d, dv);
    return sizeof(WsHeader);
}

la_status la_forward_causal_gated(const void *q, const void *k, const void *v, float *y, int B,
                                  int H, int N, int d, int dv, la_dtype dt, float eps, la_phi phi,
                                  const float *gate, int gate_dim, const float *S_in,
                                  const float *z_in, float *S_out, float *z_out, void *workspace,
                                  size_t workspace_bytes, void *stream) {
    la_status st = check_common(q, k, v, y, B, H, N, d, dv, dt, eps);
    if (st != LA_OK) return st;
    if (phi != LA_PHI_ELU1 && phi != LA_PHI_IDENTITY) return LA_ERR_UNSUPPORTED;
    if (gate && gate_dim != 1 && gate_dim != d) return LA_ERR_INVALID_ARG;
    if (gate && (reinterpret_cast<uintptr_t>(gate) & 3u) != 0) return LA_ERR_INVALID_ARG;
    if ((st = check_state(S_in, z_in, false)) != LA_OK) return st;
    if ((st = check_state(S_out, z_out, false)) != LA_OK) return st;
    const size_t T = (size_t)B * H * N, sb = (size_t)B * H * d * dv * 4, zb = (size_t)B * H * d * 4;
    const size_t gb = gate ? T * gate_dim * 4 : 0;
    if (overlap(y, T * dv * 4, S_in, sb) || overlap(y, T * dv * 4, z_in, zb) ||
        overlap(y, T * dv * 4, S_out, sb) || overlap(y, T * dv * 4, z_out, zb) ||
        overlap(y, T * dv * 4, gate, gb) || overlap(S_out, sb, gate, gb) ||
        overlap(z_out, zb, gate, gb))
        return LA_ERR_INVALID_ARG;
    const size_t need = gate ? la_causal_gated_workspace_bytes(B, H, N, d, dv, dt, phi, gate_dim)
                             : sizeof(WsHeader);
    if ((st = check_ws(workspace, workspace_bytes, need)) != LA_OK) return st;
    if (overlap(workspace, need, y, T * dv * 4) || overlap(workspace, need, gate, gb) ||
        overlap(workspace, need, S_out, sb) || overlap(workspace, need, z_out, zb))
        return LA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // a fresh run-time status for every call (the tensor-core path also clears its flags)
    if (cudaMemsetAsync(workspace, 0, sizeof(WsHeader), s) != cudaSuccess) return LA_ERR_CUDA;
    if (N == 0) {  // no tokens: the final state is the initial state
        if (S_out) {
            cudaError_t e = cudaSuccess;
            if (!S_in) e = cudaMemsetAsync(S_out, 0, sb, s);
            else if (S_in != S_out)
                e = cudaMemcpyAsync(S_out, S_in, sb, cudaMemcpyDeviceToDevice, s);
            if (e == cudaSuccess) {
                if (!z_in) e = cudaMemsetAsync(z_out, 0, zb, s);
                else if (z_in != z_out)
                    e = cudaMemcpyAsync(z_out, z_in, zb, cudaMemcpyDeviceToDevice, s);
            }
            return from_cuda(e);
        }
        return LA_OK;
    }
    FwdArgs a{q, k, v, y, B, H, N, d, dv, dt, eps, S_in, z_in, S_out, z_out, workspace,
              workspace_bytes, s};
    a.phi = (int)phi;
    a.gate = gate;
    a.gate_dim = gate ? gate_dim : 1;
    return from_cuda(launch_causal_gated(a));
}

la_status la_decode_step_gated(const void *q, const void *k, const void *v, float *y, float *S,
                               float *z, int B, int H, int d, int dv, la_dtype dt, float eps,
                               la_phi phi, const float *gate, int gate_dim, void *stream) {
    la_status st = check_common(q, k, v, y, B, H, 1, d, dv, dt, eps);
    if (st != LA_OK) return st;
    if (phi != LA_PHI_ELU1 && phi != LA_PHI_IDENTITY) return LA_ERR_UNSUPPORTED;
    if (gate && gate_dim != 1 && gate_dim != d) return LA_ERR_INVALID_ARG;
    if (gate && (reinterpret_cast<uintptr_t>(gate) & 3u) != 0) return LA_ERR_INVALID_ARG;
    if ((st = check_state(S, z, true)) != LA_OK) return st;
    const size_t yb = (size_t)B * H * dv * 4, sb = (size_t)B * H * d * dv * 4,
                 zb = (size_t)B * H * d * 4, gb = gate ? (size_t)B * H * gate_dim * 4 : 0;
    if (overlap(y, yb, S, sb) || overlap(y, yb, z, zb) || overlap(S, sb, z, zb) ||
        overlap(gate, gb, S, sb) || overlap(gate, gb, z, zb) || overlap(gate, gb, y, yb))
        return LA_ERR_INVALID_ARG;
    DecodeArgs a{q, k, v, y, S, z, B, H, d, dv, dt, eps, static_cast<cudaStream_t>(stream)};
    a.phi = (int)phi;
    a.gate = gate;
    a.gate_dim = gate ? gate_dim : 1;
    return from_cuda(launch_decode_simt(a));
}

size_t la_noncausal_phi_workspace_bytes(int B, int H, int N, int d, int dv, la_dtype dt,
                                        la_phi phi) {
    if (phi == LA_PHI_ELU1) return la_noncausal_workspace_bytes(B, H, N, d, dv, dt);
    if (phi != LA_PHI_IDENTITY || B < 1 || H < 1 || N < 1 || !dim_ok(d) || !dim_ok(dv)) return 0;
    return noncausal_simt_workspace(B * H, N, d, dv);
}

la_status la_forward_noncausal_phi(const void *q, const void *k, const void *v, float *y, int B,
                                   int H, int N, int d, int dv, la_dtype dt, float eps,
                                   la_phi phi, float *S_out, float *z_out, void *workspace,
                                   size_t workspace_bytes, void *stream) {
    if (phi == LA_PHI_ELU1)
        return la_forward_noncausal(q, k, v, y, B, H, N, d, dv, dt, eps, S_out, z_out, workspace,
                                    workspace_bytes, stream);
    if (phi != LA_PHI_IDENTITY) return LA_ERR_UNSUPPORTED;
    la_status st = check_common(q, k, v, y, B, H, N, d, dv, dt, eps);
    if (st != LA_OK) return st;
    if (N < 1) return LA_ERR_INVALID_ARG;
    if ((st = check_state(S_out, z_out, false)) != LA_OK) return st;
    const size_t T = (size_t)B * H * N, sb = (size_t)B * H * d * dv * 4, zb = (size_t)B * H * d * 4;
    if (overlap(y, T * dv * 4, S_out, sb) || overlap(y, T * dv * 4, z_out, zb))
        return LA_ERR_INVALID_ARG;
    const size_t need = la_noncausal_phi_workspace_bytes(B, H, N, d, dv, dt, phi);
    if ((st = check_ws(workspace, workspace_bytes, need)) != LA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, sizeof(WsHeader), s) != cudaSuccess) return LA_ERR_CUDA;
    FwdArgs a{q, k, v, y, B, H, N, d, dv, dt, eps, nullptr, nullptr, S_out, z_out,
              workspace, workspace_bytes, s};
    a.phi = (int)phi;
    return from_cuda(launch_noncausal_simt(a));
}

la_status la_random_features(const void *x, float *phi_out, long long rows, int d, int m,
                             la_dtype dt, const float *W, void *stream) {
    if (dt != LA_DTYPE_F32 && dt != LA_DTYPE_BF16) return LA_ERR_UNSUPPORTED;
    if (rows < 0 || d < 1 || d > 128 || m < 1 || m > 256) return LA_ERR_INVALID_ARG;
    if (rows == 0) return LA_OK;
    if (!x || !phi_out || !W) return LA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & (esize(dt) - 1)) != 0 ||
        (reinterpret_cast<uintptr_t>(phi_out) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(W) & 3u) != 0)
        return LA_ERR_INVALID_ARG;
    const size_t ob = (size_t)rows * m * 4;
    if (overlap(phi_out, ob, x, (size_t)rows * d * esize(dt)) ||
        overlap(phi_out, ob, W, (size_t)m * d * 4))
        return LA_ERR_INVALID_ARG;
    return from_cuda(launch_random_features(x, phi_out, rows, d, m, dt, W,
                                            static_cast<cudaStream_t>(stream)));
}

size_t la_causal_backward_workspace_bytes(int B, int H, int N, int d, int dv, la_dtype dt) {
    if (B < 1 || H < 1 || N < 1 || !dim_ok(d) || !dim_ok(dv)) return 0;
    if (dt != LA_DTYPE_F32 && dt != LA_DTYPE_BF16) return 0;
    if ((long long)B * H * N * (d > dv ? d : dv) >= (1LL << 31)) return 0;
    return causal_backward_workspace(B * H, N, d, dv);
}

}  // extern "C"

namespace la {
namespace {

// la_backward_causal and la_backward_causal_decay (gamma null: no decay).
la_status backward_impl(const void *q, const void *k, const void *v, const float *dy,
                        float *grad_q, float *grad_k, float *grad_v, int B, int H, int N, int d,
                        int dv, la_dtype dt, float eps, const float *gamma, const float *S_in,
                        const float *z_in, float *grad_S_in, float *grad_z_in, void *workspace,
                        size_t workspace_bytes, void *stream) {
    la_status st = check_common(q, k, v, grad_v, B, H, N, d, dv, dt, eps);
    if (st != LA_OK) return st;
    if ((st = check_state(S_in, z_in, false)) != LA_OK) return st;
    if ((st = check_state(grad_S_in, grad_z_in, false)) != LA_OK) return st;
    const size_t BH = (size_t)B * H, T = BH * N, es = esize(dt);
    const size_t sb = BH * d * dv * 4, zb = BH * d * 4;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T > 0) {
        if (!dy || !grad_q || !grad_k) return LA_ERR_INVALID_ARG;
        if (!aligned16(dy) || !aligned16(grad_q) || !aligned16(grad_k)) return LA_ERR_INVALID_ARG;
    }
    const size_t need = la_causal_backward_workspace_bytes(B, H, N, d, dv, dt);
    // no output may overlap an input, the workspace or another output
    const struct { const void *p; size_t n; } outs[] = {
        {grad_q, T * d * 4}, {grad_k, T * d * 4}, {grad_v, T * dv * 4},
        {grad_S_in, grad_S_in ? sb : 0}, {grad_z_in, grad_z_in ? zb : 0}};
    const struct { const void *p; size_t n; } ins[] = {
        {q, T * d * es}, {k, T * d * es}, {v, T * dv * es}, {dy, T * dv * 4},
        {S_in, S_in ? sb : 0}, {z_in, z_in ? zb : 0}, {workspace, need}};
    for (size_t i = 0; i < sizeof(outs) / sizeof(outs[0]); ++i) {
        for (const auto &in : ins)
            if (overlap(outs[i].p, outs[i].n, in.p, in.n)) return LA_ERR_INVALID_ARG;
        for (size_t j = i + 1; j < sizeof(outs) / sizeof(outs[0]); ++j)
            if (overlap(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return LA_ERR_INVALID_ARG;
    }
    if (T == 0) {   // no tokens: the initial state gets no gradient
        if (grad_S_in) {
            cudaError_t e = cudaMemsetAsync(grad_S_in, 0, sb, s);
            if (e == cudaSuccess) e = cudaMemsetAsync(grad_z_in, 0, zb, s);
            return from_cuda(e);
        }
        return LA_OK;
    }
    if ((st = check_ws(workspace, workspace_bytes, need)) != LA_OK) return st;
    if (cudaMemsetAsync(workspace, 0, sizeof(WsHeader), s) != cudaSuccess) return LA_ERR_CUDA;
    BwdArgs a{q, k, v, dy, grad_q, grad_k, grad_v, B, H, N, d, dv, dt, eps, S_in, z_in,
              grad_S_in, grad_z_in, workspace, workspace_bytes, s};
    a.gamma = gamma;
    return from_cuda(launch_causal_backward(a));
}

}  // namespace
}  // namespace la

extern "C" {

la_status la_backward_causal(const void *q, const void *k, const void *v, const float *dy,
                             float *grad_q, float *grad_k, float *grad_v, int B, int H, int N,
                             int d, int dv, la_dtype dt, float eps, const float *S_in,
                             const float *z_in, float *grad_S_in, float *grad_z_in,
                             void *workspace, size_t workspace_bytes, void *stream) {
    return backward_impl(q, k, v, dy, grad_q, grad_k, grad_v, B, H, N, d, dv, dt, eps, nullptr,
                         S_in, z_in, grad_S_in, grad_z_in, workspace, workspace_bytes, stream);
}

la_status la_backward_causal_decay(const void *q, const void *k, const void *v,
                                   const float *dy, float *grad_q, float *grad_k,
                                   float *grad_v, int B, int H, int N, int d, int dv,
                                   la_dtype dt, float eps, const float *gamma,
                                   const float *S_in, const float *z_in, float *grad_S_in,
                                   float *grad_z_in, void *workspace, size_t workspace_bytes,
                                   void *stream) {
    if (!gamma || (reinterpret_cast<uintptr_t>(gamma) & 3u) != 0) return LA_ERR_INVALID_ARG;
    const size_t T = (size_t)B * H * (N > 0 ? N : 0);
    if (overlap(gamma, (size_t)H * 4, grad_q, T * d * 4) ||
        overlap(gamma, (size_t)H * 4, grad_k, T * d * 4) ||
        overlap(gamma, (size_t)H * 4, grad_v, T * dv * 4))
        return LA_ERR_INVALID_ARG;
    return backward_impl(q, k, v, dy, grad_q, grad_k, grad_v, B, H, N, d, dv, dt, eps, gamma,
                         S_in, z_in, grad_S_in, grad_z_in, workspace, workspace_bytes, stream);
}


la_status la_workspace_status(const void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace || workspace_bytes < sizeof(WsHeader)) return LA_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return LA_ERR_CUDA;
    WsHeader h;
    if (cudaMemcpy(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
        return LA_ERR_CUDA;
    return h.error == 0 ? LA_OK : static_cast<la_status>(h.error);
}

void la_debug_set_fault(int drop_load_item, long long wait_limit_ns) {
    debug_fault().drop_load_item = drop_load_item;
    debug_fault().wait_limit_ns = wait_limit_ns;
}

}  // extern "C"
