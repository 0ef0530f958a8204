// host.cu -- causal forward on host buffers, with the host<->device copies
// overlapped with the kernels.
//
// The B*H heads are cut into groups.  Group i goes through three streams:
// its q, k, v copies on an upload stream, its forward on the caller's stream,
// and its y (and final state) copies on a download stream, ordered by events.
// Three device staging sets rotate between the groups, so the upload of
// group i+1, the forward of group i and the download of group i-1 can run at
// once, and uploads and downloads use both directions of the host link.
// Every group is an ordinary la_forward_causal call on device pointers: heads
// are independent, so the result equals the one-shot call up to summation
// order (the group sizes change how the sequence axis is split).
#include <algorithm>
#include <cmath>
#include <cstring>

#include "la_internal.h"

namespace la {
namespace {

constexpr int kHostGroups = 16;   // head groups per call (fewer when there are fewer heads)
constexpr int kHostSets = 3;      // device staging sets

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

struct HostPlan {
    int BH = 0, group_heads = 0, ngroups = 0;
    size_t q = 0, v = 0, y = 0, S = 0, z = 0, ws = 0, set = 0, err = 0;
};

HostPlan make_plan(int B, int H, int N, int d, int dv, la_dtype dt) {
    HostPlan p;
    p.BH = B * H;
    const int g = std::min(kHostGroups, p.BH);
    p.group_heads = (p.BH + g - 1) / g;
    p.ngroups = (p.BH + p.group_heads - 1) / p.group_heads;
    const size_t es = dt == LA_DTYPE_BF16 ? 2 : 4, T = (size_t)p.group_heads * N;
    p.q = up256(T * d * es);
    p.v = up256(T * dv * es);
    p.y = up256(T * dv * 4);
    p.S = up256((size_t)p.group_heads * d * dv * 4);
    p.z = up256((size_t)p.group_heads * d * 4);
    p.ws = up256(la_causal_workspace_bytes(1, p.group_heads, N, d, dv, dt));
    p.set = 2 * p.q + p.v + p.y + p.S + p.z + p.ws;
    p.err = up256(sizeof(unsigned int) * kHostGroups);
    return p;
}

bool sizes_ok(int B, int H, int N, int d, int dv, la_dtype dt) {
    auto dim_ok = [](int x) { return x == 32 || x == 64 || x == 128; };
    return B >= 1 && H >= 1 && N >= 0 && dim_ok(d) && dim_ok(dv) &&
           (dt == LA_DTYPE_F32 || dt == LA_DTYPE_BF16);
}

bool overlap(const void *p, size_t n, const void *q, size_t m) {
    if (!p || !q || n == 0 || m == 0) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + m && b < a + n;
}

// Streams and events of one call; destroyed when the call returns.
struct CallResources {
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t in[kHostGroups] = {}, done[kHostGroups] = {}, out[kHostGroups] = {};
    bool ok = true;
    CallResources() {
        ok = cudaStreamCreateWithFlags(&up, cudaStreamNonBlocking) == cudaSuccess &&
             cudaStreamCreateWithFlags(&down, cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&start, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; ok && i < kHostGroups; ++i)
            ok = cudaEventCreateWithFlags(&in[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&done[i], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&out[i], cudaEventDisableTiming) == cudaSuccess;
    }
    ~CallResources() {
        for (int i = 0; i < kHostGroups; ++i) {
            if (in[i]) cudaEventDestroy(in[i]);
            if (done[i]) cudaEventDestroy(done[i]);
            if (out[i]) cudaEventDestroy(out[i]);
        }
        if (start) cudaEventDestroy(start);
        if (up) cudaStreamDestroy(up);
        if (down) cudaStreamDestroy(down);
    }
};

}  // namespace
}  // namespace la

using namespace la;

extern "C" {

size_t la_causal_host_buffer_bytes(int B, int H, int N, int d, int dv, la_dtype dt) {
    if (!sizes_ok(B, H, N, d, dv, dt) || N == 0) return 0;
    const HostPlan p = make_plan(B, H, N, d, dv, dt);
    return p.err + kHostSets * p.set;
}

la_status la_forward_causal_host(const void *q, const void *k, const void *v, float *y, int B,
                                 int H, int N, int d, int dv, la_dtype dt, float eps,
                                 float *S_out, float *z_out, void *dev_buf,
                                 size_t dev_buf_bytes, void *stream) {
    if (dt != LA_DTYPE_F32 && dt != LA_DTYPE_BF16) return LA_ERR_UNSUPPORTED;
    if (B < 1 || H < 1 || N < 0) return LA_ERR_INVALID_ARG;
    if (!sizes_ok(B, H, N, d, dv, dt)) return LA_ERR_UNSUPPORTED;
    if (!(eps > 0.f) || !std::isfinite(eps)) return LA_ERR_INVALID_ARG;
    if ((S_out == nullptr) != (z_out == nullptr)) return LA_ERR_INVALID_ARG;
    if ((long long)B * H * (N > 0 ? N : 1) * std::max(d, dv) >= (1LL << 31))
        return LA_ERR_INVALID_ARG;
    const size_t BH = (size_t)B * H, es = dt == LA_DTYPE_BF16 ? 2 : 4;
    if (N == 0) {   // no tokens: the final state is zero
        if (S_out) {
            std::memset(S_out, 0, BH * d * dv * sizeof(float));
            std::memset(z_out, 0, BH * d * sizeof(float));
        }
        return LA_OK;
    }
    if (!q || !k || !v || !y) return LA_ERR_INVALID_ARG;
    const size_t T = BH * N;
    if (overlap(y, T * dv * 4, q, T * d * es) || overlap(y, T * dv * 4, k, T * d * es) ||
        overlap(y, T * dv * 4, v, T * dv * es))
        return LA_ERR_INVALID_ARG;
    const HostPlan p = make_plan(B, H, N, d, dv, dt);
    if (!dev_buf || dev_buf_bytes < p.err + kHostSets * p.set ||
        (reinterpret_cast<uintptr_t>(dev_buf) & 255u) != 0)
        return LA_ERR_WORKSPACE;

    CallResources r;
    if (!r.ok) return LA_ERR_CUDA;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    char *base = static_cast<char *>(dev_buf);
    unsigned int *err_dev = reinterpret_cast<unsigned int *>(base);
    bool cuda_ok = cudaMemsetAsync(err_dev, 0, p.err, cs) == cudaSuccess &&
                   cudaEventRecord(r.start, cs) == cudaSuccess &&
                   cudaStreamWaitEvent(r.up, r.start, 0) == cudaSuccess &&
                   cudaStreamWaitEvent(r.down, r.start, 0) == cudaSuccess;
    la_status st = LA_OK;
    const char *qh = static_cast<const char *>(q), *kh = static_cast<const char *>(k),
               *vh = static_cast<const char *>(v);
    for (int i = 0; cuda_ok && st == LA_OK && i < p.ngroups; ++i) {
        const int h0 = i * p.group_heads, hc = std::min(p.group_heads, p.BH - h0);
        const size_t Tc = (size_t)hc * N, tok0 = (size_t)h0 * N;
        char *set = base + p.err + (size_t)(i % kHostSets) * p.set;
        char *qd = set, *kd = qd + p.q, *vd = kd + p.q, *yd = vd + p.v;
        float *Sd = reinterpret_cast<float *>(yd + p.y);
        float *zd = reinterpret_cast<float *>(reinterpret_cast<char *>(Sd) + p.S);
        char *ws = reinterpret_cast<char *>(zd) + p.z;
        // the staging set is free once the download of group i - kHostSets is done
        if (i >= kHostSets) cuda_ok = cudaStreamWaitEvent(r.up, r.out[i - kHostSets], 0) == cudaSuccess;
        cuda_ok = cuda_ok &&
                  cudaMemcpyAsync(qd, qh + tok0 * d * es, Tc * d * es, cudaMemcpyHostToDevice, r.up) == cudaSuccess &&
                  cudaMemcpyAsync(kd, kh + tok0 * d * es, Tc * d * es, cudaMemcpyHostToDevice, r.up) == cudaSuccess &&
                  cudaMemcpyAsync(vd, vh + tok0 * dv * es, Tc * dv * es, cudaMemcpyHostToDevice, r.up) == cudaSuccess &&
                  cudaEventRecord(r.in[i], r.up) == cudaSuccess &&
                  cudaStreamWaitEvent(cs, r.in[i], 0) == cudaSuccess;
        if (!cuda_ok) break;
        st = la_forward_causal(qd, kd, vd, reinterpret_cast<float *>(yd), 1, hc, N, d, dv, dt, eps,
                               nullptr, nullptr, S_out ? Sd : nullptr, S_out ? zd : nullptr,
                               p.ws ? ws : nullptr, p.ws, cs);
        if (st != LA_OK) break;
        // keep the group's run-time status (its workspace header is reused)
        if (p.ws >= sizeof(WsHeader))
            cuda_ok = cudaMemcpyAsync(err_dev + i, ws, sizeof(unsigned int),
                                      cudaMemcpyDeviceToDevice, cs) == cudaSuccess;
        cuda_ok = cuda_ok && cudaEventRecord(r.done[i], cs) == cudaSuccess &&
                  cudaStreamWaitEvent(r.down, r.done[i], 0) == cudaSuccess &&
                  cudaMemcpyAsync(y + tok0 * dv, yd, Tc * dv * 4, cudaMemcpyDeviceToHost, r.down) == cudaSuccess;
        if (cuda_ok && S_out)
            cuda_ok = cudaMemcpyAsync(S_out + (size_t)h0 * d * dv, Sd, (size_t)hc * d * dv * 4,
                                      cudaMemcpyDeviceToHost, r.down) == cudaSuccess &&
                      cudaMemcpyAsync(z_out + (size_t)h0 * d, zd, (size_t)hc * d * 4,
                                      cudaMemcpyDeviceToHost, r.down) == cudaSuccess;
        cuda_ok = cuda_ok && cudaEventRecord(r.out[i], r.down) == cudaSuccess;
    }
    // wait for everything that was issued, whatever happened
    const bool synced = cudaStreamSynchronize(r.up) == cudaSuccess &&
                        cudaStreamSynchronize(cs) == cudaSuccess &&
                        cudaStreamSynchronize(r.down) == cudaSuccess;
    if (st != LA_OK) return st;
    if (!cuda_ok || !synced) return LA_ERR_CUDA;
    unsigned int errs[kHostGroups] = {};
    if (cudaMemcpy(errs, err_dev, sizeof(errs), cudaMemcpyDeviceToHost) != cudaSuccess)
        return LA_ERR_CUDA;
    for (int i = 0; i < p.ngroups; ++i)
        if (errs[i] != 0) return static_cast<la_status>(errs[i]);
    return LA_OK;
}

}  // extern "C"
