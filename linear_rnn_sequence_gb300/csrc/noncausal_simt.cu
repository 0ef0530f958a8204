// noncausal_simt.cu -- non-causal linear attention on CUDA cores, fp32, with
// the feature map elu + 1 or the identity ("Mapas de características").
//
// "Linear Attention/es", "Reformulación con núcleos": S = sum_j phi(k_j) v_j^T
// and z = sum_j phi(k_j) do not depend on the query, so they are reduced once
// and reused by every query: y_i = phi(q_i)^T S / max(phi(q_i)^T z, eps).
//
// Pass 1 (state_partials): CTA (head, split, column block) sums its token
//   range into a partial S[:, cols] (registers) and z; partials go to the
//   workspace.
// Pass 2 (queries): CTA (head, token tile, column block) adds the partials in
//   a fixed order (deterministic), then evaluates its queries.
#include "la_device.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kC = 32, kCols = 32, kThreads = 256, kTile = 64;

int num_splits(int BH, int N) {
    // about 256 tokens per split, at most 64 splits, enough CTAs for 152 SMs
    int s = (N + 255) / 256;
    if (s > 64) s = 64;
    if (s < 1) s = 1;
    (void)BH;
    return s;
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads)
state_partials_kernel(const T *__restrict__ k, const T *__restrict__ v, int N, int DV, int nsplit,
                      float *__restrict__ Sp, float *__restrict__ zp, int phi)
{
    constexpr int QS = D + 1, RPT = D / 8;
    __shared__ float Ks[kC * QS];
    __shared__ float Vs[kC * kCols];
    const int head = blockIdx.x, split = blockIdx.y, col0 = blockIdx.z * kCols;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (N + nsplit - 1) / nsplit;
    const int tb = split * per, te = min(N, tb + per);
    const T *kh = k + (long)head * N * D;
    const T *vh = v + (long)head * N * DV;
    float acc[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) acc[r] = 0.f;
    float zacc = 0.f;
    for (int t0 = tb; t0 < te; t0 += kC) {
        const int L = min(kC, te - t0);
        __syncthreads();
        for (int e = tid; e < kC * D; e += kThreads) {
            const int j = e / D, a = e % D;
            Ks[j * QS + a] = j < L ? feature_f(to_f(kh[(long)(t0 + j) * D + a]), phi) : 0.f;
        }
        for (int e = tid; e < kC * kCols; e += kThreads) {
            const int j = e / kCols, c = e % kCols;
            Vs[e] = j < L ? to_f(vh[(long)(t0 + j) * DV + col0 + c]) : 0.f;
        }
        __syncthreads();
        for (int j = 0; j < kC; ++j) {
            const float vj = Vs[j * kCols + lane];
#pragma unroll
            for (int r = 0; r < RPT; ++r) acc[r] = fmaf(Ks[j * QS + warp + 8 * r], vj, acc[r]);
        }
        if (tid < D)
            for (int j = 0; j < kC; ++j) zacc += Ks[j * QS + tid];
    }
    float *Sdst = Sp + ((long)head * nsplit + split) * D * DV;
#pragma unroll
    for (int r = 0; r < RPT; ++r) Sdst[(long)(warp + 8 * r) * DV + col0 + lane] = acc[r];
    if (blockIdx.z == 0 && tid < D) zp[((long)head * nsplit + split) * D + tid] = zacc;
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads)
queries_kernel(const T *__restrict__ q, float *__restrict__ y, int N, int DV, int nsplit,
               const float *__restrict__ Sp, const float *__restrict__ zp, float eps,
               float *__restrict__ S_out, float *__restrict__ z_out, int phi)
{
    constexpr int QS = D + 1;
    extern __shared__ float sm[];
    float *Ss = sm;                  // [D][kCols]
    float *zs = Ss + D * kCols;      // [D]
    float *Qs = zs + D;              // [kTile][QS]
    float *dens = Qs + kTile * QS;   // [kTile]
    const int head = blockIdx.x, t0 = blockIdx.y * kTile, col0 = blockIdx.z * kCols;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = min(kTile, N - t0);

    for (int e = tid; e < D * kCols; e += kThreads) {
        const int a = e / kCols, c = e % kCols;
        float s = 0.f;
        for (int p = 0; p < nsplit; ++p)
            s += Sp[(((long)head * nsplit + p) * D + a) * DV + col0 + c];
        Ss[e] = s;
    }
    for (int a = tid; a < D; a += kThreads) {
        float s = 0.f;
        for (int p = 0; p < nsplit; ++p) s += zp[((long)head * nsplit + p) * D + a];
        zs[a] = s;
    }
    const T *qh = q + (long)head * N * D;
    for (int e = tid; e < kTile * D; e += kThreads) {
        const int i = e / D, a = e % D;
        Qs[i * QS + a] = i < L ? feature_f(to_f(qh[(long)(t0 + i) * D + a]), phi) : 0.f;
    }
    __syncthreads();
    if (blockIdx.y == 0) {
        if (S_out)
            for (int e = tid; e < D * kCols; e += kThreads) {
                const int a = e / kCols, c = e % kCols;
                S_out[((long)head * D + a) * DV + col0 + c] = Ss[e];
            }
        if (z_out && blockIdx.z == 0)
            for (int a = tid; a < D; a += kThreads) z_out[(long)head * D + a] = zs[a];
    }
    if (tid < kTile) {
        float s = 0.f;
        for (int a = 0; a < D; ++a) s = fmaf(Qs[tid * QS + a], zs[a], s);
        dens[tid] = fmaxf(s, eps);
    }
    __syncthreads();
    const int i0 = warp * 8;
    float acc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = 0.f;
    for (int a = 0; a < D; ++a) {
        const float s = Ss[a * kCols + lane];
#pragma unroll
        for (int r = 0; r < 8; ++r) acc[r] = fmaf(Qs[(i0 + r) * QS + a], s, acc[r]);
    }
    float *yh = y + (long)head * N * DV;
#pragma unroll
    for (int r = 0; r < 8; ++r)
        if (i0 + r < L) yh[(long)(t0 + i0 + r) * DV + col0 + lane] = acc[r] / dens[i0 + r];
}

template <int D, typename T>
cudaError_t launch_t(const FwdArgs &a) {
    const int BH = a.BH(), ns = num_splits(BH, a.N);
    float *Sp = reinterpret_cast<float *>(static_cast<char *>(a.ws) + sizeof(WsHeader));
    float *zp = Sp + (size_t)BH * ns * a.d * a.dv;
    state_partials_kernel<D, T><<<dim3(BH, ns, a.dv / kCols), kThreads, 0, a.stream>>>(
        (const T *)a.k, (const T *)a.v, a.N, a.dv, ns, Sp, zp, a.phi);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = sizeof(float) * (D * kCols + D + kTile * (D + 1) + kTile);
    auto kern = queries_kernel<D, T>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(BH, (a.N + kTile - 1) / kTile, a.dv / kCols), kThreads, smem, a.stream>>>(
        (const T *)a.q, a.y, a.N, a.dv, ns, Sp, zp, a.eps, a.S_out, a.z_out, a.phi);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const FwdArgs &a) {
    return a.dt == LA_DTYPE_BF16 ? launch_t<D, __nv_bfloat16>(a) : launch_t<D, float>(a);
}

}  // namespace

size_t noncausal_simt_workspace(int BH, int N, int d, int dv) {
    const size_t ns = num_splits(BH, N);
    return sizeof(WsHeader) + sizeof(float) * (size_t)BH * ns * ((size_t)d * dv + d);
}

cudaError_t launch_noncausal_simt(const FwdArgs &a) {
    switch (a.d) {
    case 32: return launch_d<32>(a);
    case 64: return launch_d<64>(a);
    case 128: return launch_d<128>(a);
    }
    return cudaErrorInvalidValue;
}

}  // namespace la
