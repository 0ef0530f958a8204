// causal_simt.cu -- causal linear attention on CUDA cores, fp32, token by
// token, with an optional per-head decay.
//
// The recurrence of "Linear Attention/es", "Forma recurrente e inferencia
// autorregresiva":
//   S_t = gamma S_{t-1} + phi(k_t) v_t^T,  z_t = gamma z_{t-1} + phi(k_t),
//   y_t = phi(q_t)^T S_t / max(phi(q_t)^T z_t, eps)
// with gamma = 1 for the plain form and one gamma per head for RetNet's
// decay ("Variantes y extensiones"; z is decayed like S so that y stays a
// normalised average).  Everything is fp32 FMA, so this is the path for
// float32 inputs, for d or dv = 32, and for the decay.
//
// One CTA owns one head for the whole sequence.  Its state S lives in
// registers: warp w owns a band of value columns and lane l a few feature
// rows of each, so phi(q_t)^T S_t (a sum over rows) is a reduce-scatter
// inside the warp and every lane finishes one column of y_t.  z_t and the
// denominators of a 32-token chunk are formed before its token loop (one
// thread per feature walks the chunk; one warp per token takes the dot
// product), and the next chunk's q, k, v are in flight from HBM during the
// current chunk's tokens.  Per token and state element: one multiply (decay
// only) and two FMAs.
//
// With a decay the normaliser is carried split, z = n 1 + zeta with n the
// decayed token count (in fp64, one thread) and zeta = sum gamma^(t-j)
// psi(k_j): z settles near 1/(1 - gamma), where fp32 roundings of
// gamma z + phi(k) all lean the same way and would bias it by up to
// 2^-24 / (1 - gamma); the increments of zeta are small, so its bias is not.
#include "la_device.cuh"
#include "la_internal.h"
#include "simt_tiles.cuh"

namespace la {
namespace {

using namespace tiles;

template <int D, int DV>
struct FwdCfg {
    static constexpr int kNT = D * DV >= 2048 ? 512 : 256;   // threads per CTA
    static constexpr size_t kSmemFloats = 3 * (size_t)kBC * D + 2 * (size_t)kBC * DV + kBC;
};

template <int D, int DV, typename T, bool DECAY>
__global__ void __launch_bounds__(FwdCfg<D, DV>::kNT, 1)
causal_rec_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                  float *__restrict__ y, int N, int H, float eps,
                  const float *__restrict__ gamma, const float *__restrict__ S_in,
                  const float *__restrict__ z_in, float *__restrict__ S_out,
                  float *__restrict__ z_out, bool skip_tc_heads)
{
    constexpr int NT = FwdCfg<D, DV>::kNT, NW = NT / 32;
    using CT = WarpRows<NT, DV, D>;   // warp: CT::RPW value columns; lane: CT::CPL features
    static_assert(NT >= D, "one thread per feature");
    extern __shared__ float4 smem4[];
    float *sFq = reinterpret_cast<float *>(smem4);  // [kBC][D] phi(q)
    float *sFk = sFq + kBC * D;                     // [kBC][D] phi(k)
    float *sZt = sFk + kBC * D;                     // [kBC][D] z_t
    float *sV = sZt + kBC * D;                      // [kBC][DV]
    float *sY = sV + kBC * DV;                      // [kBC][DV]
    float *sDinv = sY + kBC * DV;                   // [kBC] 1 / max(den_t, eps)
    const int head = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b0 = warp * CT::RPW, a0 = lane * CT::CPL;
    const int my_col = b0 + CT::row_of(lane);
    const bool writer = CT::writer(lane);
    const float g = DECAY ? gamma[head % H] : 1.f;
    // heads the tensor-core kernel has already computed (whole CTA leaves)
    if (DECAY && skip_tc_heads && decay_on_tensor_cores(g)) return;

    // S[a0 + j][b0 + i] in S2p[i / 2][j], packed pairs of value columns
    // (2i', 2i' + 1); S_in is read in full before S_out is written
    constexpr int RP = CT::RPW / 2;
    uint64_t S2p[RP][CT::CPL];
    const float *Sh_in = S_in ? S_in + (size_t)head * D * DV : nullptr;
#pragma unroll
    for (int i = 0; i < RP; ++i)
#pragma unroll
        for (int j = 0; j < CT::CPL; ++j)
            S2p[i][j] = Sh_in ? pk2(Sh_in[(a0 + j) * DV + b0 + 2 * i], Sh_in[(a0 + j) * DV + b0 + 2 * i + 1])
                              : pk2(0.f, 0.f);
    const uint64_t g2 = pk2(g, g);
    // thread a < D carries z[a] (with a decay: zeta[a]); thread NT - 1 the
    // decayed count n, which starts at the mean of z_in
    float z = (tid < D && z_in) ? z_in[(size_t)head * D + tid] : 0.f;
    double n = 0.0;
    if constexpr (DECAY) {
        if (tid == NT - 1 && z_in) {
            for (int a = 0; a < D; ++a) n += z_in[(size_t)head * D + a];
            n /= D;
            sDinv[0] = (float)n;
        }
        __syncthreads();
        if (tid < D && z_in) z -= sDinv[0];
    }

    const T *qh = q + (size_t)head * N * D, *kh = k + (size_t)head * N * D;
    const T *vh = v + (size_t)head * N * DV;
    float *yh = y + (size_t)head * N * DV;
    ChunkLoad<D, T, NT> lq, lk;
    ChunkLoad<DV, T, NT> lv;
    if (N > 0) {
        const int L = min(kBC, N);
        lq.load(qh, L); lk.load(kh, L); lv.load(vh, L);
    }
    for (int t0 = 0; t0 < N; t0 += kBC) {
        const int L = min(kBC, N - t0);
        __syncthreads();   // the previous chunk is consumed and its y written
        lq.store(sFq, L, Phi());
        lk.store(sFk, L, Phi());
        lv.store(sV, L, Ident());
        __syncthreads();
        if (t0 + kBC < N) {   // the next chunk flies in during this one
            const int n0 = t0 + kBC, nL = min(kBC, N - n0);
            lq.load(qh + (size_t)n0 * D, nL); lk.load(kh + (size_t)n0 * D, nL);
            lv.load(vh + (size_t)n0 * DV, nL);
        }
        // z_t (with a decay: zeta_t and n_t) for every token of the chunk
        if (tid < D)
            for (int t = 0; t < L; ++t) {
                z = DECAY ? fmaf(g, z, sFk[t * D + tid] - 1.f) : z + sFk[t * D + tid];
                sZt[t * D + tid] = z;
            }
        if (DECAY && tid == NT - 1)
            for (int t = 0; t < L; ++t) {
                n = fma((double)g, n, 1.0);
                sY[t] = (float)n;   // sY is free until the token loop
            }
        __syncthreads();
        // den_t = phi(q_t) . z_t (with a decay: n_t sum(phi(q_t)) + phi(q_t) . zeta_t)
        for (int t = warp; t < L; t += NW) {
            float s = 0.f, sq = 0.f;
            for (int x = lane; x < D; x += 32) {
                s = fmaf(sFq[t * D + x], sZt[t * D + x], s);
                if (DECAY) sq += sFq[t * D + x];
            }
            s = warp_sum(s);
            if (DECAY) s = fmaf(sY[t], warp_sum(sq), s);
            if (lane == 0) sDinv[t] = 1.f / fmaxf(s, eps);
        }
        __syncthreads();
        // S_t = gamma S_{t-1} + phi(k_t) v_t^T, then y_t = phi(q_t)^T S_t / D_t
        for (int t = 0; t < L; ++t) {
            float fk[CT::CPL], fq[CT::CPL], vv[CT::RPW], acc[CT::RPW];
            ldn(sFk + t * D + a0, fk);
            ldn(sFq + t * D + a0, fq);
            ldn(sV + t * DV + b0, vv);   // warp-uniform
            // each FMA updates a pair of value columns (packed), with the same
            // operations per element as the scalar form
            uint64_t fkb[CT::CPL], fqb[CT::CPL];   // each feature in both lanes
#pragma unroll
            for (int j = 0; j < CT::CPL; ++j) {
                fkb[j] = pk2(fk[j], fk[j]);
                fqb[j] = pk2(fq[j], fq[j]);
            }
#pragma unroll
            for (int i = 0; i < RP; ++i) {
                const uint64_t vp = pk2(vv[2 * i], vv[2 * i + 1]);
                uint64_t accp = pk2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < CT::CPL; ++j) {
                    S2p[i][j] = fma2(fkb[j], vp, DECAY ? mul2(g2, S2p[i][j]) : S2p[i][j]);
                    accp = fma2(S2p[i][j], fqb[j], accp);
                }
                unpk2(accp, acc[2 * i], acc[2 * i + 1]);
            }
            const float num = reduce_scatter<CT::RPW>(acc, lane);
            if (writer) sY[t * DV + my_col] = num * sDinv[t];
        }
        __syncthreads();
        for (int e = tid * 4; e < L * DV; e += NT * 4) st4(yh + (size_t)t0 * DV + e, ld4(sY + e));
    }
    if (S_out) {
        float *So = S_out + (size_t)head * D * DV;
#pragma unroll
        for (int i = 0; i < RP; ++i)
#pragma unroll
            for (int j = 0; j < CT::CPL; ++j)
                unpk2(S2p[i][j], So[(a0 + j) * DV + b0 + 2 * i], So[(a0 + j) * DV + b0 + 2 * i + 1]);
    }
    if constexpr (DECAY) {
        __syncthreads();
        if (tid == NT - 1) sDinv[0] = (float)n;
        __syncthreads();
        z += sDinv[0];
    }
    if (z_out && tid < D) z_out[(size_t)head * D + tid] = z;
}

template <int D, int DV, typename T, bool DECAY>
cudaError_t launch_typed(const FwdArgs &a) {
    constexpr size_t smem = FwdCfg<D, DV>::kSmemFloats * sizeof(float);
    auto kern = causal_rec_kernel<D, DV, T, DECAY>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<a.BH(), FwdCfg<D, DV>::kNT, smem, a.stream>>>(
        (const T *)a.q, (const T *)a.k, (const T *)a.v, a.y, a.N, a.H, a.eps, a.gamma, a.S_in,
        a.z_in, a.S_out, a.z_out, a.skip_tc_heads);
    return cudaGetLastError();
}

template <int D, int DV>
cudaError_t launch_dims(const FwdArgs &a) {
    if (a.gamma)
        return a.dt == LA_DTYPE_BF16 ? launch_typed<D, DV, __nv_bfloat16, true>(a)
                                     : launch_typed<D, DV, float, true>(a);
    return a.dt == LA_DTYPE_BF16 ? launch_typed<D, DV, __nv_bfloat16, false>(a)
                                 : launch_typed<D, DV, float, false>(a);
}

template <int D>
cudaError_t launch_d(const FwdArgs &a) {
    switch (a.dv) {
    case 32: return launch_dims<D, 32>(a);
    case 64: return launch_dims<D, 64>(a);
    case 128: return launch_dims<D, 128>(a);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_causal_simt(const FwdArgs &a) {
    switch (a.d) {
    case 32: return launch_d<32>(a);
    case 64: return launch_d<64>(a);
    case 128: return launch_d<128>(a);
    }
    return cudaErrorInvalidValue;
}

}  // namespace la
