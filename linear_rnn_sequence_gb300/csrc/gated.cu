// gated.cu -- the gated recurrence and the feature-map choices on CUDA cores
// (fp32), and the random-feature map.
//
// Gated linear attention ("Linear Attention/es", "Variantes y extensiones":
// a data-dependent gate replaces RetNet's scalar decay):
//   S_t = diag(g_t) S_{t-1} + phi(k_t) v_t^T,  z_t = g_t * z_{t-1} + phi(k_t),
//   y_t = phi(q_t)^T S_t / max(phi(q_t)^T z_t, eps)
// with g_t in [0, 1] given per token, one value (gate_dim = 1) or one per
// feature row of S (gate_dim = d); without a gate g_t = 1.  phi is elu + 1 or
// the identity ("Mapas de características").
//
// causal_gated_kernel: one CTA per head walks the sequence token by token,
// as the fp32 causal kernel does (causal_simt.cu): S lives in registers
// (warp w owns a band of value columns, lane l a few feature rows), so
// phi(q_t)^T S_t is a reduce-scatter inside the warp.  Per 32-token chunk the
// features, the gates (broadcast to [chunk][d]) and z_t are staged in shared
// memory first; the next chunk's q, k, v are in flight meanwhile.  Per token
// and state element: one multiply by the gate and two FMAs.  z is carried in
// fp32 per feature (no split normaliser: with gates that vary per token the
// fp32 roundings of g z + phi(k) do not all lean one way, as they do under a
// fixed decay).
//
// random_features_kernel: phi(x) = exp(W x - ||x||^2 / 2) / sqrt(m) for
// every row x (the positive random features of "Mapas de características",
// Performer), W [m][d] staged in shared memory, one warp per row.
#include "la_device.cuh"
#include "la_internal.h"
#include "simt_tiles.cuh"

namespace la {
namespace {

using namespace tiles;

template <int D, int DV>
struct GatedCfg {
    static constexpr int kNT = D * DV >= 2048 ? 512 : 256;   // threads per CTA
    // sFq, sFk, sZt, sG [kBC][D]; sV, sY [kBC][DV]; sDinv [kBC]
    static constexpr size_t kSmemFloats = 4 * (size_t)kBC * D + 2 * (size_t)kBC * DV + kBC;
};

struct Feature {
    int kind;
    __device__ float operator()(float x) const { return feature_f(x, kind); }
};

template <int D, int DV, typename T>
__global__ void __launch_bounds__(GatedCfg<D, DV>::kNT, 1)
causal_gated_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                    float *__restrict__ y, int N, float eps, int phi,
                    const float *__restrict__ gate, int gate_dim,
                    const float *__restrict__ S_in, const float *__restrict__ z_in,
                    float *__restrict__ S_out, float *__restrict__ z_out,
                    const unsigned int *__restrict__ tc_skip)
{
    constexpr int NT = GatedCfg<D, DV>::kNT, NW = NT / 32;
    // heads the tensor-core kernel took are left alone (before any read or
    // write, so an S_in aliased by S_out stays intact for the other heads)
    if (tc_skip && tc_skip[blockIdx.x] == 0u) return;
    using CT = WarpRows<NT, DV, D>;   // warp: CT::RPW value columns; lane: CT::CPL features
    static_assert(NT >= D, "one thread per feature");
    extern __shared__ float4 smem4[];
    float *sFq = reinterpret_cast<float *>(smem4);  // [kBC][D] phi(q)
    float *sFk = sFq + kBC * D;                     // [kBC][D] phi(k)
    float *sZt = sFk + kBC * D;                     // [kBC][D] z_t
    float *sG = sZt + kBC * D;                      // [kBC][D] gate of token t, feature a
    float *sV = sG + kBC * D;                       // [kBC][DV]
    float *sY = sV + kBC * DV;                      // [kBC][DV]
    float *sDinv = sY + kBC * DV;                   // [kBC] 1 / max(den_t, eps)
    const int head = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b0 = warp * CT::RPW, a0 = lane * CT::CPL;
    const int my_col = b0 + CT::row_of(lane);
    const bool writer = CT::writer(lane);
    const Feature feat{phi};

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
    float z = (tid < D && z_in) ? z_in[(size_t)head * D + tid] : 0.f;   // thread a < D: z[a]

    const T *qh = q + (size_t)head * N * D, *kh = k + (size_t)head * N * D;
    const T *vh = v + (size_t)head * N * DV;
    const float *gh = gate ? gate + (size_t)head * N * gate_dim : nullptr;
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
        lq.store(sFq, L, feat);
        lk.store(sFk, L, feat);
        lv.store(sV, L, Ident());
        for (int e = tid; e < kBC * D; e += NT) {   // gates, broadcast over features
            const int t = e / D, a = e - t * D;
            sG[e] = (gh && t < L) ? gh[(size_t)(t0 + t) * gate_dim + (gate_dim == 1 ? 0 : a)] : 1.f;
        }
        __syncthreads();
        if (t0 + kBC < N) {   // the next chunk flies in during this one
            const int n0 = t0 + kBC, nL = min(kBC, N - n0);
            lq.load(qh + (size_t)n0 * D, nL); lk.load(kh + (size_t)n0 * D, nL);
            lv.load(vh + (size_t)n0 * DV, nL);
        }
        // z_t for every token of the chunk (thread a < D walks feature a)
        if (tid < D)
            for (int t = 0; t < L; ++t) {
                z = fmaf(sG[t * D + tid], z, sFk[t * D + tid]);
                sZt[t * D + tid] = z;
            }
        __syncthreads();
        // den_t = phi(q_t) . z_t
        for (int t = warp; t < L; t += NW) {
            float s = 0.f;
            for (int x = lane; x < D; x += 32) s = fmaf(sFq[t * D + x], sZt[t * D + x], s);
            s = warp_sum(s);
            if (lane == 0) sDinv[t] = 1.f / fmaxf(s, eps);
        }
        __syncthreads();
        // S_t = diag(g_t) S_{t-1} + phi(k_t) v_t^T, then y_t = phi(q_t)^T S_t / D_t
        for (int t = 0; t < L; ++t) {
            float fk[CT::CPL], fq[CT::CPL], gf[CT::CPL], vv[CT::RPW], acc[CT::RPW];
            ldn(sFk + t * D + a0, fk);
            ldn(sFq + t * D + a0, fq);
            ldn(sG + t * D + a0, gf);
            ldn(sV + t * DV + b0, vv);   // warp-uniform
            // each FMA updates a pair of value columns (packed), with the same
            // operations per element as the scalar form
            uint64_t fkb[CT::CPL], fqb[CT::CPL], gfb[CT::CPL];   // both lanes alike
#pragma unroll
            for (int j = 0; j < CT::CPL; ++j) {
                fkb[j] = pk2(fk[j], fk[j]);
                fqb[j] = pk2(fq[j], fq[j]);
                gfb[j] = pk2(gf[j], gf[j]);
            }
#pragma unroll
            for (int i = 0; i < RP; ++i) {
                const uint64_t vp = pk2(vv[2 * i], vv[2 * i + 1]);
                uint64_t accp = pk2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < CT::CPL; ++j) {
                    S2p[i][j] = fma2(fkb[j], vp, mul2(gfb[j], S2p[i][j]));
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
    if (z_out && tid < D) z_out[(size_t)head * D + tid] = z;
}

template <int D, int DV, typename T>
cudaError_t launch_typed(const FwdArgs &a) {
    constexpr size_t smem = GatedCfg<D, DV>::kSmemFloats * sizeof(float);
    auto kern = causal_gated_kernel<D, DV, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<a.BH(), GatedCfg<D, DV>::kNT, smem, a.stream>>>(
        (const T *)a.q, (const T *)a.k, (const T *)a.v, a.y, a.N, a.eps, a.phi, a.gate,
        a.gate_dim, a.S_in, a.z_in, a.S_out, a.z_out, a.gate_skip);
    return cudaGetLastError();
}

template <int D, int DV>
cudaError_t launch_dims(const FwdArgs &a) {
    return a.dt == LA_DTYPE_BF16 ? launch_typed<D, DV, __nv_bfloat16>(a)
                                 : launch_typed<D, DV, float>(a);
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

// ------------------------------------------------------------------ random features
constexpr int kRfWarps = 8;
constexpr int kRfRowsPerWarp = 4;

template <typename T>
__global__ void __launch_bounds__(kRfWarps * 32)
random_features_kernel(const T *__restrict__ x, float *__restrict__ out, long long rows, int d,
                       int m, const float *__restrict__ W)
{
    extern __shared__ float sW[];   // [m][d + 1] (padded: lanes read different rows)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ld = d + 1;
    for (int e = tid; e < m * d; e += kRfWarps * 32) sW[(e / d) * ld + e % d] = W[e];
    __syncthreads();
    const float scale = rsqrtf((float)m);
    float xr[4];   // this lane's features of the current row: x[lane + 32 c], d <= 128
    const long long r0 = ((long long)blockIdx.x * kRfWarps + warp) * kRfRowsPerWarp;
    for (int rr = 0; rr < kRfRowsPerWarp; ++rr) {
        const long long r = r0 + rr;
        if (r >= rows) break;
        float nrm = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int a = lane + 32 * c;
            xr[c] = a < d ? to_f(x[r * d + a]) : 0.f;
            nrm = fmaf(xr[c], xr[c], nrm);
        }
        nrm = warp_sum(nrm);
        // feature f = lane + 32 j: w_f . x with x broadcast from its owner lane
        for (int f0 = 0; f0 < m; f0 += 32) {
            const int f = f0 + lane;
            float wx = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (32 * c >= d) break;
                for (int l = 0; l < 32; ++l) {
                    const float xa = __shfl_sync(0xffffffffu, xr[c], l);
                    if (f < m) wx = fmaf(sW[f * ld + 32 * c + l], xa, wx);
                }
            }
            if (f < m) out[r * m + f] = scale * expf(wx - 0.5f * nrm);
        }
    }
}

}  // namespace

cudaError_t launch_causal_gated(const FwdArgs &a) {
    if (gated_tc_supported(a)) {
        // the tensor cores take the heads whose gates all lie in [2^-1/2, 1];
        // this kernel follows for the others
        cudaError_t e = cudaMemsetAsync(a.ws, 0, gated_tc_clear_bytes(a.BH()), a.stream);
        if (e == cudaSuccess) e = launch_gated_tc(a);
        if (e != cudaSuccess) return e;
        FwdArgs b = a;
        b.gate_skip = reinterpret_cast<const unsigned int *>(static_cast<const char *>(a.ws) +
                                                             sizeof(WsHeader));
        return launch_causal_gated_simt(b);
    }
    return launch_causal_gated_simt(a);
}

cudaError_t launch_causal_gated_simt(const FwdArgs &a) {
    switch (a.d) {
    case 32: return launch_d<32>(a);
    case 64: return launch_d<64>(a);
    case 128: return launch_d<128>(a);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_random_features(const void *x, float *out, long long rows, int d, int m,
                                   la_dtype dt, const float *W, cudaStream_t stream) {
    const size_t smem = sizeof(float) * (size_t)m * (d + 1);
    const long long per_cta = (long long)kRfWarps * kRfRowsPerWarp;
    const unsigned grid = (unsigned)((rows + per_cta - 1) / per_cta);
    if (dt == LA_DTYPE_BF16) {
        auto kern = random_features_kernel<__nv_bfloat16>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kRfWarps * 32, smem, stream>>>(static_cast<const __nv_bfloat16 *>(x), out,
                                                     rows, d, m, W);
    } else {
        auto kern = random_features_kernel<float>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<grid, kRfWarps * 32, smem, stream>>>(static_cast<const float *>(x), out, rows, d,
                                                     m, W);
    }
    return cudaGetLastError();
}

}  // namespace la
