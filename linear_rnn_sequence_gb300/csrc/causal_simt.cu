// causal_simt.cu -- chunked causal linear attention on CUDA cores, fp32.
//
// Blockwise form of "Linear Attention/es", "Entrenamiento: forma paralela":
// per block of C tokens, y_i = [sum_{j<=i in block} w_ij v_j + phi(q_i)^T S_prev]
//                            / max(sum_{j<=i in block} w_ij + phi(q_i)^T z_prev, eps)
// with w_ij = phi(q_i)^T phi(k_j), followed by S_prev += sum_j phi(k_j) v_j^T
// and z_prev += sum_j phi(k_j).  Everything is fp32 (FFMA), so this is the
// path for float32 inputs and for sizes the tensor-core kernel does not take.
//
// One CTA owns one head and one block of 32 value columns (columns of S and
// y are independent; the denominator is recomputed by each column block).
// The state S[:, cols] (d x 32) and z live in shared memory for the whole
// sequence; only q, k, v are read and y written.
//
// With a per-head decay gamma (RetNet in "Variantes y extensiones":
// S_t = gamma S_{t-1} + phi(k_t) v_t^T, z alike) token i of a block sees the
// pairs j <= i weighted by gamma^(i-j) and the state of the previous blocks
// by gamma^(i+1); after a block of L tokens the state becomes
// gamma^L S_prev + sum_j gamma^(L-1-j) phi(k_j) v_j^T.
#include "la_device.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kC = 32;        // tokens per block
constexpr int kCols = 32;     // value columns per CTA
constexpr int kThreads = 256;

template <int D>
struct SimtSmem {
    static constexpr int QS = D + 1;  // padded row stride for phi(Q), phi(K)
    static constexpr size_t bytes =
        sizeof(float) * (2 * kC * QS + kC * kCols + D * kCols + D + kC * (kC + 1) + 2 * kC + kC + 1);
};

template <int D, typename T, bool DECAY>
__global__ void __launch_bounds__(kThreads)
causal_simt_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   float *__restrict__ y, int N, int DV, float eps,
                   const float *__restrict__ S_in, const float *__restrict__ z_in,
                   float *__restrict__ S_out, float *__restrict__ z_out,
                   const float *__restrict__ gamma, int H)
{
    constexpr int QS = SimtSmem<D>::QS;
    extern __shared__ float sm[];
    float *Qs = sm;                       // [kC][QS]  phi(q)
    float *Ks = Qs + kC * QS;             // [kC][QS]  phi(k)
    float *Vs = Ks + kC * QS;             // [kC][kCols]
    float *Ss = Vs + kC * kCols;          // [D][kCols]
    float *zs = Ss + D * kCols;           // [D]
    float *Ps = zs + D;                   // [kC][kC+1] masked w_ij
    float *dinter = Ps + kC * (kC + 1);   // [kC] phi(q_i)^T z_prev
    float *dens = dinter + kC;            // [kC] clamped denominators
    float *pw = dens + kC;                // [kC+1] gamma^m

    const int head = blockIdx.x;
    const int col0 = blockIdx.y * kCols;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T *qh = q + (long)head * N * D;
    const T *kh = k + (long)head * N * D;
    const T *vh = v + (long)head * N * DV;
    float *yh = y + (long)head * N * DV;

    for (int i = tid; i < D * kCols; i += kThreads) {
        const int a = i / kCols, c = i % kCols;
        Ss[i] = S_in ? S_in[((long)head * D + a) * DV + col0 + c] : 0.f;
    }
    for (int a = tid; a < D; a += kThreads) zs[a] = z_in ? z_in[(long)head * D + a] : 0.f;
    if (DECAY && tid == 0) {
        const float g = gamma[head % H];
        float p = 1.f;
        for (int m = 0; m <= kC; ++m) {
            pw[m] = p;
            p *= g;
        }
    }

    for (int t0 = 0; t0 < N; t0 += kC) {
        const int L = min(kC, N - t0);
        __syncthreads();  // previous block's state update is complete
        for (int e = tid; e < kC * D; e += kThreads) {
            const int i = e / D, a = e % D;
            float fq = 0.f, fk = 0.f;  // rows past the end contribute nothing
            if (i < L) {
                fq = phi_f(to_f(qh[(long)(t0 + i) * D + a]));
                fk = phi_f(to_f(kh[(long)(t0 + i) * D + a]));
            }
            Qs[i * QS + a] = fq;
            Ks[i * QS + a] = fk;
        }
        for (int e = tid; e < kC * kCols; e += kThreads) {
            const int j = e / kCols, c = e % kCols;
            Vs[e] = j < L ? to_f(vh[(long)(t0 + j) * DV + col0 + c]) : 0.f;
        }
        __syncthreads();

        // w_ij for j <= i (thread: column j = lane, rows 4*warp .. 4*warp+3)
        {
            const int j = lane, i0 = warp * 4;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int a = 0; a < D; ++a) {
                const float kv = Ks[j * QS + a];
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[r] = fmaf(Qs[(i0 + r) * QS + a], kv, acc[r]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
                Ps[(i0 + r) * (kC + 1) + j] =
                    (j <= i0 + r) ? (DECAY ? acc[r] * pw[i0 + r - j] : acc[r]) : 0.f;
        }
        if (tid < kC) {
            float s = 0.f;
            for (int a = 0; a < D; ++a) s = fmaf(Qs[tid * QS + a], zs[a], s);
            dinter[tid] = DECAY ? s * pw[tid + 1] : s;
        }
        __syncthreads();
        if (tid < kC) {
            float s = dinter[tid];
            for (int j = 0; j <= tid; ++j) s += Ps[tid * (kC + 1) + j];
            dens[tid] = fmaxf(s, eps);
        }
        __syncthreads();

        // numerators and outputs (thread: column c = lane, rows 4*warp ..)
        {
            const int c = lane, i0 = warp * 4;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int a = 0; a < D; ++a) {
                const float s = Ss[a * kCols + c];
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[r] = fmaf(Qs[(i0 + r) * QS + a], s, acc[r]);
            }
            if (DECAY)
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[r] *= pw[i0 + r + 1];
            for (int j = 0; j < kC; ++j) {
                const float vj = Vs[j * kCols + c];
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[r] = fmaf(Ps[(i0 + r) * (kC + 1) + j], vj, acc[r]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
                if (i0 + r < L) yh[(long)(t0 + i0 + r) * DV + col0 + c] = acc[r] / dens[i0 + r];
        }
        __syncthreads();

        // state update: S[a][c] += sum_j phi(k_j)[a] v_j[c];  z += sum_j phi(k_j)
        if (DECAY) {   // gamma^L S_prev + sum_{j<L} gamma^(L-1-j) phi(k_j) v_j^T
            for (int e = tid; e < D * kCols; e += kThreads) {
                const int a = e / kCols, c = e % kCols;
                float s = Ss[e] * pw[L];
                for (int j = 0; j < L; ++j) s = fmaf(Ks[j * QS + a] * pw[L - 1 - j], Vs[j * kCols + c], s);
                Ss[e] = s;
            }
            for (int a = tid; a < D; a += kThreads) {
                float s = zs[a] * pw[L];
                for (int j = 0; j < L; ++j) s = fmaf(Ks[j * QS + a], pw[L - 1 - j], s);
                zs[a] = s;
            }
        } else {
            for (int e = tid; e < D * kCols; e += kThreads) {
                const int a = e / kCols, c = e % kCols;
                float s = Ss[e];
                for (int j = 0; j < kC; ++j) s = fmaf(Ks[j * QS + a], Vs[j * kCols + c], s);
                Ss[e] = s;
            }
            for (int a = tid; a < D; a += kThreads) {
                float s = zs[a];
                for (int j = 0; j < kC; ++j) s += Ks[j * QS + a];
                zs[a] = s;
            }
        }
    }
    __syncthreads();
    if (S_out)
        for (int i = tid; i < D * kCols; i += kThreads) {
            const int a = i / kCols, c = i % kCols;
            S_out[((long)head * D + a) * DV + col0 + c] = Ss[i];
        }
    if (z_out && blockIdx.y == 0)
        for (int a = tid; a < D; a += kThreads) z_out[(long)head * D + a] = zs[a];
}

template <int D, typename T, bool DECAY>
cudaError_t launch_t(const FwdArgs &a) {
    const size_t smem = SimtSmem<D>::bytes;
    auto kern = causal_simt_kernel<D, T, DECAY>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.BH(), a.dv / kCols);
    kern<<<grid, kThreads, smem, a.stream>>>((const T *)a.q, (const T *)a.k, (const T *)a.v,
                                             a.y, a.N, a.dv, a.eps, a.S_in, a.z_in, a.S_out,
                                             a.z_out, a.gamma, a.H);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const FwdArgs &a) {
    if (a.gamma)
        return a.dt == LA_DTYPE_BF16 ? launch_t<D, __nv_bfloat16, true>(a) : launch_t<D, float, true>(a);
    return a.dt == LA_DTYPE_BF16 ? launch_t<D, __nv_bfloat16, false>(a) : launch_t<D, float, false>(a);
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
