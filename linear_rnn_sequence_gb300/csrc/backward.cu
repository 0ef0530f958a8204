// backward.cu -- gradients of the causal form on CUDA cores, fp32.
//
// Training through the causal recurrence ("Linear Attention/es",
// "Entrenamiento: forma paralela") needs dL/dq, dL/dk, dL/dv for an upstream
// gradient dy = dL/dy.  By the chain rule through the recurrence of
// "Forma recurrente e inferencia autorregresiva", with
//   z_t = z_in + sum_{j<=t} phi(k_j),  S_t = S_in + sum_{j<=t} phi(k_j) v_j^T,
//   den_t = phi(q_t)^T z_t,  D_t = max(den_t, eps),  y_t = S_t^T phi(q_t) / D_t:
//   g_t = dy_t / D_t,  h_t = S_t g_t
//   e_t = -(phi(q_t) . h_t) / D_t  if den_t >= eps, else 0      (dL/d den_t)
//   dL/dphi(q_t) = h_t + z_t e_t
//   Sh_t = sum_{s>=t} phi(q_s) g_s^T,  zh_t = sum_{s>=t} phi(q_s) e_s
//   dL/dphi(k_t) = Sh_t v_t + zh_t,    dL/dv_t = Sh_t^T phi(k_t)
//   dL/dS_in = Sh_1,  dL/dz_in = zh_1
// and dL/dx = dL/dphi(x) * phi'(x), phi'(x) = 1 (x > 0), e^x (x <= 0), which
// is min(phi(x), 1).
//
// Precision.  y_t is a weighted mean of the v_j, so in dL/dphi(q_t) the two
// terms h_t and z_t e_t agree to leading order and their difference is about
// ten times smaller than either; the rounding of S_t, summed over thousands
// of tokens, would be amplified by that factor.  phi = 1 + psi (psi = elu) is
// therefore carried split, as S_t = 1 u_t^T + R_t and z_t = n_t 1 + zeta_t
// with u_t = sum v_j, n_t the token count, R_t = sum psi(k_j) v_j^T and
// zeta_t = sum psi(k_j) (an initial state is split the same way, u_in and
// n_in being its row means).  With hR = R_t g_t, and den_t = n_t sum(phi(q_t))
// + phi(q_t).zeta_t, the leading terms cancel algebraically:
//   dL/dphi(q_t) = c_t 1 + hR + zeta_t e_t,
//   c_t = ((u_t.g_t)(phi(q_t).zeta_t) - n_t (phi(q_t).hR)) / D_t,
//   e_t = -(sum(phi(q_t)) (u_t.g_t) + phi(q_t).hR) / D_t
// (when the clamp is active e_t = 0 and c_t = u_t.g_t).  Everything is fp32 FMA.
//
// Decay.  With RetNet's per-head decay ("Variantes y extensiones":
// S_t = gamma S_{t-1} + phi(k_t) v_t^T, z alike) every recurrence above
// carries gamma (Sh_t = phi(q_t) g_t^T + gamma Sh_{t+1}), the split holds with
// decayed u, n, zeta and R, and dL/dS_in = gamma Sh_1.  The decayed count n
// is kept in fp64: near its steady state 1/(1 - gamma) every fp32 rounding
// of gamma n + 1 leans the same way.  For gamma >= 1/4 the states are carried
// rescaled within each chunk, so the decay costs no multiply per element.
//
// Work split: the sequence of each head is cut into P segments of whole
// 32-token chunks.  Up to six launches:
//   0. seed        split S_in, z_in into (R, zeta, u, n)         (S_in only)
//   1. kv_states   per (head, segment < P-1): its (R, zeta, u, n) sums (P > 1)
//   2. scan        exclusive prefix over segments, from the seed
//   3. dq          per (head, segment), tokens in order from the prefix:
//                  dq; per token 1/D_t and e_t into the workspace; the
//                  segment's own sums of phi(q) g^T and phi(q) e
//   4. scan        exclusive suffix over segments of those sums (P > 1;
//                  with one segment the reverse pass starts from zero)
//   5. dkdv        per (head, segment), tokens in reverse from the suffix:
//                  dk, dv; segment 0 ends with dL/dS_in, dL/dz_in
// Inside a CTA the state lives in registers: warp w owns a band of rows and
// lane l a few columns of each, so the row's operands are warp-uniform
// broadcasts from shared memory and a reduction over value columns stays in
// the warp (a reduce-scatter: each lane ends with one finished row).  dv needs
// reductions over rows; the reverse pass writes per-warp partial sums to
// shared memory and adds them across the warps every 8 tokens.  While a chunk
// is processed the next one is already in flight from global memory into
// registers.
#include <algorithm>
#include <type_traits>

#include "la_device.cuh"
#include "la_internal.h"
#include "simt_tiles.cuh"

namespace la {
namespace {

using namespace tiles;

// Accumulator type of the decayed token count (see bwd_dq_kernel).
template <bool DECAY>
using NAcc = typename std::conditional<DECAY, double, float>::type;

template <int D, int DV>
struct Cfg {
    static constexpr int kNT = D * DV >= 2048 ? 512 : 256;   // threads per CTA
    // per (head, segment): R or Sh [D][DV], zeta or zh [D], u [DV], n, padding
    static constexpr int kE = D * DV + D + DV + 4;
    static constexpr int kOffZ = D * DV, kOffU = D * DV + D, kOffN = D * DV + D + DV;
};

struct Seg {
    int h, p, t0, t1;
};
__device__ __forceinline__ Seg segment(int P, int seg_chunks, int N) {
    Seg s;
    s.h = blockIdx.x / P;
    s.p = blockIdx.x % P;
    s.t0 = s.p * seg_chunks * kBC;
    s.t1 = min(N, s.t0 + seg_chunks * kBC);
    return s;
}

// ---- 0. split an initial state into (R, zeta, u, n) -------------------------
template <int D, int DV>
__global__ void bwd_seed_kernel(const float *__restrict__ S_in, const float *__restrict__ z_in,
                                float *__restrict__ seed)
{
    using C = Cfg<D, DV>;
    __shared__ float su[DV];
    __shared__ float sn;
    const int h = blockIdx.x;
    const float *S = S_in + (size_t)h * D * DV, *z = z_in + (size_t)h * D;
    float *o = seed + (size_t)h * C::kE;
    for (int b = threadIdx.x; b < DV; b += blockDim.x) {
        float s = 0.f;
        for (int a = 0; a < D; ++a) s += S[a * DV + b];
        su[b] = s / D;
        o[C::kOffU + b] = su[b];
    }
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int a = 0; a < D; ++a) s += z[a];
        sn = s / D;
        o[C::kOffN] = sn;
        o[C::kOffN + 1] = o[C::kOffN + 2] = o[C::kOffN + 3] = 0.f;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < D * DV; e += blockDim.x) o[e] = S[e] - su[e % DV];
    for (int a = threadIdx.x; a < D; a += blockDim.x) o[C::kOffZ + a] = z[a] - sn;
}

// ---- 1. per-segment sums (R, zeta, u, n) ------------------------------------
// DECAY: the sums are of the decayed recurrence, each token weighted by
// gamma^(segment end - 1 - token).
template <int D, int DV, typename T, bool DECAY>
__global__ void __launch_bounds__(Cfg<D, DV>::kNT, 1)
bwd_kv_states_kernel(const T *__restrict__ k, const T *__restrict__ v, int N, int P,
                     int seg_chunks, float *__restrict__ states, const float *__restrict__ gamma,
                     int H)
{
    using C = Cfg<D, DV>;
    constexpr int NT = C::kNT;
    using RT = WarpRows<NT, D, DV>;
    extern __shared__ float4 smem4[];
    float *sPk = reinterpret_cast<float *>(smem4);   // [kBC][D] psi(k)
    float *sV = sPk + kBC * D;                        // [kBC][DV]
    const Seg sg = segment(P, seg_chunks, N);
    if (sg.p == P - 1) return;   // no later segment reads the last one's sums
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = warp * RT::RPW, c0 = lane * RT::CPL;
    const float gm = DECAY ? gamma[sg.h % H] : 1.f;
    const uint64_t gm2 = pk2(gm, gm);
    // R as packed pairs of rows: Rp[i][c] = (R[2i][c], R[2i+1][c])
    constexpr int RP = RT::RPW / 2;
    uint64_t Rp[RP][RT::CPL];
#pragma unroll
    for (int i = 0; i < RP; ++i)
#pragma unroll
        for (int c = 0; c < RT::CPL; ++c) Rp[i][c] = pk2(0.f, 0.f);
    float zeta = 0.f, u = 0.f;
    ChunkLoad<D, T, NT> lk;
    ChunkLoad<DV, T, NT> lv;
    lk.load(k + ((size_t)sg.h * N + sg.t0) * D, min(kBC, sg.t1 - sg.t0));
    lv.load(v + ((size_t)sg.h * N + sg.t0) * DV, min(kBC, sg.t1 - sg.t0));
    for (int t0 = sg.t0; t0 < sg.t1; t0 += kBC) {
        const int L = min(kBC, sg.t1 - t0);
        __syncthreads();
        lk.store(sPk, L, Psi());
        lv.store(sV, L, Ident());
        __syncthreads();
        if (t0 + kBC < sg.t1) {
            const size_t nrow = (size_t)sg.h * N + t0 + kBC;
            const int nL = min(kBC, sg.t1 - t0 - kBC);
            lk.load(k + nrow * D, nL);
            lv.load(v + nrow * DV, nL);
        }
        if (tid < D)
            for (int t = 0; t < L; ++t)
                zeta = DECAY ? fmaf(gm, zeta, sPk[t * D + tid]) : zeta + sPk[t * D + tid];
        else if (tid < D + DV)
            for (int t = 0; t < L; ++t)
                u = DECAY ? fmaf(gm, u, sV[t * DV + tid - D]) : u + sV[t * DV + tid - D];
        for (int t = 0; t < L; ++t) {
            float pk[RT::RPW], x[RT::CPL];
            ldn(sPk + t * D + r0, pk);
            ldn(sV + t * DV + c0, x);
#pragma unroll
            for (int i = 0; i < RP; ++i) {
                const uint64_t pkp = pk2(pk[2 * i], pk[2 * i + 1]);
#pragma unroll
                for (int c = 0; c < RT::CPL; ++c)
                    Rp[i][c] = fma2(pkp, pk2(x[c], x[c]), DECAY ? mul2(gm2, Rp[i][c]) : Rp[i][c]);
            }
        }
    }
    float *out = states + ((size_t)sg.h * P + sg.p) * C::kE;
#pragma unroll
    for (int i = 0; i < RP; ++i)
#pragma unroll
        for (int c = 0; c < RT::CPL; ++c)
            unpk2(Rp[i][c], out[(r0 + 2 * i) * DV + c0 + c], out[(r0 + 2 * i + 1) * DV + c0 + c]);
    if (tid < D) out[C::kOffZ + tid] = zeta;
    else if (tid < D + DV) out[C::kOffU + tid - D] = u;
    if (tid < 4) {
        // the (decayed) token count; with a decay in fp64: near its steady
        // state 1/(1 - gamma) every fp32 rounding of gamma n + 1 leans the
        // same way, a bias of up to 2^-24 / (1 - gamma)
        NAcc<DECAY> n = 0;
        if (tid == 0)
            for (int t = sg.t0; t < sg.t1; ++t) n = DECAY ? fma((NAcc<DECAY>)gm, n, NAcc<DECAY>(1)) : n + 1;
        out[C::kOffN + tid] = (float)n;
    }
}

// ---- 2./4. exclusive scan over segments, one thread per state element -----
// Forward (reverse == 0): entry p becomes the state before segment p, from
// the seed: run_{p+1} = decay run_p + entry p (the last segment's entry is
// never read).  Reverse: entry p becomes the reverse state after segment p,
// run_{p-1} = entry p + decay run_p.  decay = gamma^(segment length) with a
// decay (every segment that contributes is full), else 1.
__global__ void bwd_scan_kernel(float *__restrict__ states, int P, int E, int blocks_per_head,
                                const float *__restrict__ seed, int reverse,
                                const float *__restrict__ gamma, int H, int seg_len)
{
    const int h = blockIdx.x / blocks_per_head;
    const int e = (blockIdx.x % blocks_per_head) * blockDim.x + threadIdx.x;
    if (e >= E) return;
    const float f = gamma ? powf(gamma[h % H], (float)seg_len) : 1.f;
    float *col = states + (size_t)h * P * E + e;
    float run = 0.f;
    if (!reverse) {
        if (seed) run = seed[(size_t)h * E + e];
        for (int p = 0; p < P; ++p) {
            const float x = p < P - 1 ? col[(size_t)p * E] : 0.f;
            col[(size_t)p * E] = run;
            run = fmaf(f, run, x);
        }
    } else {
        for (int p = P - 1; p >= 0; --p) {
            const float x = col[(size_t)p * E];
            col[(size_t)p * E] = run;
            run = fmaf(f, run, x);
        }
    }
}

// ---- 3. dq, 1/D_t, e_t, and the segment's sums of phi(q) g^T, phi(q) e ----
template <int D, int DV>
struct DqSmem {
    static constexpr size_t floats = 4 * (size_t)kBC * D + 3 * (size_t)kBC * DV + DV + 11 * kBC + 8;
    static constexpr size_t bytes = floats * sizeof(float);
};

// SEG: the sequence is split (P > 1), so the segment's sums of phi(q) g^T
// and phi(q) e are needed by the reverse scan; with one segment the reverse
// pass starts from zero and they are skipped.  DECAY: the recurrence carries
// a per-head decay; the segment sums are then weighted by gamma^(token -
// segment start), as the reverse state they feed decays towards earlier tokens.
template <int D, int DV, typename T, bool SEG, bool DECAY>
__global__ void __launch_bounds__(Cfg<D, DV>::kNT, 1)
bwd_dq_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
              const float *__restrict__ dy, float *__restrict__ dq, int N, int P, int seg_chunks,
              float eps, const float *__restrict__ prefix, float *__restrict__ rev_local,
              float *__restrict__ dinv_out, float *__restrict__ e_out,
              const float *__restrict__ gamma, int H)
{
    using C = Cfg<D, DV>;
    constexpr int NT = C::kNT, NW = NT / 32;
    using RT = WarpRows<NT, D, DV>;
    static_assert(NT >= D + DV, "one thread per feature and per value column");
    extern __shared__ float4 smem4[];
    float *sFq = reinterpret_cast<float *>(smem4);  // [kBC][D] phi(q)
    float *sPk = sFq + kBC * D;                     // [kBC][D] psi(k)
    float *sZt = sPk + kBC * D;                     // [kBC][D] zeta_t
    float *sH = sZt + kBC * D;                      // [kBC][D] hR_t = R_t g_t
    float *sV = sH + kBC * D;                       // [kBC][DV]
    float *sG = sV + kBC * DV;                      // [kBC][DV] dy_t, then g_t
    float *sUt = sG + kBC * DV;                     // [kBC][DV] u_t
    float *sUrun = sUt + kBC * DV;                  // [DV] u before the chunk
    float *sDinv = sUrun + DV;                      // [kBC] 1 / D_t
    float *sAct = sDinv + kBC;                      // [kBC] 1 where den_t >= eps
    float *sSq = sAct + kBC;                        // [kBC] sum of phi(q_t)
    float *sFz = sSq + kBC;                         // [kBC] phi(q_t) . zeta_t
    float *sUg = sFz + kBC;                         // [kBC] u_t . g_t
    float *sNt = sUg + kBC;                         // [kBC] n_t
    float *sE = sNt + kBC;                          // [kBC] e_t
    float *sC = sE + kBC;                           // [kBC] c_t
    float *sPw = sC + kBC;                          // [kBC] gamma^(token - segment start)
    float *sGp = sPw + kBC;                         // [kBC + 1] gamma^m
    float *sGip = sGp + kBC + 4;                    // [kBC + 1] gamma^-m
    const Seg sg = segment(P, seg_chunks, N);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = warp * RT::RPW, c0 = lane * RT::CPL;
    const int my_row = r0 + RT::row_of(lane);
    const bool writer = RT::writer(lane);

    // R and Sh as packed pairs of rows: Rp[i][c] = (R[2i][c], R[2i+1][c])
    constexpr int RP = RT::RPW / 2;
    uint64_t Rp[RP][RT::CPL], Shp[RP][RT::CPL];
    const float *pre = prefix + ((size_t)sg.h * P + sg.p) * C::kE;
#pragma unroll
    for (int i = 0; i < RP; ++i) {
        float ra[RT::CPL], rb[RT::CPL];
        ldn(pre + (r0 + 2 * i) * DV + c0, ra);
        ldn(pre + (r0 + 2 * i + 1) * DV + c0, rb);
#pragma unroll
        for (int c = 0; c < RT::CPL; ++c) {
            Rp[i][c] = pk2(ra[c], rb[c]);
            Shp[i][c] = pk2(0.f, 0.f);
        }
    }
    float zeta_run = tid < D ? pre[C::kOffZ + tid] : 0.f;   // thread a < D: zeta[a]
    if (tid >= D && tid < D + DV) sUrun[tid - D] = pre[C::kOffU + tid - D];
    NAcc<DECAY> n_acc = pre[C::kOffN];   // advanced by thread NT - 1
    NAcc<DECAY> pw_acc = 1;              // gamma^(token - segment start), thread NT - 1
    float zh = 0.f;
    const float gm = DECAY ? gamma[sg.h % H] : 1.f;
    // For gamma >= 1/4 the decay costs no multiply per state element: within
    // a chunk R_t = gamma^(i+1) Rt_i with Rt_i = R_prev + sum_{j<=i}
    // gamma^-(j+1) psi(k_j) v_j^T (i, j counted in the chunk, so
    // gamma^-(j+1) <= 2^64), R g scaled by gamma^(i+1), R rescaled per chunk.
    const bool scaled = DECAY && gm >= 0.25f;
    if (scaled && tid == 0) {
        float p = 1.f, ip = 1.f;
        for (int m = 0; m <= kBC; ++m) {
            sGp[m] = p;
            sGip[m] = ip;
            p *= gm;
            ip /= gm;
        }
    }

    ChunkLoad<D, T, NT> lq, lk;
    ChunkLoad<DV, T, NT> lv;
    ChunkLoad<DV, float, NT> ldy;
    {
        const size_t row0 = (size_t)sg.h * N + sg.t0;
        const int L = min(kBC, sg.t1 - sg.t0);
        lq.load(q + row0 * D, L); lk.load(k + row0 * D, L);
        lv.load(v + row0 * DV, L); ldy.load(dy + row0 * DV, L);
    }
    for (int t0 = sg.t0; t0 < sg.t1; t0 += kBC) {
        const int L = min(kBC, sg.t1 - t0);
        const size_t row0 = (size_t)sg.h * N + t0;
        __syncthreads();   // the previous chunk is consumed
        lq.store(sFq, L, Phi());
        lk.store(sPk, L, Psi());
        lv.store(sV, L, Ident());
        ldy.store(sG, L, Ident());
        __syncthreads();
        if (t0 + kBC < sg.t1) {   // the next chunk flies in while this one is processed
            const size_t nrow = row0 + kBC;
            const int nL = min(kBC, sg.t1 - t0 - kBC);
            lq.load(q + nrow * D, nL); lk.load(k + nrow * D, nL);
            lv.load(v + nrow * DV, nL); ldy.load(dy + nrow * DV, nL);
        }
        // zeta_t, u_t and n_t for every token of the chunk (all include token t)
        if (tid < D) {
            float run = zeta_run;
            for (int t = 0; t < L; ++t) {
                run = DECAY ? fmaf(gm, run, sPk[t * D + tid]) : run + sPk[t * D + tid];
                sZt[t * D + tid] = run;
            }
            zeta_run = run;
        } else if (tid < D + DV) {
            const int b = tid - D;
            float run = sUrun[b];
            for (int t = 0; t < L; ++t) {
                run = DECAY ? fmaf(gm, run, sV[t * DV + b]) : run + sV[t * DV + b];
                sUt[t * DV + b] = run;
            }
            sUrun[b] = run;
        } else if (tid == NT - 1) {
            // the (decayed) token count; with a decay in fp64: near its
            // steady state 1/(1 - gamma) every fp32 rounding of gamma n + 1
            // leans the same way, a bias of up to 2^-24 / (1 - gamma) that dq
            // would inherit (zeta's increments are small, its bias is not)
            for (int t = 0; t < L; ++t) {
                n_acc = DECAY ? fma((NAcc<DECAY>)gm, n_acc, NAcc<DECAY>(1)) : n_acc + 1;
                sNt[t] = (float)n_acc;
                sPw[t] = (float)pw_acc;
                pw_acc *= gm;
            }
        }
        __syncthreads();
        // per token: den_t = n_t sum(phi(q_t)) + phi(q_t).zeta_t, u_t.dy_t; one warp per token
        for (int t = warp; t < L; t += NW) {
            float sq = 0.f, fz = 0.f, ug = 0.f;
            for (int x = lane; x < D; x += 32) {
                const float f = sFq[t * D + x];
                sq += f;
                fz = fmaf(f, sZt[t * D + x], fz);
            }
            for (int b = lane; b < DV; b += 32) ug = fmaf(sUt[t * DV + b], sG[t * DV + b], ug);
            sq = warp_sum(sq);
            fz = warp_sum(fz);
            ug = warp_sum(ug);
            if (lane == 0) {
                const float den = fmaf(sNt[t], sq, fz);
                const float dinv = 1.f / fmaxf(den, eps);
                sDinv[t] = dinv;
                sAct[t] = den >= eps ? 1.f : 0.f;
                sSq[t] = sq;
                sFz[t] = fz;
                sUg[t] = ug * dinv;
            }
        }
        __syncthreads();
        for (int e = tid; e < L * DV; e += NT) sG[e] *= sDinv[e / DV];
        __syncthreads();
        // the recurrence: R_t = R_{t-1} + psi(k_t) v_t^T, hR_t = R_t g_t;
        // and the segment's sum of phi(q_t) g_t^T.  Each FMA updates a pair of
        // rows (packed), with the same operations per element as the scalar form.
        const uint64_t gm2 = pk2(gm, gm);
        auto token_loop = [&](auto scaled_tag) {
            constexpr bool SC = decltype(scaled_tag)::value;
            // two tokens per iteration overlap one token's reduce-scatter with the
            // next token's FMAs (not with the segment sums: too many registers)
#pragma unroll (SEG ? 1 : 2)
            for (int t = 0; t < L; ++t) {
                float pk[RT::RPW], fq[RT::RPW], x[RT::CPL], g[RT::CPL], acc[RT::RPW];
                ldn(sPk + t * D + r0, pk);      // warp-uniform
                ldn(sFq + t * D + r0, fq);      // warp-uniform
                ldn(sV + t * DV + c0, x);
                ldn(sG + t * DV + c0, g);
                if constexpr (SC) {
                    const float ip = sGip[t + 1];
#pragma unroll
                    for (int r = 0; r < RT::RPW; ++r) pk[r] *= ip;
                }
                if constexpr (SEG && DECAY) {
                    const float w = sPw[t];
#pragma unroll
                    for (int r = 0; r < RT::RPW; ++r) fq[r] *= w;
                }
                uint64_t xb[RT::CPL], gb[RT::CPL];   // each column value in both lanes
#pragma unroll
                for (int c = 0; c < RT::CPL; ++c) {
                    xb[c] = pk2(x[c], x[c]);
                    gb[c] = pk2(g[c], g[c]);
                }
#pragma unroll
                for (int i = 0; i < RP; ++i) {
                    const uint64_t pkp = pk2(pk[2 * i], pk[2 * i + 1]);
                    uint64_t accp = pk2(0.f, 0.f);
#pragma unroll
                    for (int c = 0; c < RT::CPL; ++c) {
                        Rp[i][c] = fma2(pkp, xb[c], (DECAY && !SC) ? mul2(gm2, Rp[i][c]) : Rp[i][c]);
                        accp = fma2(Rp[i][c], gb[c], accp);
                        if constexpr (SEG) Shp[i][c] = fma2(pk2(fq[2 * i], fq[2 * i + 1]), gb[c], Shp[i][c]);
                    }
                    unpk2(accp, acc[2 * i], acc[2 * i + 1]);
                }
                float hsum = reduce_scatter<RT::RPW>(acc, lane);
                if constexpr (SC) hsum *= sGp[t + 1];
                if (writer) sH[t * D + my_row] = hsum;
            }
            if constexpr (SC) {
                const uint64_t pL = pk2(sGp[L], sGp[L]);
#pragma unroll
                for (int i = 0; i < RP; ++i)
#pragma unroll
                    for (int c = 0; c < RT::CPL; ++c) Rp[i][c] = mul2(Rp[i][c], pL);
            }
        };
        if (scaled) token_loop(std::true_type{});
        else token_loop(std::false_type{});
        __syncthreads();
        // e_t and c_t (see the header: the leading terms cancel algebraically)
        for (int t = warp; t < L; t += NW) {
            float fh = 0.f;
            for (int x = lane; x < D; x += 32) fh = fmaf(sFq[t * D + x], sH[t * D + x], fh);
            fh = warp_sum(fh);
            if (lane == 0) {
                float e = 0.f, c = sUg[t];
                if (sAct[t] != 0.f) {
                    e = -fmaf(sSq[t], sUg[t], fh) * sDinv[t];
                    c = fmaf(sUg[t], sFz[t], -sNt[t] * fh) * sDinv[t];
                }
                sE[t] = e;
                sC[t] = c;
            }
        }
        __syncthreads();
        // dq_t = (c_t + hR_t + zeta_t e_t) * phi'(q_t)
        for (int e = tid; e < L * D; e += NT) {
            const int t = e / D;
            dq[row0 * D + e] = (sC[t] + fmaf(sZt[e], sE[t], sH[e])) * fminf(sFq[e], 1.f);
        }
        if (tid < L) {
            dinv_out[row0 + tid] = sDinv[tid];
            e_out[row0 + tid] = sE[tid];
        }
        if (SEG && tid < D)
            for (int t = 0; t < L; ++t)
                zh = fmaf(DECAY ? sFq[t * D + tid] * sPw[t] : sFq[t * D + tid], sE[t], zh);
    }
    if constexpr (SEG) {
        float *out = rev_local + ((size_t)sg.h * P + sg.p) * C::kE;
#pragma unroll
        for (int i = 0; i < RP; ++i)
#pragma unroll
            for (int c = 0; c < RT::CPL; ++c)
                unpk2(Shp[i][c], out[(r0 + 2 * i) * DV + c0 + c], out[(r0 + 2 * i + 1) * DV + c0 + c]);
        if (tid < D) out[C::kOffZ + tid] = zh;
        for (int e = tid; e < DV + 4; e += NT) out[C::kOffU + e] = 0.f;   // unused slots
    }
}

// ---- 5. dk, dv (and dL/dS_in, dL/dz_in from segment 0) --------------------
template <int D, int DV>
struct DkdvSmem {
    static constexpr int kGrp = 8;   // tokens whose dv partial sums are reduced together
    static constexpr size_t floats = 3 * (size_t)kBC * D + 3 * (size_t)kBC * DV + 4 * kBC + 8 +
                                     (size_t)kGrp * (Cfg<D, DV>::kNT / 32) * DV;
    static constexpr size_t bytes = floats * sizeof(float);
};

// DECAY: Sh_t = phi(q_t) g_t^T + gamma Sh_{t+1} (zh alike), and the state
// gradient gains the factor gamma of the first token's update.
template <int D, int DV, typename T, bool DECAY>
__global__ void __launch_bounds__(Cfg<D, DV>::kNT, 1)
bwd_dkdv_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                const float *__restrict__ dy, float *__restrict__ dk, float *__restrict__ dvg,
                int N, int P, int seg_chunks, const float *__restrict__ suffix,
                const float *__restrict__ dinv, const float *__restrict__ e_in,
                float *__restrict__ grad_S, float *__restrict__ grad_z,
                const float *__restrict__ gamma, int H)
{
    using C = Cfg<D, DV>;
    constexpr int NT = C::kNT;
    constexpr int NW = NT / 32, kGrp = DkdvSmem<D, DV>::kGrp;
    using RT = WarpRows<NT, D, DV>;   // Sh: a band of rows per warp, a few columns per lane
    extern __shared__ float4 smem4[];
    float *sFq = reinterpret_cast<float *>(smem4);  // [kBC][D]
    float *sFk = sFq + kBC * D;                     // [kBC][D]
    float *sDK = sFk + kBC * D;                     // [kBC][D] zh_t, then dk_t
    float *sV = sDK + kBC * D;                      // [kBC][DV]
    float *sG = sV + kBC * DV;                      // [kBC][DV] dy_t, then g_t
    float *sDV = sG + kBC * DV;                     // [kBC][DV]
    float *sE = sDV + kBC * DV;                     // [kBC]
    float *sDinv = sE + kBC;                        // [kBC]
    float *sGp = sDinv + kBC;                       // [kBC + 1] gamma^m (kBC + 4 keeps sPart 16-byte aligned)
    float *sGip = sGp + kBC + 4;                    // [kBC + 1] gamma^-m
    float *sPart = sGip + kBC + 4;                  // [kGrp][NW][DV] per-warp partial dv
    const Seg sg = segment(P, seg_chunks, N);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = warp * RT::RPW, c0 = lane * RT::CPL;
    const int my_row = r0 + RT::row_of(lane);
    const bool wr1 = RT::writer(lane);

    // Sh as packed pairs of rows: S1p[i][c] = (Sh[2i][c], Sh[2i+1][c])
    constexpr int RP = RT::RPW / 2;
    uint64_t S1p[RP][RT::CPL];
    const float *suf = suffix + ((size_t)sg.h * P + sg.p) * C::kE;
#pragma unroll
    for (int i = 0; i < RP; ++i) {
        float ra[RT::CPL], rb[RT::CPL];
        ldn(suf + (r0 + 2 * i) * DV + c0, ra);
        ldn(suf + (r0 + 2 * i + 1) * DV + c0, rb);
#pragma unroll
        for (int c = 0; c < RT::CPL; ++c) S1p[i][c] = pk2(ra[c], rb[c]);
    }
    float zh = tid < D ? suf[C::kOffZ + tid] : 0.f;   // thread a < D carries zh[a]
    const float gm = DECAY ? gamma[sg.h % H] : 1.f;
    // gamma >= 1/4: Sh carried rescaled within a chunk, as in bwd_dq_kernel
    // (counted from the chunk's last token backwards)
    const bool scaled = DECAY && gm >= 0.25f;
    if (scaled && tid == 0) {
        float p = 1.f, ip = 1.f;
        for (int m = 0; m <= kBC; ++m) {
            sGp[m] = p;
            sGip[m] = ip;
            p *= gm;
            ip /= gm;
        }
    }

    ChunkLoad<D, T, NT> lq, lk;
    ChunkLoad<DV, T, NT> lv;
    ChunkLoad<DV, float, NT> ldy;
    float pdinv = 0.f, pe = 0.f;
    const int nch = (sg.t1 - sg.t0 + kBC - 1) / kBC;
    auto issue = [&](int c) {
        const int t0 = sg.t0 + c * kBC, L = min(kBC, sg.t1 - t0);
        const size_t row0 = (size_t)sg.h * N + t0;
        lq.load(q + row0 * D, L); lk.load(k + row0 * D, L);
        lv.load(v + row0 * DV, L); ldy.load(dy + row0 * DV, L);
        pdinv = tid < L ? __ldg(dinv + row0 + tid) : 0.f;
        pe = tid < L ? __ldg(e_in + row0 + tid) : 0.f;
    };
    issue(nch - 1);
    for (int c = nch - 1; c >= 0; --c) {
        const int t0 = sg.t0 + c * kBC, L = min(kBC, sg.t1 - t0);
        const size_t row0 = (size_t)sg.h * N + t0;
        __syncthreads();   // the previous chunk's outputs are written
        lq.store(sFq, L, Phi());
        lk.store(sFk, L, Phi());
        lv.store(sV, L, Ident());
        ldy.store(sG, L, Ident());
        if (tid < kBC) {
            sE[tid] = pe;
            sDinv[tid] = pdinv;
        }
        __syncthreads();
        if (c > 0) issue(c - 1);
        for (int e = tid; e < kBC * DV; e += NT) sG[e] *= sDinv[e / DV];
        // zh_t = zh_{t+1} + phi(q_t) e_t for every token of the chunk, last first
        if (tid < D)
            for (int t = L - 1; t >= 0; --t) {
                zh = DECAY ? fmaf(gm, zh, sFq[t * D + tid] * sE[t]) : fmaf(sFq[t * D + tid], sE[t], zh);
                sDK[t * D + tid] = zh;
            }
        __syncthreads();
        const uint64_t gm2 = pk2(gm, gm);
        auto token_loop = [&](auto scaled_tag) {
            constexpr bool SC = decltype(scaled_tag)::value;
            int slot = 0;
            // two tokens per iteration overlap one token's reduce-scatter with the
            // next token's FMAs
#pragma unroll 2
            for (int t = L - 1; t >= 0; --t) {
                // Sh_t = Sh_{t+1} + phi(q_t) g_t^T; dk_t from Sh_t v_t (a reduction
                // over columns, inside the warp); dv_t = Sh_t^T phi(k_t) from per-warp
                // partial sums over the warp's rows, added across warps every kGrp tokens
                float fq[RT::RPW], fk[RT::RPW], g[RT::CPL], x[RT::CPL], acc[RT::RPW], pv[RT::CPL];
                ldn(sFq + t * D + r0, fq);       // warp-uniform
                ldn(sFk + t * D + r0, fk);       // warp-uniform
                ldn(sG + t * DV + c0, g);
                ldn(sV + t * DV + c0, x);
                const int m = L - t;             // tokens of the chunk processed, this one included
                if constexpr (SC) {
                    const float ip = sGip[m];
#pragma unroll
                    for (int r = 0; r < RT::RPW; ++r) fq[r] *= ip;
                }
                // each FMA updates a pair of rows (packed); pv keeps the even and
                // odd rows' partial sums in its two lanes until the end
                uint64_t gb[RT::CPL], xb[RT::CPL], pvp[RT::CPL];
#pragma unroll
                for (int cc = 0; cc < RT::CPL; ++cc) {
                    gb[cc] = pk2(g[cc], g[cc]);
                    xb[cc] = pk2(x[cc], x[cc]);
                    pvp[cc] = pk2(0.f, 0.f);
                }
#pragma unroll
                for (int i = 0; i < RP; ++i) {
                    const uint64_t fqp = pk2(fq[2 * i], fq[2 * i + 1]);
                    const uint64_t fkp = pk2(fk[2 * i], fk[2 * i + 1]);
                    uint64_t accp = pk2(0.f, 0.f);
#pragma unroll
                    for (int cc = 0; cc < RT::CPL; ++cc) {
                        S1p[i][cc] = fma2(fqp, gb[cc], (DECAY && !SC) ? mul2(gm2, S1p[i][cc]) : S1p[i][cc]);
                        accp = fma2(S1p[i][cc], xb[cc], accp);
                        pvp[cc] = fma2(S1p[i][cc], fkp, pvp[cc]);
                    }
                    unpk2(accp, acc[2 * i], acc[2 * i + 1]);
                }
#pragma unroll
                for (int cc = 0; cc < RT::CPL; ++cc) {
                    float a0, a1;
                    unpk2(pvp[cc], a0, a1);
                    pv[cc] = a0 + a1;
                }
                float dfk = reduce_scatter<RT::RPW>(acc, lane);
                if constexpr (SC) {
                    const float p = sGp[m];
                    dfk *= p;
#pragma unroll
                    for (int cc = 0; cc < RT::CPL; ++cc) pv[cc] *= p;
                }
                if (wr1)   // dk_t = (Sh_t v_t + zh_t) * phi'(k_t)
                    sDK[t * D + my_row] = (dfk + sDK[t * D + my_row]) * fminf(sFk[t * D + my_row], 1.f);
                stn(sPart + (slot * NW + warp) * DV + c0, pv);
                if (++slot == kGrp || t == 0) {   // uniform across the CTA
                    __syncthreads();
                    // slot s holds token t + slot - 1 - s
                    for (int e = tid; e < slot * DV; e += NT) {
                        const int s = e / DV, b = e % DV;
                        float sum = 0.f;
#pragma unroll
                        for (int w = 0; w < NW; ++w) sum += sPart[(s * NW + w) * DV + b];
                        sDV[(t + slot - 1 - s) * DV + b] = sum;
                    }
                    __syncthreads();
                    slot = 0;
                }
            }
            if constexpr (SC) {
                const uint64_t pL = pk2(sGp[L], sGp[L]);
#pragma unroll
                for (int i = 0; i < RP; ++i)
#pragma unroll
                    for (int cc = 0; cc < RT::CPL; ++cc) S1p[i][cc] = mul2(S1p[i][cc], pL);
            }
        };
        if (scaled) token_loop(std::true_type{});
        else token_loop(std::false_type{});
        __syncthreads();
        for (int e = tid * 4; e < L * D; e += NT * 4) st4(dk + row0 * D + e, ld4(sDK + e));
        for (int e = tid * 4; e < L * DV; e += NT * 4) st4(dvg + row0 * DV + e, ld4(sDV + e));
    }
    if (sg.p == 0 && grad_S) {
        float *gS = grad_S + (size_t)sg.h * D * DV;
#pragma unroll
        for (int i = 0; i < RP; ++i)
#pragma unroll
            for (int cc = 0; cc < RT::CPL; ++cc) {
                float a0, a1;
                unpk2(S1p[i][cc], a0, a1);
                gS[(r0 + 2 * i) * DV + c0 + cc] = gm * a0;
                gS[(r0 + 2 * i + 1) * DV + c0 + cc] = gm * a1;
            }
        if (tid < D) grad_z[(size_t)sg.h * D + tid] = gm * zh;
    }
}

// ---- host side --------------------------------------------------------------
struct BwdPlan {
    int P = 1, seg_chunks = 1, E = 0;
    size_t seed_off = 0, fwd_off = 0, rev_off = 0, dinv_off = 0, e_off = 0, total = 0;
};

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return 148;
    return n;
}

// Segments per head: minimise (waves of one CTA per SM) x (chunks per
// segment), where a split sequence costs about 1.4 times as much per chunk
// (the segment sums of the kv pass and of the dq pass: 7 instead of 5 FMAs
// per state element and token) plus two chunks of fixed cost for the scans.
BwdPlan make_plan(int BH, int N, int d, int dv) {
    BwdPlan pl;
    const int nchunks = std::max(1, (N + kBC - 1) / kBC);
    const long slots = sm_count();
    long best = -1;
    for (int P = 1; P <= std::min(nchunks, 64); ++P) {
        const int sc = (nchunks + P - 1) / P;
        if ((nchunks + sc - 1) / sc != P) continue;   // no empty segments
        const long waves = ((long)BH * P + slots - 1) / slots;
        const long cost = waves * (P > 1 ? 7L * sc + 10 : 5L * sc);
        if (best < 0 || cost < best) { best = cost; pl.P = P; pl.seg_chunks = sc; }
    }
    pl.E = d * dv + d + dv + 4;
    const size_t st = up256((size_t)BH * pl.P * pl.E * sizeof(float));
    pl.seed_off = sizeof(WsHeader);
    pl.fwd_off = pl.seed_off + up256((size_t)BH * pl.E * sizeof(float));
    pl.rev_off = pl.fwd_off + st;
    pl.dinv_off = pl.rev_off + st;
    pl.e_off = pl.dinv_off + up256((size_t)BH * N * sizeof(float));
    pl.total = pl.e_off + up256((size_t)BH * N * sizeof(float));
    return pl;
}

template <int D, int DV, typename T, bool DECAY>
cudaError_t launch_typed(const BwdArgs &a, const BwdPlan &pl) {
    using C = Cfg<D, DV>;
    const int BH = a.B * a.H;
    char *ws = static_cast<char *>(a.ws);
    float *seed = reinterpret_cast<float *>(ws + pl.seed_off);
    float *fwd = reinterpret_cast<float *>(ws + pl.fwd_off);
    float *rev = reinterpret_cast<float *>(ws + pl.rev_off);
    float *dinv = reinterpret_cast<float *>(ws + pl.dinv_off);
    float *ev = reinterpret_cast<float *>(ws + pl.e_off);
    const T *q = static_cast<const T *>(a.q), *k = static_cast<const T *>(a.k),
            *v = static_cast<const T *>(a.v);
    const int grid = BH * pl.P, bph = (pl.E + 255) / 256;
    constexpr size_t kv_smem = sizeof(float) * kBC * (D + DV);
    constexpr size_t dq_smem = DqSmem<D, DV>::bytes, dkdv_smem = DkdvSmem<D, DV>::bytes;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(bwd_dq_kernel<D, DV, T, true, DECAY>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dq_smem)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_dq_kernel<D, DV, T, false, DECAY>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dq_smem)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(bwd_dkdv_kernel<D, DV, T, DECAY>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dkdv_smem)) != cudaSuccess)
        return e;
    if (a.S_in) {
        bwd_seed_kernel<D, DV><<<BH, 128, 0, a.stream>>>(a.S_in, a.z_in, seed);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (pl.P > 1) {
        bwd_kv_states_kernel<D, DV, T, DECAY><<<grid, C::kNT, kv_smem, a.stream>>>(
            k, v, a.N, pl.P, pl.seg_chunks, fwd, a.gamma, a.H);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const int seg_len = pl.seg_chunks * kBC;
    bwd_scan_kernel<<<BH * bph, 256, 0, a.stream>>>(fwd, pl.P, pl.E, bph, a.S_in ? seed : nullptr, 0,
                                                    a.gamma, a.H, seg_len);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (pl.P > 1) {
        bwd_dq_kernel<D, DV, T, true, DECAY><<<grid, C::kNT, dq_smem, a.stream>>>(
            q, k, v, a.dy, a.dq, a.N, pl.P, pl.seg_chunks, a.eps, fwd, rev, dinv, ev, a.gamma, a.H);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        bwd_scan_kernel<<<BH * bph, 256, 0, a.stream>>>(rev, pl.P, pl.E, bph, nullptr, 1, a.gamma,
                                                        a.H, seg_len);
    } else {   // one segment: the reverse pass starts from the zero state
        bwd_dq_kernel<D, DV, T, false, DECAY><<<grid, C::kNT, dq_smem, a.stream>>>(
            q, k, v, a.dy, a.dq, a.N, pl.P, pl.seg_chunks, a.eps, fwd, rev, dinv, ev, a.gamma, a.H);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = cudaMemsetAsync(rev, 0, (size_t)BH * pl.E * sizeof(float), a.stream)) != cudaSuccess)
            return e;
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_dkdv_kernel<D, DV, T, DECAY><<<grid, C::kNT, dkdv_smem, a.stream>>>(
        q, k, v, a.dy, a.dk, a.dv_grad, a.N, pl.P, pl.seg_chunks, rev, dinv, ev, a.grad_S_in,
        a.grad_z_in, a.gamma, a.H);
    return cudaGetLastError();
}

template <int D, int DV>
cudaError_t launch_dims(const BwdArgs &a, const BwdPlan &pl) {
    if (a.gamma)
        return a.dt == LA_DTYPE_BF16 ? launch_typed<D, DV, __nv_bfloat16, true>(a, pl)
                                     : launch_typed<D, DV, float, true>(a, pl);
    return a.dt == LA_DTYPE_BF16 ? launch_typed<D, DV, __nv_bfloat16, false>(a, pl)
                                 : launch_typed<D, DV, float, false>(a, pl);
}

template <int D>
cudaError_t launch_dv(const BwdArgs &a, const BwdPlan &pl) {
    switch (a.dv) {
    case 32: return launch_dims<D, 32>(a, pl);
    case 64: return launch_dims<D, 64>(a, pl);
    default: return launch_dims<D, 128>(a, pl);
    }
}

}  // namespace

size_t causal_backward_workspace(int BH, int N, int d, int dv) {
    return make_plan(BH, N, d, dv).total;
}

cudaError_t launch_causal_backward(const BwdArgs &a) {
    const BwdPlan pl = make_plan(a.B * a.H, a.N, a.d, a.dv);
    if (a.ws_bytes < pl.total) return cudaErrorInvalidValue;
    switch (a.d) {
    case 32: return launch_dv<32>(a, pl);
    case 64: return launch_dv<64>(a, pl);
    default: return launch_dv<128>(a, pl);
    }
}

}  // namespace la
