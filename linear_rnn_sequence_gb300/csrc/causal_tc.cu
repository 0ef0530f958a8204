// causal_tc.cu -- chunkwise causal elu(x)+1 linear attention on the sm_103a
// tensor cores (tcgen05 MMA, TMEM accumulators, TMA tiles, mbarriers).
//
// Method ("Linear Attention/es", "Entrenamiento: forma paralela"): split the
// sequence into blocks of C = 128 tokens.  For query i of block c
//   num_i = sum_{j <= i in c} w_ij v_j + phi(q_i)^T S_prev
//   den_i = sum_{j <= i in c} w_ij     + phi(q_i)^T z_prev,   w_ij = phi(q_i)^T phi(k_j)
//   y_i   = num_i / max(den_i, eps)
// then S_prev += sum_{j in c} phi(k_j) v_j^T and z_prev += sum_{j in c} phi(k_j)
// (the state recursion of "Forma recurrente e inferencia autorregresiva").
//
// Precision scheme.  Every feature is split per token as phi(x) = c + psi_c(x),
// psi_c = phi - c, with c = 1 for inputs of order one or below (psi_1 = elu)
// and c near the token's typical phi when its features are mostly strongly
// negative (split_const in tc_common.cuh).  For inputs of order 1/sqrt(d)
// every phi is close to 1, so w_ij ~ d with small variations and the output
// is a near-uniform average; bf16 operands holding phi itself lose those
// variations.  The kernel therefore feeds only the residuals (small values)
// to the tensor cores and carries the constants exactly:
//   w_ij            = d c_i c'_j + c_i beta_j + c'_j alpha_i + a_i . b_j
//                       (a = bf16 psi_c(q), b = bf16 psi_c'(k); alpha_i and beta_j
//                        the sums of the residuals before rounding, which moves
//                        w by about 1e-5 of itself, a constant per row or per key;
//                        c_i of the query, c'_j of the key)
//   S               = 1 u^T + R,  u = sum_j c'_j v_j,  R = sum_j b_j v_j^T
//   z               = n 1 + zeta, n = sum_j c'_j,   zeta = sum_j b_j
//   phi(q_i)^T S    = (d c_i + alpha_i) u + c_i r + a_i R,        r = sum_j beta_j v_j = colsum(R)
//   phi(q_i)^T z    = (d c_i + alpha_i) n + c_i rho + a_i . zeta, rho = sum_j beta_j
// The constant parts enter the MMAs through one extra K = 16 slice of the
// residual q operand (carrying c, alpha and d c as bf16 hi/lo pairs) against
// small tiles holding beta, c', u, r, n and rho, so the tensor core returns
// the full weight w, numerator and inter-block denominator.  The intra-block weights
// w_ij (about d) are split into bf16 hi + lo parts for the P.V product, so
// their rounding error is about 2^-17 of w.  All accumulation is fp32 (TMEM).
// The result is the exact attention of the features c + bf16(psi_c(x)); the
// outputs are float32.
//
// Decay (DECAY = true; RetNet's S_t = gamma S_{t-1} + phi(k_t) v_t^T, z alike,
// "Linear Attention/es", "Variantes y extensiones").  For query i of a block
// of L tokens starting from state (S_b, z_b),
//   num_i = gamma^(i+1) [ phi(q_i)^T S_b + sum_{j <= i} gamma^-(j+1) w_ij v_j ]
// and den_i alike, so the common factor gamma^(i+1) cancels in y_i except in
// the clamp, which becomes max(den', eps gamma^-(i+1)).  Key j enters scaled
// by s_j = gamma^(L-1-j) <= 1 (psi(k_j) before its bf16 rounding, and the
// 1 and beta parts as bf16 hi/lo pairs), which is its weight in the state
// after the block.  The inter-block terms use S_b unscaled.  The carried
// state is decayed without touching TMEM on most blocks: TMEM holds it
// divided by a running scale G (DecayScale below) that shrinks by gamma^L per
// block, the keys enter multiplied by s_j / G, and the export multiplies by G.
// The weight tile then holds s_j w_ij / G, and the weight epilogue multiplies
// it by gamma^-L G to get gamma^-(j+1) w_ij.  Only when G would fall below
// 2^-48 is the state rescaled in TMEM.  All factors stay within 2^+-112 for gamma >= 2^-1/2; smaller
// decays are left to the CUDA-core kernel.  One work item per head (no
// sequence split).
//
// One CTA owns one (head, segment) work item and walks its blocks in order.
// Warp roles (18 warps):
//   warp 0       TMA producer: Q (1 stage), K and V (2 stages) tiles, 128B swizzle
//   warp 1       TMEM allocator and single-thread MMA issuer
//   warps 2..9   group A, two warps per TMEM lane quarter (the pair splits a
//                token row): psi(q) into TMEM, then the weight epilogue
//                (G -> w hi/lo in TMEM, row sums)
//   warps 10..17 group B, likewise: psi(k) in place in shared memory, the
//                state export (R -> bf16 operand, zeta, u, r, n, rho) and the
//                output epilogue (16x256b TMEM loads, 32-byte-sector stores)
// The two groups work on neighbouring blocks at once, so the psi passes, the
// weight epilogue, the tensor-core MMAs and the output epilogue overlap.
// TMEM columns: R [0,dv) | Y [128,128+dv) | G/P [256,384) | psi(q) and its
// augmentation [384,384+d/2+8) | a.zeta [464,480) | zeta [480,496) | u,r [496,512).
// Every wait is bounded in time; a wait that runs out records LA_ERR_TIMEOUT
// in the workspace header and the CTA unwinds (no trap, no hang).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstring>
#include <mutex>

#include "la_internal.h"
#include "tc_common.cuh"
#include "tc_state.cuh"

// Optional per-block timeline of CTA 0 (SM cycle counter) for performance
// work; compiled in only with -DLA_TRACE, and then read with la_trace_fetch.
#ifdef LA_TRACE
__device__ unsigned long long la_trace_buf[256 * 32];
#define LA_TRACE_POINT(c, ev)                                                   \
    do {                                                                        \
        if (blockIdx.x == 0 && (c) < 256) la_trace_buf[(c) * 32 + (ev)] = clock64(); \
    } while (0)
#else
#define LA_TRACE_POINT(c, ev) \
    do {                      \
    } while (0)
#endif

namespace la {
namespace {

using namespace tc;

constexpr int kThreads = 576;    // 18 warps: producer, MMA, group A (8), group B (8)
constexpr int kWarpA = 2;        // first warp of group A
constexpr int kWarpB = 10;       // first warp of group B
static_assert(kThreads == (kWarpB + 8) * 32 && kWarpB - kWarpA == 8,
              "eight warps per row-worker group, two per TMEM lane quarter");

constexpr uint32_t kColR = 0, kColY = 128, kColG = 256, kColAq = 384, kColYz = 464,
                   kColZ = 480, kColUV = 496;
constexpr uint32_t kTmemCols = 512;

// Augmentation step.  One extra K = 16 slice on the residual q operand
// carries per-row constants, so the MMAs add the exact parts of the split form:
//   A' row i  = [c, c, alpha_hi, alpha_lo, d c, alpha_hi, d c, 0...]  (TMEM, after psi_c(q))
//   B' key j  = [beta_hi, beta_lo, s_hi, s_hi, s_hi, s_lo, s_lo, 0...]   (s = c'_j, or its
//               decayed weight)    -> G  = d c_i s_j + c_i beta_j + s_j alpha_i + a_i.b_j
//   B'' col c = [r_hi, r_lo, u_hi, u_hi, u_hi, u_lo, u_lo, 0...]
//                                  -> Y  = (d c_i + alpha_i) u + c_i r + a_i R
//   Bz  col 0 = [rho_hi, rho_lo, n_hi, n_hi, n_hi, n_lo, n_lo, 0...]
//                                  -> Yz = (d c_i + alpha_i) n + c_i rho + a_i.zeta
// (x_hi = bf16(x), x_lo = bf16(x - x_hi): the pairs carry x to about 2^-17
// of its value; the dropped alpha_lo * u_lo term is smaller still).  Each
// B tile is [rows x 16] bf16, K-major without swizzle.
constexpr uint32_t kAugCols = 8;   // TMEM columns of the A' slice (16 bf16)
static_assert(kColAq + 64 + kAugCols <= kColYz, "psi(q) and its augmentation fit below Yz");

// Byte offset of (row n, k) in a [rows x 16] K-major no-swizzle bf16 tile.
__device__ __forceinline__ uint32_t k16_off(int n, int k) {
    return (uint32_t)((n >> 3) * 256 + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2);
}

constexpr int kSmallBytes = 6 * 1024;   // the Small area of every layout

template <int D, int DV, int DK = 0>
struct Layout {
    static constexpr int kQ = kC * D * 2;           // one Q stage
    static constexpr int kK = kC * D * 2;
    static constexpr int kV = kC * DV * 2;
    static constexpr bool kExtY = D == 64 && DV == 64;   // as kExt below
    // bf16 R operand, 128B-swizzled MN-major; ext: a zeta box follows (column 0
    // = zeta~), so [R~ | zeta box] is one N = dv + 64 operand
    static constexpr int kRt = D * DV * 2 + (kExtY ? D * 128 : 0);
    static constexpr int kUVB = 16 * kC * 2;        // [1|beta_hi|beta_lo] operand, [16 x C]
    static constexpr int kZt = 16 * D * 2;          // zeta operand, [16 x d]
    static constexpr int kGB = kC * 16 * 2;         // B' (G augmentation), [C x 16]
    // B'' (Y augmentation), [dv x 16]; ext: row dv is Bz's row (rows dv+1..dv+15 zero)
    static constexpr int kYB = (DV + (kExtY ? 16 : 0)) * 16 * 2;
    static constexpr int kZB = 16 * 16 * 2;         // Bz (Yz augmentation), [16 x 16]
    // d = dv = 64 ("ext"): each K stage is followed by an extension box whose
    // first columns hold the keys' weights and residual row sums, and each V
    // stage by a ones box, so one MMA per 16 tokens updates R, zeta, u and r
    // together (the accumulator is [R | zeta ...] over dv + 64 columns, with
    // rows 64..67 holding s_hi, s_lo, beta_hi, beta_lo times V).  The [1|beta]
    // operand area is then free and serves as scratch (ExtScratch).
    static constexpr bool kExt = D == 64 && DV == 64;
    static constexpr int kKs = kExt ? 2 * kK : kK;  // K stage stride
    static constexpr int kVs = kExt ? 2 * kV : kV;  // V stage stride
    static constexpr int oQ = 0;
    static constexpr int oK = oQ + kQ;              // 2 stages
    static constexpr int oV = oK + 2 * kKs;         // 2 stages
    static constexpr int oRt = oV + 2 * kVs;
    static constexpr int oUVB = oRt + kRt;          // 2 stages
    static constexpr int oZt = oUVB + 2 * kUVB;
    static constexpr int oGB = oZt + kZt;           // 2 stages
    static constexpr int oYB = oGB + 2 * kGB;
    static constexpr int oZB = oYB + kYB;
    static constexpr int oSmall = oZB + kZB;
    static constexpr int kSmall = kSmallBytes;
    static constexpr int oDecay = oSmall + kSmall;  // decay kernel only: DecaySmall
    static constexpr int kDecay = DK ? 2 * 1024 : 0;
    static constexpr int bytes = oDecay + kDecay;
    // request enough that only one CTA fits per SM (TMEM: 512 columns each)
    static constexpr int request = (bytes + 1024) > 120 * 1024 ? bytes + 1024 : 120 * 1024;
    static_assert(request <= 227 * 1024, "shared memory per CTA");
};

// Small shared-memory area.  Per-block values are kept by block parity:
// [c & 1] holds block c (or, for the state, the state after block c).
struct Small {
    alignas(16) float rowsum[2][2][kC];   // [block parity][half] partial sums_{j<=i} w_ij
    alignas(16) float u[2][128];
    alignas(16) float zeta[128];       // last exported zeta (fp32), for the final state
    alignas(16) float rho_part[2][4];
    alignas(16) float s_part[2][4];    // per-warp sums of the key weights s_j
    alignas(16) float e_inv[2][kC];    // output epilogue: 1 / max(den, eps) per row, per half
    alignas(16) float alpha_part[kC];  // psi(q) row sums of the second half
    alignas(16) float beta_part[kC];   // psi(k) row sums of the second half
    float n_s[2], rho_s[2];
    uint64_t q_full, q_empty, kv_full[2], kv_empty[2];
    uint64_t phik_done[2];             // by K/V stage: a waiter is never two phases behind
    uint64_t h_ready[2];               // by block parity: group A may run a block ahead of B
    uint64_t phiq_done, g_full, aq_free, st_full, rt_ready, y_full, y_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(offsetof(Small, u) % 16 == 0 && offsetof(Small, q_full) % 8 == 0,
              "vector loads and mbarriers need aligned fields");
static_assert(sizeof(Small) <= kSmallBytes, "small area");

// Shared values of the decay kernel only (after Small; the plain kernel's
// layout does not have them).
struct DecaySmall {
    alignas(16) float gpow[2][kC + 2]; // [0][m] = gamma^m, [1][m] = gamma^-m
};
static_assert(sizeof(DecaySmall) <= 2 * 1024, "decay area");
__device__ __forceinline__ DecaySmall &decay_area(Small &S) {
    return *reinterpret_cast<DecaySmall *>(reinterpret_cast<uint8_t *>(&S) + kSmallBytes);
}


// Scratch of the ext layout (d = dv = 64) in the otherwise unused [1|beta]
// operand area: rows 64..67 of the state accumulator over the dv columns, and
// the initial state's r.
struct ExtScratch {
    alignas(16) float uv[4][128];
    alignas(16) float r0[128];
};
static_assert(sizeof(ExtScratch) <= 2 * 16 * kC * 2, "ext scratch fits the operand area");

// The decay factors of a block, from a fixed decay (DK = 1: the per-head table
// of gamma powers in shared memory) or from per-token gates (DK = 2: the
// block's table of gate products in global memory).  For block c of L tokens:
//   pw(c, m)  = the decay over its first m tokens (gamma^m, or P_m)
//   ipw(c, m) = 1 / pw(c, m)
//   key_weight(c, L, j) = the decay after key j to the block's end, pw(c, L) / pw(c, j + 1)
template <int DK>
struct DecayPow {
    const float (*gpow)[kC + 2];   // DK = 1
    const float *tab;              // DK = 2: the table of the work item's first block
    __device__ __forceinline__ float pw(int c, int m) const {
        return DK == 2 ? __ldg(tab + (size_t)c * kGateTab + m) : gpow[0][m];
    }
    __device__ __forceinline__ float ipw(int c, int m) const {
        return DK == 2 ? __ldg(tab + (size_t)c * kGateTab + kGateInv + m) : gpow[1][m];
    }
    __device__ __forceinline__ float key_weight(int c, int L, int j) const {
        return DK == 2 ? pw(c, L) * ipw(c, j + 1) : gpow[0][L - 1 - j];
    }
    // what DecayScale starts from (any value but 1 gives the restart value 3/4)
    __device__ __forceinline__ float first() const {
        return DK == 1 ? gpow[0][1] : (DK == 2 ? 0.5f : 1.f);
    }
};

// Where each instantiation keeps the slow path of its bounded waits (the W of
// mbar_wait), per feature width and decay mode, as measured on the workloads:
// the d = 128 plain kernel inline, the others partly or wholly out of line.
template <int D, int DK>
struct WaitPolicy {
    static constexpr int value = D == 128 ? (DK == 0 ? 0 : (DK == 1 ? 2 : 1)) : (DK == 0 ? 2 : 1);
};

// ------------------------------------------------------------------ producer
template <int D, int DV, int W>
__device__ __forceinline__ void producer_role(Small &S, uint8_t *sQ, uint8_t *sK, uint8_t *sV,
                                              const CUtensorMap *qmap, const CUtensorMap *kmap,
                                              const CUtensorMap *vmap, int head, int tok0,
                                              int nchunks, bool drop_first, const Guard &g) {
    using Lay = Layout<D, DV>;
    constexpr uint32_t qbytes = kC * D * 2, kvbytes = kC * (D + DV) * 2;
    int last_q = -1, last_kv[2] = {-1, -1};
    for (int c = 0; c < nchunks; ++c) {
        const int t0 = tok0 + c * kC, s = c & 1;
        // block 0's copies read only q, k, v; every later wait may depend on
        // the initial state, which the previous kernel (if any) writes
        if (c == 1) griddep_wait();
        if (c >= 2 && !mbar_wait<W>(&S.kv_empty[s], ((c >> 1) - 1) & 1, g, 11)) break;
        mbar_arrive_expect_tx(&S.kv_full[s], kvbytes);
        if (!(drop_first && c == 0)) {   // test hook: a copy that never arrives
#pragma unroll
            for (int bx = 0; bx < D / 64; ++bx)
                tma_load_3d(sK + s * Lay::kKs + bx * kC * 128, kmap, &S.kv_full[s], bx * 64, t0, head);
#pragma unroll
            for (int bx = 0; bx < DV / 64; ++bx)
                tma_load_3d(sV + s * Lay::kVs + bx * kC * 128, vmap, &S.kv_full[s], bx * 64, t0, head);
            last_kv[s] = c;
        }
        LA_TRACE_POINT(c, 13);
        if (c > 0 && !mbar_wait<W>(&S.q_empty, (c - 1) & 1, g, 10)) break;
        mbar_arrive_expect_tx(&S.q_full, qbytes);
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx)
            tma_load_3d(sQ + bx * kC * 128, qmap, &S.q_full, bx * 64, t0, head);
        last_q = c;
        LA_TRACE_POINT(c, 14);
    }
    if (*g.abort) {  // let the copies already issued land before the CTA exits
        if (last_q >= 0) drain_wait(&S.q_full, last_q & 1, g.limit_ns);
        for (int s = 0; s < 2; ++s)
            if (last_kv[s] >= 0) drain_wait(&S.kv_full[s], (last_kv[s] >> 1) & 1, g.limit_ns);
    }
}

// ------------------------------------------------------------------ MMA issuer
// Per block c (one thread issues, in this order):
//   G  = psi(Q) psi(K)^T + A' B'^T = w         after psi(q), psi(k) of block c
//   R += psi(K)^T V, zeta += psi(K)^T 1,       after the previous state's export
//   [. r u] += V^T [1 beta_hi beta_lo s_hi s_lo]
//   Y  = psi(Q) R~ + A' B''^T,                 after the previous output epilogue
//   Yz = psi(Q) zeta~ + A' Bz^T
//   Y += P_hi V + P_lo V                       after the weight epilogue
// The export of the state after block c waits for both st_full and aq_free:
// the second says Y and Yz no longer read the operands it overwrites.
template <int D, int DV, int W>
__device__ __forceinline__ void mma_role(Small &S, uint32_t tb, uint8_t *sK, uint8_t *sV,
                                         uint8_t *sRt, uint8_t *sUVB, uint8_t *sZt, uint8_t *sGB,
                                         uint8_t *sYB, uint8_t *sZB, int nchunks,
                                         const Guard &g) {
    using Lay = Layout<D, DV>;
    constexpr uint32_t iG = idesc_bf16(128, kC, 0, 0);   // A = psi(q) in TMEM, B = psi(k) K-major
    constexpr uint32_t iY = idesc_bf16(128, DV, 0, 1);   // A in TMEM, B MN-major (R~ or V)
    constexpr uint32_t iYk = idesc_bf16(128, DV, 0, 0);  // A in TMEM, B'' K-major
    constexpr uint32_t iYz = idesc_bf16(128, 16, 0, 0);  // A in TMEM, B = zeta~ no swizzle
    constexpr uint32_t iYe = idesc_bf16(128, DV + 64, 0, 1);   // ext: B = [R~ | zeta box]
    constexpr uint32_t iYke = idesc_bf16(128, DV + 16, 0, 0);  // ext: B = [B'' ; Bz row]
    constexpr uint32_t iR = idesc_bf16(128, DV, 1, 1);   // A = psi(k)^T MN-major, B = V MN-major
    constexpr uint32_t iZ = idesc_bf16(128, 16, 1, 0);   // A MN-major, B = [1|beta] no swizzle
    constexpr uint32_t iE = idesc_bf16(128, DV + 64, 1, 1);   // ext: A, B MN-major, N = dv + 64
    constexpr uint32_t aAug = kColAq + D / 2;            // A' columns
    const uint32_t rb = smem_u32(sRt), zb = smem_u32(sZt);
    const uint64_t yaug = smem_desc(smem_u32(sYB), 128, 256, kSwizzleNone);
    const uint64_t zaug = smem_desc(smem_u32(sZB), 128, 256, kSwizzleNone);
    for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1;
        if (!mbar_wait<W>(&S.kv_full[s], (c >> 1) & 1, g, 20)) break;
        if (!mbar_wait<W>(&S.phik_done[s], (c >> 1) & 1, g, 21)) break;
        if (!mbar_wait<W>(&S.phiq_done, c & 1, g, 22)) break;
        LA_TRACE_POINT(c, 10);
        tc_fence_after();
        const uint32_t kb = smem_u32(sK + s * Lay::kKs), vb = smem_u32(sV + s * Lay::kVs);
        const uint32_t ub = smem_u32(sUVB + s * Lay::kUVB);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t bd =
                smem_desc(kb + (ks >> 2) * (kC * 128) + (ks & 3) * 32, 16, 1024, kSwizzle128B);
            mma_ts(tb + kColG, tb + kColAq + ks * 8, bd, iG, ks > 0);
        }
        // + d + alpha_i + beta_j: G is the full weight w_ij
        mma_ts(tb + kColG, tb + aAug, smem_desc(smem_u32(sGB + s * Lay::kGB), 128, 256, kSwizzleNone),
               iG, 1);
        mma_commit(&S.g_full);
        // state update first: it only has to wait for the export of the
        // previous state (out of TMEM), and fills the tensor pipe while the
        // output epilogue of the previous block still reads Y
        if (!mbar_wait<W>(&S.rt_ready, c & 1, g, 23)) break;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kC / 16; ++ks) {
            const uint64_t ad = smem_desc(kb + ks * 2048, kC * 128, 1024, kSwizzle128B);
            const uint64_t vd = smem_desc(vb + ks * 2048, kC * 128, 1024, kSwizzle128B);
            const uint64_t ud = smem_desc(ub + ks * 256, 128, 2048, kSwizzleNone);
            if (Lay::kExt) {   // [psi(K)^T ; weights^T] [V | 1]: R, zeta, u, r at once
                mma_ss(tb + kColR, ad, vd, iE, 1);
            } else {
                mma_ss(tb + kColR, ad, vd, iR, 1);
                mma_ss(tb + kColZ, ad, ud, iZ, 1);
                mma_ss(tb + kColUV, vd, ud, iZ, 1);
            }
        }
        mma_commit(&S.st_full);
        LA_TRACE_POINT(c, 24);
        if (!mbar_wait<W>(&S.y_empty, c & 1, g, 24)) break;
        LA_TRACE_POINT(c, 11);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t bd = smem_desc(rb + ks * 2048, D * 128, 1024, kSwizzle128B);
            if (Lay::kExt) {   // [Y | den ...] = psi(Q) [R~ | zeta~]
                mma_ts(tb + kColY, tb + kColAq + ks * 8, bd, iYe, ks > 0);
            } else {
                mma_ts(tb + kColY, tb + kColAq + ks * 8, bd, iY, ks > 0);
                const uint64_t zd = smem_desc(zb + ks * 256, 128, D * 16, kSwizzleNone);
                mma_ts(tb + kColYz, tb + kColAq + ks * 8, zd, iYz, ks > 0);
            }
        }
        // + (d + alpha_i) u + r and + (d + alpha_i) n + rho
        if (Lay::kExt) {
            mma_ts(tb + kColY, tb + aAug, yaug, iYke, 1);
        } else {
            mma_ts(tb + kColY, tb + aAug, yaug, iYk, 1);
            mma_ts(tb + kColYz, tb + aAug, zaug, iYz, 1);
        }
        // psi(q) and the exported state operands (R~, zeta~, B'', Bz) are free
        mma_commit(&S.aq_free);
        LA_TRACE_POINT(c, 25);
        if (!mbar_wait<W>(&S.h_ready[c & 1], (c >> 1) & 1, g, 25)) break;
        LA_TRACE_POINT(c, 12);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kC / 16; ++ks) {
            const uint64_t vd = smem_desc(vb + ks * 2048, kC * 128, 1024, kSwizzle128B);
            mma_ts(tb + kColY, tb + kColG + ks * 16, vd, iY, 1);
            mma_ts(tb + kColY, tb + kColG + ks * 16 + 8, vd, iY, 1);
        }
        mma_commit(&S.y_full);
        mma_commit(&S.kv_empty[s]);
    }
    // every MMA issued so far has completed once `drain` flips
    mma_commit(&S.drain);
    drain_wait(&S.drain, 0, g.limit_ns);
}

// ------------------------------------------------------------------ state operands
template <int D, int DV>
__device__ __forceinline__ void export_row_bf16(uint8_t *sRt, int row, int grp,
                                                const uint32_t (&rv)[16]) {
    uint32_t pk[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) pk[m] = pack_bf16x2(u2f(rv[2 * m]), u2f(rv[2 * m + 1]));
    const int b0 = grp * 16;
    uint8_t *box = sRt + (b0 >> 6) * (D * 128);
    *reinterpret_cast<uint4 *>(box + sw128_off(row, b0 & 63)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    *reinterpret_cast<uint4 *>(box + sw128_off(row, (b0 & 63) + 8)) =
        make_uint4(pk[4], pk[5], pk[6], pk[7]);
}

// zeta~ operand: [16 x d] K-major, no swizzle; row 0 holds bf16(zeta), rows 1..15 zero.
__device__ __forceinline__ uint32_t zt_off(int n, int k, int D) {
    return (uint32_t)((n >> 3) * (D * 16) + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2);
}

// ------------------------------------------------------------------ group A
// Eight warps, two per TMEM lane quarter; the two threads of a token row
// (halves h = 0, 1) share its work.  Block c: psi(q) of half the features
// each -> TMEM (A operand); h = 0 then adds the augmentation slice A' (with
// alpha_i = sum of psi(q_i) over both halves, before rounding, and d).  Once
// G = w is ready, every other 16-column group each: w_ij (j <= i, else 0)
// split into bf16 hi + lo pairs written back over G, and the partial row sums.
template <int D, int DV, int DK>
__device__ __forceinline__ void group_a_role(Small &S, uint32_t tb, uint8_t *sQ,
                                             int nchunks, int nloc, const Guard &g,
                                             const float *gtab) {
    constexpr int kW = WaitPolicy<D, DK>::value;
    constexpr bool DECAY = DK != 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wq = warp & 3, row = wq * 32 + lane;
    const int h = (warp - kWarpA) >> 2;
    const DecayPow<DK> P{decay_area(S).gpow, gtab};   // touched only with a decay or gates
    // state scale G of block c (the plain layout has no table)
    DecayScale ds(P.first());
    const uint32_t lb = (uint32_t)(wq * 32) << 16;
    const float dd = (float)D;
    // groups entirely above this warp's rows are all zero (causal mask)
    const int last_grp = (wq * 32 + 31) >> 4;
    // the block's decay over its L tokens and its inverse (gsc below); with
    // gates they come from global memory and are loaded one block ahead
    float pL_next = 1.f, ipL_next = 1.f;
    auto fetch = [&](int c) {
        if (DK == 2 && c < nchunks) {
            const int L = min(kC, nloc - c * kC);
            pL_next = P.pw(c, L);
            ipL_next = P.ipw(c, L);
        }
    };
    fetch(0);
    for (int c = 0; c < nchunks; ++c) {
        const int cb = c & 1;
        const int Lc = min(kC, nloc - c * kC);
        const float pL = DK == 2 ? pL_next : (DECAY ? P.pw(c, Lc) : 1.f);
        const float ipL = DK == 2 ? ipL_next : (DECAY ? P.ipw(c, Lc) : 1.f);
        fetch(c + 1);
        if (DECAY) ds.step(pL);
        // Gated kernel: psi(q) is formed as soon as the Q tile has landed, in
        // place over the tile, while the previous block's Y MMAs may still read
        // the TMEM operand, and copied into TMEM once they have completed (h = 0
        // keeps its first eight features' residuals in registers: both halves
        // read those features for the split constant).  That takes psi(q) off
        // the chain to the next G.  The plain and fixed-decay kernels form
        // psi(q) straight into TMEM after that wait: there, the idle time it
        // leaves goes to group B's output epilogue, and the early form was
        // measured 7% slower; the gated kernel gains 3%.
        constexpr bool kEarly = DK == 2;
        bool ok = wait_warp<kW>(&S.q_full, c & 1, g, 40);
        if (!kEarly && ok && c > 0) ok = wait_warp<kW>(&S.aq_free, (c - 1) & 1, g, 41);
        if (lane == 0 && wq == 3 && h == 0) LA_TRACE_POINT(c, 0);
        float alpha = 0.f, cq = 1.f;
        uint64_t alpha2 = f2pack(0.f, 0.f);
        uint4 held = make_uint4(0u, 0u, 0u, 0u);
        auto q_chunk = [&](int f) {
            return reinterpret_cast<uint4 *>(sQ + (f >> 3) * (kC * 128) + sw128_off(row, (f & 7) * 8));
        };
        if (ok) {
            if (!kEarly) tc_fence_after();   // the MMAs that read the previous psi(q) have completed
            // the query's split constant, from its first eight features
            cq = split_const(*reinterpret_cast<const uint4 *>(sQ + sw128_off(row, 0)));
            const SplitC kq = split_pairs(cq);
            // a real loop over 32-feature groups keeps the hot code small
#pragma unroll 1
            for (int gq = 0; gq < D / 64; ++gq) {
                const int grp = h * (D / 64) + gq;   // 32 features -> 16 TMEM columns
                uint4 raw[4];
#pragma unroll
                for (int f4 = 0; f4 < 4; ++f4) raw[f4] = *q_chunk(grp * 4 + f4);
                uint32_t v[16];
#pragma unroll
                for (int f4 = 0; f4 < 4; ++f4) {
                    const uint32_t w[4] = {raw[f4].x, raw[f4].y, raw[f4].z, raw[f4].w};
#pragma unroll
                    for (int hw = 0; hw < 4; ++hw) v[f4 * 4 + hw] = feat_bf16x2_sum(w[hw], kq, alpha2);
                }
                if (kEarly) {
#pragma unroll
                    for (int f4 = 0; f4 < 4; ++f4) {
                        const uint4 o = make_uint4(v[f4 * 4], v[f4 * 4 + 1], v[f4 * 4 + 2], v[f4 * 4 + 3]);
                        if (grp == 0 && f4 == 0) held = o; else *q_chunk(grp * 4 + f4) = o;
                    }
                } else {
                    tmem_st16(tb + lb + kColAq + grp * 16, v);
                }
            }
            if (!kEarly) mbar_arrive(&S.q_empty);
            alpha = f2sum(alpha2);
            if (h == 1) S.alpha_part[row] = alpha;
            if (!kEarly) {
                tmem_wait_st();
                tc_fence_before();
            }
        }
        if (kEarly && ok && c > 0) ok = wait_warp<kW>(&S.aq_free, (c - 1) & 1, g, 41);
        if (kEarly && ok) {
            tc_fence_after();   // the MMAs that read the previous psi(q) have completed
#pragma unroll 1
            for (int gq = 0; gq < D / 64; ++gq) {
                const int grp = h * (D / 64) + gq;
                uint32_t v[16];
#pragma unroll
                for (int f4 = 0; f4 < 4; ++f4) {
                    const uint4 x = (grp == 0 && f4 == 0) ? held : *q_chunk(grp * 4 + f4);
                    v[f4 * 4 + 0] = x.x; v[f4 * 4 + 1] = x.y; v[f4 * 4 + 2] = x.z; v[f4 * 4 + 3] = x.w;
                }
                tmem_st16(tb + lb + kColAq + grp * 16, v);
            }
            fence_proxy_async();   // the in-place writes precede the next copy into the tile
            mbar_arrive(&S.q_empty);
            tmem_wait_st();
            tc_fence_before();
        }
        // both halves of psi(q) are in TMEM, and alpha_part is written, past here
        if (group_any<kBarA, 2 * kWG>(!ok)) break;
        if (h == 0) {   // A' = [c, c, alpha_hi, alpha_lo, d c, alpha_hi, d c, 0, ...]
            alpha += S.alpha_part[row];
            const float ah = bf16_round(alpha), dc = dd * cq;   // d c is exact in bf16
            const uint32_t aug0[4] = {pack_bf16x2(cq, cq), pack_bf16x2(ah, alpha - ah),
                                      pack_bf16x2(dc, ah), pack_bf16x2(dc, 0.f)};
            const uint32_t aug1[4] = {0u, 0u, 0u, 0u};
            tmem_st4(tb + lb + kColAq + D / 2, aug0);
            tmem_st4(tb + lb + kColAq + D / 2 + 4, aug1);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&S.phiq_done);
            if (lane == 0) LA_TRACE_POINT(c, 16 + wq);
            if (lane == 0 && wq == 3) LA_TRACE_POINT(c, 1);
        }
        ok = wait_warp<kW>(&S.g_full, c & 1, g, 43);
        if (ok) {
            tc_fence_after();
            if (lane == 0 && wq == 3 && h == 0) LA_TRACE_POINT(c, 2);
            // decay: the weight tile holds gamma^(L-1-j) w_ij / G (keys
            // pre-scaled), so multiplying by gamma^-L G gives gamma^-(j+1) w_ij,
            // the weight relative to row i's common factor gamma^(i+1)
            const float gsc = DECAY ? ipL * ds.G : 1.f;
            // one 16-column group: w_ij for j <= i (else 0) -> bf16 hi, lo pairs
            // (hi + lo equals w to within about 2^-17 w), on packed fp32 pairs;
            // groups wholly below the warp's rows keep every weight, the
            // diagonal ones mask j > i
            uint64_t rowsum2 = f2pack(0.f, 0.f);
            const uint64_t gsc2 = f2pack(gsc, gsc);
            auto weights = [&](int grp, const uint32_t (&gc)[16]) {
                uint32_t out[16];
                if (grp > last_grp) {
#pragma unroll
                    for (int m = 0; m < 16; ++m) out[m] = 0u;
                } else {
                    const bool full = wq * 32 >= grp * 16 + 15;   // warp-uniform
                    const int lim = full ? 15 : row - grp * 16;
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 2) {
                        uint64_t w2 = f2pack(u2f(gc[jj]), u2f(gc[jj + 1]));
                        if (DECAY) w2 = f2mul(w2, gsc2);
                        if (!full) {
                            float w0, w1;
                            f2unpack(w2, w0, w1);
                            w2 = f2pack(jj <= lim ? w0 : 0.f, jj + 1 <= lim ? w1 : 0.f);
                        }
                        float w0, w1;
                        f2unpack(w2, w0, w1);
                        const uint32_t hi = pack_bf16x2(w0, w1);
                        float l0, l1;
                        f2unpack(f2sub(w2, f2pack(bf16_lo_f(hi), bf16_hi_f(hi))), l0, l1);
                        rowsum2 = f2add(rowsum2, w2);
                        out[jj >> 1] = hi;
                        out[8 + (jj >> 1)] = pack_bf16x2(l0, l1);
                    }
                }
                tmem_st16(tb + lb + kColG + grp * 16, out);
            };
            // this half's groups h, h + 2, h + 4, h + 6, two per loop trip
            // (ping-pong buffers: the TMEM load of the next group overlaps
            // this group's math, and the hot code stays small)
            uint32_t gA[16], gB[16];
            if (h <= last_grp) {
                tmem_ld16(tb + lb + kColG + h * 16, gA);
                tmem_wait_ld();
            }
#pragma unroll 1
            for (int t = 0; t < kC / 64; ++t) {
                const int g0 = h + 4 * t, g1 = g0 + 2, g2 = g0 + 4;
                const bool more = t + 1 < kC / 64;
                if (g1 <= last_grp) tmem_ld16(tb + lb + kColG + g1 * 16, gB);
                weights(g0, gA);
                if (g1 <= last_grp) tmem_wait_ld();
                if (more && g2 <= last_grp) tmem_ld16(tb + lb + kColG + g2 * 16, gA);
                weights(g1, gB);
                if (more && g2 <= last_grp) tmem_wait_ld();
            }
            S.rowsum[cb][h][row] = f2sum(rowsum2);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&S.h_ready[cb]);
            if (lane == 0 && h == 1) LA_TRACE_POINT(c, 20 + wq);
            if (lane == 0 && wq == 3 && h == 1) LA_TRACE_POINT(c, 3);
        }
        if (group_any<kBarA, 2 * kWG>(!ok)) break;
    }
}

// ------------------------------------------------------------------ group B
// Eight warps, two per TMEM lane quarter, the two threads of a row (halves
// h = 0, 1) sharing its work: psi(k) in place over half of the features,
// the state export of half of R's columns, half of the output columns.
template <int D, int DV, int DK>
__device__ __forceinline__ void group_b_role(Small &S, uint32_t tb, uint8_t *sK, uint8_t *sV,
                                             uint8_t *sRt,
                                             uint8_t *sUVB, uint8_t *sZt, uint8_t *sGB,
                                             uint8_t *sYB, uint8_t *sZB,
                                             const TcParams &p, int head, int slot,
                                             int tok0, int nloc, bool last_seg, int nchunks,
                                             const Guard &g, const float *gtab) {
    constexpr int kW = WaitPolicy<D, DK>::value;
    using Lay = Layout<D, DV>;
    constexpr bool DECAY = DK != 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wq = warp & 3, row = wq * 32 + lane;
    const int h = (warp - kWarpB) >> 2;
    const DecayPow<DK> P{decay_area(S).gpow, gtab};   // touched only with a decay or gates
    // scales of the block whose keys phi_k prepares and of the state in TMEM
    // (the export's block); the plain layout has no table
    DecayScale ks(P.first());
    DecayScale xs(P.first());
    const int wtid = tid - kWarpB * 32;   // 0..255
    const uint32_t lb = (uint32_t)(wq * 32) << 16;
    const int N = nloc;   // tokens of this work item (segment)
    constexpr int kRGroups = DV / 32;     // 16-column groups of R (and Y) per half

    ExtScratch &XS = *reinterpret_cast<ExtScratch *>(sUVB);   // ext only
    if (Lay::kExt) {
        // extension boxes zero (the first 16 bytes of a key's row are written
        // per block), ones boxes: first column 1, the rest 0
        for (int e = wtid; e < 2 * kC * 8; e += 2 * kWG) {
            const int st = e / (kC * 8), r = (e / 8) % kC, ch = e % 8;
            *reinterpret_cast<uint4 *>(sK + st * Lay::kKs + Lay::kK + sw128_off(r, ch * 8)) =
                make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4 *>(sV + st * Lay::kVs + Lay::kV + sw128_off(r, ch * 8)) =
                ch == 0 ? make_uint4(pack_bf16x2(1.f, 0.f), 0u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
        }
    } else {
        // operand rows: [1|beta|s] row 0 = ones, rows 5..15 zero (rows 1..4 are
        // written per block by psi(k))
        for (int e = wtid; e < 2 * 16 * kC; e += 2 * kWG) {
            const int s = e / (16 * kC), rem = e % (16 * kC), n = rem / kC, k = rem % kC;
            *reinterpret_cast<__nv_bfloat16 *>(sUVB + s * Lay::kUVB + (n >> 3) * 2048 +
                                               (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2) =
                __float2bfloat16_rn(n == 0 ? 1.f : 0.f);
        }
    }
    // zeta~ all zero
    for (int e = wtid; e < 16 * D; e += 2 * kWG)
        *reinterpret_cast<__nv_bfloat16 *>(sZt + zt_off(e / D, e % D, D)) = __float2bfloat16_rn(0.f);
    // B' rows: slots 8..15 are zero for good (slots 0..7 are written per block)
    *reinterpret_cast<uint4 *>(sGB + h * Lay::kGB + k16_off(row, 8)) = make_uint4(0u, 0u, 0u, 0u);
    // B'' row of column c, Bz row 0: [x_hi, x_lo, y_hi, y_hi, y_hi, y_lo, y_lo, 0 | 0...]
    // for (x, y) = (r_c, u_c) and (rho, n)
    auto aug_row = [](uint8_t *tile, int n, float x, float y) {
        const float xh = bf16_round(x), yh = bf16_round(y);
        const float yl = y - yh;
        *reinterpret_cast<uint4 *>(tile + k16_off(n, 0)) =
            make_uint4(pack_bf16x2(xh, x - xh), pack_bf16x2(yh, yh), pack_bf16x2(yh, yl),
                       pack_bf16x2(yl, 0.f));
        *reinterpret_cast<uint4 *>(tile + k16_off(n, 8)) = make_uint4(0u, 0u, 0u, 0u);
    };
    if (wtid > 0 && wtid < 16) aug_row(sZB, wtid, 0.f, 0.f);   // rows 1..15 of Bz stay zero
    if (Lay::kExt) {
        // the zeta box (column 0 written per export) and B'' rows dv+1..dv+15 zero
        for (int e = wtid; e < D * 8; e += 2 * kWG)
            *reinterpret_cast<uint4 *>(sRt + D * DV * 2 + sw128_off(e / 8, (e % 8) * 8)) =
                make_uint4(0u, 0u, 0u, 0u);
        if (wtid > 0 && wtid < 16) aug_row(sYB, DV + wtid, 0.f, 0.f);
    }
    mbar_arrive(&S.y_empty);   // Y is free for block 0


    // ---- initial state in split form S = 1 u^T + R, z = n 1 + zeta (u = first row
    //      of S, n = first entry of z; zero when absent); buffers [1] = "block -1"
    {
        // initial state of this work item: the caller's state for a whole
        // head, or the exclusive prefix of this segment
        const float *Sin = p.S_in ? p.S_in + (size_t)slot * D * DV : nullptr;
        const float *zin = p.z_in ? p.z_in + (size_t)slot * D : nullptr;
        // decay: the initial state enters TMEM divided by G0, and already
        // multiplied by gamma^L of block 0 when the scale restarts there
        const float p0 = DECAY ? P.pw(0, min(kC, N)) : 1.f;
        if (DECAY) xs.step(p0);
        const float g0 = DECAY ? (xs.renorm ? p0 : 1.f) / xs.G0 : 1.f;
        // u = the first row of S, r = the column sums of R = S - 1 u^T (per dv
        // column: thread row takes column row)
        float u0 = 0.f, r0 = 0.f;
        if (h == 0 && Sin && row < DV) {
            u0 = Sin[row];
            // independent loads, issued 16 at a time ahead of the sums
#pragma unroll 16
            for (int a = 1; a < D; ++a) r0 += Sin[(size_t)a * DV + row] - u0;
        }
        if (Lay::kExt) {   // rows 64 and 66 of the accumulator start from u and r
            if (h == 0 && row < DV) {
                S.u[1][row] = u0;
                XS.r0[row] = r0;
            }
            named_bar(kBarB, 2 * kWG);
        }
#pragma unroll
        for (int gq = 0; gq < kRGroups; ++gq) {
            const int grp = h * kRGroups + gq;
            uint32_t v[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) {
                const int b = grp * 16 + jj;
                float x = (Sin && row < D) ? Sin[(size_t)row * DV + b] - Sin[b] : 0.f;
                if (Lay::kExt && row == 64) x = S.u[1][b];
                if (Lay::kExt && row == 66) x = XS.r0[b];
                v[jj] = f2u(x);
            }
            if (row < D) export_row_bf16<D, DV>(sRt, row, grp, v);
            if (DECAY) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) v[jj] = f2u(u2f(v[jj]) * g0);
            }
            tmem_st16(tb + lb + kColR + grp * 16, v);
        }
        float zeta0 = 0.f;
        if (h == 0) {
            zeta0 = (zin && row < D) ? zin[row] - zin[0] : 0.f;
            const uint32_t zv[4] = {f2u(zeta0 * g0), 0u, 0u, 0u};
            if (Lay::kExt) {
                tmem_st4(tb + lb + kColR + DV, zv);   // the ones column
            } else {
                tmem_st4(tb + lb + kColZ, zv);
                // columns [sum v | r_hi | r_lo | u_hi | u_lo | 0 0 0]
                const uint32_t uv[4] = {0u, f2u(r0 * g0), 0u, f2u(u0 * g0)};
                const uint32_t uw[4] = {0u, 0u, 0u, 0u};
                tmem_st4(tb + lb + kColUV, uv);
                tmem_st4(tb + lb + kColUV + 4, uw);
            }
            S.zeta[row] = zeta0;
            S.u[1][row] = u0;
            if (row < DV) aug_row(sYB, row, r0, u0);
        }
        named_bar(kBarB, 2 * kWG);  // zero rows of zeta~ written before row 0 below
        if (h == 0 && row < D) {
            if (Lay::kExt)
                *reinterpret_cast<__nv_bfloat16 *>(sRt + D * DV * 2 + sw128_off(row, 0)) =
                    __float2bfloat16_rn(zeta0);
            else
                *reinterpret_cast<__nv_bfloat16 *>(sZt + zt_off(0, row, D)) = __float2bfloat16_rn(zeta0);
        }
        if (wtid == 0) {
            float rho0 = 0.f;
            if (zin) {
                const float z0 = zin[0];
#pragma unroll 16
                for (int a = 1; a < D; ++a) rho0 += zin[a] - z0;
            }
            S.n_s[1] = zin ? zin[0] : 0.f;
            S.rho_s[1] = rho0;
            aug_row(Lay::kExt ? sYB : sZB, Lay::kExt ? DV : 0, rho0, S.n_s[1]);
        }
        tmem_wait_st();
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&S.rt_ready);   // every thread, after its own writes
    }

    // psi(k) in place (bf16) over this half's features; beta_j = sum of the
    // row (before rounding) over both halves; h = 0 writes the [1|beta] and B' rows.
    // Returns false when the group gave up (agreed at the group barrier).
    // Decay factors.  With gates they come from global memory and each is
    // loaded one call ahead: phi_k's block decay and key weight, the export's
    // decays of blocks c and c + 1, the epilogue's 1 / (decay through token i).
    float kf_pL = 1.f, kf_kw = 1.f, ex_cur = 1.f, ex_next = 1.f, ep_ipw = 1.f;
    auto kfetch = [&](int c) {
        if (DK == 2 && c < nchunks) {
            const int L = min(kC, N - c * kC);
            kf_pL = P.pw(c, L);
            kf_kw = row < L ? P.key_weight(c, L, row) : 0.f;
        }
    };
    auto bdecay = [&](int c) { return (DECAY && c < nchunks) ? P.pw(c, min(kC, N - c * kC)) : 1.f; };
    if (DK == 2) {
        kfetch(0);
        ex_cur = bdecay(0);
        ex_next = bdecay(1);
        ep_ipw = P.ipw(0, row + 1);
    }

    auto phi_k = [&](int c) -> bool {
        const int s = c & 1, cb = c & 1;
        // decay: key j of a block of L tokens enters with weight
        // s_j = gamma^(L-1-j), its share of the state after the block
        // (padding rows: 0)
        const int L = min(kC, N - c * kC);
        float sc = 1.f;
        if (DECAY) {   // s_j / G, with s_j = (decay of the whole block) / (decay up to key j)
            ks.step(DK == 2 ? kf_pL : P.pw(c, L));
            sc = (DK == 2 ? kf_kw : (row < L ? P.key_weight(c, L, row) : 0.f)) / ks.G;
        }
        kfetch(c + 1);
        const bool ok = wait_warp<kW>(&S.kv_full[s], (c >> 1) & 1, g, 50);
        if (lane == 0 && wq == 3 && h == 0) LA_TRACE_POINT(c, 6);
        uint8_t *kt = sK + s * Lay::kKs;
        // the key's split constant from its first eight features (in h = 0's
        // half; padding rows read zeros: c' = 1).  Both halves read them from
        // the tile; h = 0 writes their residuals back only after the group
        // barrier below, by which time h = 1 has read them.
        uint4 first = make_uint4(0u, 0u, 0u, 0u);
        if (ok) first = *reinterpret_cast<const uint4 *>(kt + sw128_off(row, 0));
        const float ck = split_const(first);
        const SplitC kk = split_pairs(ck);
        uint4 held = make_uint4(0u, 0u, 0u, 0u);   // h = 0: residuals of features 0..7
        float beta = 0.f;
        uint64_t beta2 = f2pack(0.f, 0.f);
        if (ok) {
            constexpr int kChunks = D / 16;                       // 8-feature chunks per half
            constexpr int kBatch = kChunks < 8 ? kChunks : 8;
            // all loads of a batch are issued before its in-place stores so
            // their latencies overlap
#pragma unroll 1
            for (int b0 = 0; b0 < kChunks; b0 += kBatch) {
                const int f0 = h * kChunks + b0;
                uint4 raw[kBatch];
#pragma unroll
                for (int f = 0; f < kBatch; ++f)
                    raw[f] = *reinterpret_cast<const uint4 *>(
                        kt + ((f0 + f) >> 3) * (kC * 128) + sw128_off(row, ((f0 + f) & 7) * 8));
#pragma unroll
                for (int f = 0; f < kBatch; ++f) {
                    uint32_t w[4] = {raw[f].x, raw[f].y, raw[f].z, raw[f].w};
#pragma unroll
                    for (int hw = 0; hw < 4; ++hw) {
                        w[hw] = DECAY ? feat_scaled_bf16x2_sum(w[hw], kk, sc, beta2)
                                      : feat_bf16x2_sum(w[hw], kk, beta2);
                    }
                    raw[f] = make_uint4(w[0], w[1], w[2], w[3]);
                }
#pragma unroll
                for (int f = 0; f < kBatch; ++f) {
                    if (f0 + f == 0)
                        held = raw[f];
                    else
                        *reinterpret_cast<uint4 *>(kt + ((f0 + f) >> 3) * (kC * 128) +
                                                   sw128_off(row, ((f0 + f) & 7) * 8)) = raw[f];
                }
            }
            beta = f2sum(beta2);
            if (h == 1) S.beta_part[row] = beta;
            fence_proxy_async();
        }
        if (group_any<kBarB, 2 * kWG>(!ok)) return false;
        if (h == 0) {
            *reinterpret_cast<uint4 *>(kt + sw128_off(row, 0)) = held;
            beta += S.beta_part[row];
            const float bh = bf16_round(beta);
            // key weight s_j = sc c'_j as a bf16 pair: the key's constant part,
            // times its decay weight over G with a decay (c'_j itself, a bf16
            // value, without one); 0 for padding rows
            const float sj = row < L ? sc * ck : 0.f;
            const float sh = bf16_round(sj), sl = bf16_round(sj - sh);
            if (Lay::kExt) {
                // the key's row of the extension box: [s_hi, s_lo, beta_hi, beta_lo, 0 ...]
                // (rows 64..67 of the state MMA's A: u and r accumulate there)
                *reinterpret_cast<uint4 *>(kt + Lay::kK + sw128_off(row, 0)) =
                    make_uint4(pack_bf16x2(sh, sl), pack_bf16x2(bh, beta - bh), 0u, 0u);
            } else {
                uint8_t *ubp = sUVB + s * Lay::kUVB + (row >> 3) * 128 + (row & 7) * 2;
                *reinterpret_cast<__nv_bfloat16 *>(ubp + 16) = __float2bfloat16_rn(bh);
                *reinterpret_cast<__nv_bfloat16 *>(ubp + 32) = __float2bfloat16_rn(beta - bh);
                // rows 3, 4 of [1|beta|s]: u += V^T s (row 0 stays 1: it also
                // feeds zeta += psi_c(K)^T 1)
                *reinterpret_cast<__nv_bfloat16 *>(ubp + 48) = __float2bfloat16_rn(sh);
                *reinterpret_cast<__nv_bfloat16 *>(ubp + 64) = __float2bfloat16_rn(sl);
            }
            // B' row of key j: [beta_hi, beta_lo, s_hi, s_hi, s_hi, s_lo, s_lo, 0]
            // (beta is the sum of the residual features, scaled with a decay)
            *reinterpret_cast<uint4 *>(sGB + s * Lay::kGB + k16_off(row, 0)) =
                make_uint4(pack_bf16x2(bh, beta - bh), pack_bf16x2(sh, sh), pack_bf16x2(sh, sl),
                           pack_bf16x2(sl, 0.f));
            const float bsum = warp_sum_f(beta);
            const float ssum = warp_sum_f(sh + sl);
            if (lane == 0) {
                S.rho_part[cb][wq] = bsum;
                S.s_part[cb][wq] = ssum;
            }
            fence_proxy_async();
            mbar_arrive(&S.phik_done[s]);
            if (lane == 0) LA_TRACE_POINT(c, 26 + wq);
            if (lane == 0 && wq == 3) LA_TRACE_POINT(c, 7);
        }
        return true;
    };

    // state after block c: R -> bf16 operand (this half's columns); h = 0:
    // zeta -> zeta~, u, r, n, rho and the augmentation rows
    auto export_state = [&](int c) -> bool {
        const int cb = c & 1, pb = (c + 1) & 1;
        const int L = min(kC, N - c * kC);
        // decay: the state after block c is G times the TMEM contents; when
        // the scale restarts at block c+1, the state is multiplied by gamma^L
        // of block c+1 over G0 and written back before that block's update
        const float G = DECAY ? xs.G : 1.f;
        // the decays of blocks c and c + 1
        const float gcur = DK == 2 ? ex_cur : bdecay(c);
        const float gL = DK == 2 ? ex_next : bdecay(c + 1);
        if (DK == 2) {
            ex_cur = ex_next;
            ex_next = bdecay(c + 2);
        }
        bool rescale = false;
        float gnext = 1.f;
        if (DECAY && c + 1 < nchunks) {
            xs.step(gL);
            rescale = xs.renorm;
            gnext = gL / xs.G0;
        }
        if (!wait_warp<kW>(&S.st_full, c & 1, g, 51) || !wait_warp<kW>(&S.aq_free, c & 1, g, 54))
            return false;
        if (lane == 0 && wq == 3 && h == 0) LA_TRACE_POINT(c, 4);
        tc_fence_after();
#pragma unroll
        for (int gq = 0; gq < kRGroups; gq += 2) {
            const int grp = h * kRGroups + gq;
            uint32_t rv0[16], rv1[16];
            tmem_ld16(tb + lb + kColR + grp * 16, rv0);
            tmem_ld16(tb + lb + kColR + (grp + 1) * 16, rv1);
            tmem_wait_ld();
            if (DECAY) {
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    rv0[m] = f2u(u2f(rv0[m]) * G);
                    rv1[m] = f2u(u2f(rv1[m]) * G);
                }
            }
            if (row < D) {
                export_row_bf16<D, DV>(sRt, row, grp, rv0);
                export_row_bf16<D, DV>(sRt, row, grp + 1, rv1);
            } else if (Lay::kExt && row < 68) {   // rows 64..67: the u and r parts
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    XS.uv[row - 64][grp * 16 + m] = u2f(rv0[m]);
                    XS.uv[row - 64][(grp + 1) * 16 + m] = u2f(rv1[m]);
                }
            }
            if (rescale) {
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    rv0[m] = f2u(u2f(rv0[m]) * gnext);
                    rv1[m] = f2u(u2f(rv1[m]) * gnext);
                }
                tmem_st16(tb + lb + kColR + grp * 16, rv0);
                tmem_st16(tb + lb + kColR + (grp + 1) * 16, rv1);
            }
        }
        if (Lay::kExt) named_bar(kBarB, 2 * kWG);   // the u and r parts are in the scratch
        if (h == 0) {
            uint32_t zv[4], uv[4] = {0u, 0u, 0u, 0u}, uw[4] = {0u, 0u, 0u, 0u};
            if (Lay::kExt) {
                tmem_ld4(tb + lb + kColR + DV, zv);   // zeta in the ones column
            } else {
                tmem_ld4(tb + lb + kColZ, zv);
                tmem_ld4(tb + lb + kColUV, uv);
                tmem_ld4(tb + lb + kColUV + 4, uw);
            }
            tmem_wait_ld();
            if (DECAY) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    zv[m] = f2u(u2f(zv[m]) * G);
                    uv[m] = f2u(u2f(uv[m]) * G);
                    uw[m] = f2u(u2f(uw[m]) * G);
                }
            }
            // u and r per dv column (thread row takes column row)
            const float u = Lay::kExt ? (row < DV ? XS.uv[0][row] + XS.uv[1][row] : 0.f)
                                      : u2f(uv[3]) + u2f(uw[0]);
            const float rr = Lay::kExt ? (row < DV ? XS.uv[2][row] + XS.uv[3][row] : 0.f)
                                       : u2f(uv[1]) + u2f(uv[2]);
            if (row < D) {
                S.zeta[row] = u2f(zv[0]);
                if (Lay::kExt)
                    *reinterpret_cast<__nv_bfloat16 *>(sRt + D * DV * 2 + sw128_off(row, 0)) =
                        __float2bfloat16_rn(u2f(zv[0]));
                else
                    *reinterpret_cast<__nv_bfloat16 *>(sZt + zt_off(0, row, D)) =
                        __float2bfloat16_rn(u2f(zv[0]));
            }
            S.u[cb][row] = u;
            if (row < DV) aug_row(sYB, row, rr, u);
            if (wtid == 0) {
                const float rsum = (S.rho_part[cb][0] + S.rho_part[cb][1]) +
                                   (S.rho_part[cb][2] + S.rho_part[cb][3]);
                // n = sum of the keys' constants (the token count when every
                // constant is 1)
                const float ssum = (S.s_part[cb][0] + S.s_part[cb][1]) +
                                   (S.s_part[cb][2] + S.s_part[cb][3]);
                if (DECAY) {   // n and rho decay like the state: x <- gamma^L x + sum_j s_j x_j
                    S.n_s[cb] = fmaf(gcur, S.n_s[pb], G * ssum);
                    S.rho_s[cb] = fmaf(gcur, S.rho_s[pb], G * rsum);
                } else {
                    S.n_s[cb] = S.n_s[pb] + ssum;
                    S.rho_s[cb] = S.rho_s[pb] + rsum;
                }
                aug_row(Lay::kExt ? sYB : sZB, Lay::kExt ? DV : 0, S.rho_s[cb], S.n_s[cb]);
            }
            if (rescale) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    zv[m] = f2u(u2f(zv[m]) * gnext);
                    uv[m] = f2u(u2f(uv[m]) * gnext);
                    uw[m] = f2u(u2f(uw[m]) * gnext);
                }
                if (Lay::kExt) {
                    tmem_st4(tb + lb + kColR + DV, zv);
                } else {
                    tmem_st4(tb + lb + kColZ, zv);
                    tmem_st4(tb + lb + kColUV, uv);
                    tmem_st4(tb + lb + kColUV + 4, uw);
                }
            }
        }
        if (rescale) tmem_wait_st();
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&S.rt_ready);
        if (lane == 0 && wq == 3 && h == 0) LA_TRACE_POINT(c, 5);
        return true;
    };

    // y = Y / max(Yz + rowsum, eps): the tensor core has already summed every
    // part of the numerator ((d + alpha) u + r + a R + P V) and the inter-block
    // denominator ((d + alpha) n + rho + a.zeta).  Each thread takes 1/den of
    // its own row; the values are then read back through the 16x256b TMEM
    // shape, where 4 neighbouring lanes hold 8 consecutive columns of one row,
    // so every warp store writes whole 32-byte sectors (8 rows x 32 bytes).
    // Half h takes the 16-lane half h of its quarter (parts h, h + 2, ...).
    auto epilogue = [&](int c) -> bool {
        const int t0 = c * kC, cb = c & 1;
        // decay: row i's numerator and denominator are both carried divided by
        // gamma^(i+1) (the decay from the block's start through token i), so
        // the clamp max(den, eps) becomes max(den', eps gamma^-(i+1))
        const float eps_row = DECAY ? p.eps * (DK == 2 ? ep_ipw : P.ipw(c, row + 1)) : p.eps;
        if (DK == 2 && c + 1 < nchunks) ep_ipw = P.ipw(c + 1, row + 1);
        if (!wait_warp<kW>(&S.h_ready[cb], (c >> 1) & 1, g, 52) || !wait_warp<kW>(&S.y_full, c & 1, g, 53))
            return false;
        if (lane == 0 && wq == 3 && h == 0) LA_TRACE_POINT(c, 8);
        tc_fence_after();
        uint32_t yz[4];
        tmem_ld4(tb + lb + (Lay::kExt ? kColY + DV : kColYz), yz);   // den (ext: the column after Y)
        tmem_wait_ld();
        S.e_inv[h][row] =
            1.f / fmaxf(u2f(yz[0]) + (S.rowsum[cb][0][row] + S.rowsum[cb][1][row]), eps_row);
        __syncwarp();
        float *ychunk = p.y + ((size_t)head * p.N + tok0 + t0) * DV;
        const int tq = lane >> 2, tc = (lane & 3) * 2;
        constexpr int kParts = 2 * (DV / 64);   // (16-lane half, 64-column block) pairs
        auto part_addr = [&](int part) {
            return tb + ((uint32_t)(wq * 32 + 16 * (part & 1)) << 16) + kColY + (part >> 1) * 64;
        };
        const float *einv = S.e_inv[h];
        auto outputs = [&](int part, const uint32_t (&vc)[32]) {
            const int half = part & 1, cblk = part >> 1;
            const int rA = wq * 32 + 16 * half + tq, rB = rA + 8;
            const uint64_t invA = f2pack(einv[rA], einv[rA]), invB = f2pack(einv[rB], einv[rB]);
            const bool okA = t0 + rA < N, okB = t0 + rB < N;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int col = cblk * 64 + 8 * k + tc;
                float2 oA, oB;
                f2unpack(f2mul(f2pack(u2f(vc[4 * k]), u2f(vc[4 * k + 1])), invA), oA.x, oA.y);
                f2unpack(f2mul(f2pack(u2f(vc[4 * k + 2]), u2f(vc[4 * k + 3])), invB), oB.x, oB.y);
                if (okA) *reinterpret_cast<float2 *>(ychunk + (size_t)rA * DV + col) = oA;
                if (okB) *reinterpret_cast<float2 *>(ychunk + (size_t)rB * DV + col) = oB;
            }
        };
        uint32_t vA[32];
#pragma unroll 1
        for (int part = h; part < kParts; part += 2) {
            tmem_ld_16x256b_x8(part_addr(part), vA);
            tmem_wait_ld();
            outputs(part, vA);
        }
        tc_fence_before();
        mbar_arrive(&S.y_empty);
        if (lane == 0 && wq == 3 && h == 0) LA_TRACE_POINT(c, 9);
        return true;
    };

    // Software pipeline, psi(k) two blocks ahead: iteration c runs the outputs
    // of block c, psi(k) of block c+2 and the state export after block c+1.
    bool aborted = !phi_k(0);
    if (!aborted && nchunks > 1) aborted = !phi_k(1);
    if (!aborted) aborted = group_any<kBarB, 2 * kWG>(!export_state(0));
    for (int c = 0; c < nchunks && !aborted; ++c) {
        bool ok = epilogue(c);
        if (group_any<kBarB, 2 * kWG>(!ok)) { aborted = true; break; }
        if (c + 2 < nchunks && !phi_k(c + 2)) { aborted = true; break; }
        if (c + 1 < nchunks) ok = export_state(c + 1);
        if (group_any<kBarB, 2 * kWG>(!ok)) aborted = true;
    }

    // ---- final state S = 1 u^T + R (R read back in fp32), z = n 1 + zeta
    if (!aborted && p.S_out && last_seg) {
        const int lbuf = (nchunks - 1) & 1;
        const float Gl = DECAY ? xs.G : 1.f;   // the last block's state scale
        tc_fence_after();
#pragma unroll
        for (int gq = 0; gq < kRGroups; ++gq) {
            const int grp = h * kRGroups + gq;
            uint32_t rv[16];
            tmem_ld16(tb + lb + kColR + grp * 16, rv);
            tmem_wait_ld();
            if (row < D) {
                float *dst = p.S_out + ((size_t)head * D + row) * DV + grp * 16;
#pragma unroll
                for (int jj = 0; jj < 16; jj += 4)
                    *reinterpret_cast<float4 *>(dst + jj) = make_float4(
                        fmaf(u2f(rv[jj]), Gl, S.u[lbuf][grp * 16 + jj]),
                        fmaf(u2f(rv[jj + 1]), Gl, S.u[lbuf][grp * 16 + jj + 1]),
                        fmaf(u2f(rv[jj + 2]), Gl, S.u[lbuf][grp * 16 + jj + 2]),
                        fmaf(u2f(rv[jj + 3]), Gl, S.u[lbuf][grp * 16 + jj + 3]));
            }
        }
        if (h == 0 && row < D) p.z_out[(size_t)head * D + row] = S.n_s[lbuf] + S.zeta[row];
    }
}

// ------------------------------------------------------------------ kernel
template <int D, int DV, int DK>
__global__ void __launch_bounds__(kThreads, 1)
causal_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap,
                 const TcParams p)
{
    using Lay = Layout<D, DV, DK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    Small &S = *reinterpret_cast<Small *>(sm + Lay::oSmall);
    uint8_t *sQ = sm + Lay::oQ, *sK = sm + Lay::oK, *sV = sm + Lay::oV;
    uint8_t *sRt = sm + Lay::oRt, *sUVB = sm + Lay::oUVB, *sZt = sm + Lay::oZt;
    uint8_t *sGB = sm + Lay::oGB, *sYB = sm + Lay::oYB, *sZB = sm + Lay::oZB;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // work item = (head, segment of seg_chunks blocks); slot: the index of
    // its initial state
    const int item = blockIdx.x;
    const int head = item / p.nseg, seg = item - head * p.nseg;
    const int slot = item;
    int tok0, nloc;
    segment_range(p, seg, tok0, nloc);
    const int nchunks = (nloc + kC - 1) / kC;
    const Guard g{&S.abort_flag, p.err, p.err_where, p.limit_ns};
    // decay: heads whose gamma this kernel does not take are left entirely to
    // the CUDA-core kernel that follows (the whole CTA leaves before any
    // barrier, TMEM allocation or write, so their y, S_out and z_out, and an
    // S_in aliased by S_out, are untouched here)
    if (DK == 1 && !decay_on_tensor_cores(p.gamma[head % p.H])) return;
    // gates: likewise for heads with a gate outside [2^-1/2, 1]
    const float *gtab = nullptr;
    if (DK == 2) {
        if (p.gate_skip[head] != 0u) return;
        gtab = p.gate_tab + ((size_t)head * p.gate_blocks + tok0 / kC) * kGateTab;
    }
    if (tid == 0) LA_TRACE_POINT(0, 15);
    // decay (one segment per head): powers of the head's gamma, read by both
    // row-worker groups (visible after the __syncthreads below)
    if (DK == 1 && tid < kC + 2) {
        DecaySmall &X = decay_area(S);
        const float gam = p.gamma[head % p.H];
        X.gpow[0][tid] = powf(gam, (float)tid);
        X.gpow[1][tid] = powf(gam, -(float)tid);
    }

    if (tid == 0) {
        S.abort_flag = 0;
        mbar_init(&S.q_full, 1);
        mbar_init(&S.q_empty, 2 * kWG);        // every group-A thread
        for (int s = 0; s < 2; ++s) {
            mbar_init(&S.kv_full[s], 1);
            mbar_init(&S.kv_empty[s], 1);
        }
        mbar_init(&S.phiq_done, kWG);          // group-A first halves
        mbar_init(&S.phik_done[0], kWG);       // group-B first halves
        mbar_init(&S.phik_done[1], kWG);
        mbar_init(&S.g_full, 1);
        mbar_init(&S.aq_free, 1);
        mbar_init(&S.h_ready[0], 2 * kWG);     // every group-A thread
        mbar_init(&S.h_ready[1], 2 * kWG);
        mbar_init(&S.st_full, 1);
        mbar_init(&S.rt_ready, 2 * kWG);       // every group-B thread
        mbar_init(&S.y_full, 1);
        mbar_init(&S.y_empty, 2 * kWG);        // every group-B thread
        mbar_init(&S.drain, 1);
        fence_mbar_init();
        prefetch_tmap(&qmap);
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
    }
    if (warp == 1) {
        tmem_alloc(&S.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem_base;

    // With the sequence split, this kernel may start while the prefix scan
    // still runs (programmatic dependent launch): every thread but the
    // producer waits for it here, before its first bounded wait or read of
    // the initial state; the producer waits after issuing block 0's copies.
    if (warp != 0) griddep_wait();
    if (warp == 0) {
        if (lane == 0) producer_role<D, DV, WaitPolicy<D, DK>::value>(S, sQ, sK, sV, &qmap, &kmap, &vmap, head, tok0, nchunks,
                                           item == p.drop_item, g);
    } else if (warp == 1) {
        if (lane == 0)
            mma_role<D, DV, WaitPolicy<D, DK>::value>(S, tb, sK, sV, sRt, sUVB, sZt, sGB, sYB, sZB,
                                                      nchunks, g);
    } else if (warp < kWarpB) {
        group_a_role<D, DV, DK>(S, tb, sQ, nchunks, nloc, g, gtab);
    } else {
        group_b_role<D, DV, DK>(S, tb, sK, sV, sRt, sUVB, sZt, sGB, sYB, sZB, p, head, slot, tok0,
                                nloc, seg == p.nseg - 1, nchunks, g, gtab);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tb, kTmemCols);
    }
}

// ------------------------------------------------------------------ segment prefix scan
// Exclusive prefix over the segments of each head, in a fixed order:
// P_0 = S_in (or 0), P_s = f_{s-1} P_{s-1} + S_{s-1}; the same for z.  f = 1,
// or with a per-head decay gamma^(segment length) (every segment but the last
// has the same length, seg_len, and the last one's state is neither used nor
// computed), or with gates the segment's product of gates (seg_decay, from
// the state pass).  One thread per state element (grid: heads x element
// blocks); the segment loop issues its loads ahead of the running sum.
constexpr int kScanThreads = 128;
__global__ void __launch_bounds__(kScanThreads)
scan_states_kernel(const float *__restrict__ S_seg, const float *__restrict__ z_seg,
                   float *__restrict__ S_pre, float *__restrict__ z_pre,
                   const float *__restrict__ S_in, const float *__restrict__ z_in, int nseg,
                   int D, int DV, const float *__restrict__ gamma, int H, int seg_len,
                   const float *__restrict__ seg_decay)
{
    griddep_launch_dependents();
    griddep_wait();   // S_seg, z_seg come from the state pass
    const int head = blockIdx.x;
    const int nS = D * DV;
    const int e = blockIdx.y * kScanThreads + threadIdx.x;
    if (e >= nS + D) return;
    const bool isS = e < nS;
    const int o = isS ? e : e - nS;
    const float *src = isS ? S_seg : z_seg;
    float *dst = isS ? S_pre : z_pre;
    const size_t stride = isS ? (size_t)nS : (size_t)D;
    float acc = 0.f;
    if (isS && S_in) acc = S_in[(size_t)head * nS + o];
    if (!isS && z_in) acc = z_in[(size_t)head * D + o];
    const float f = gamma ? powf(gamma[head % H], (float)seg_len) : 1.f;
    const size_t base = (size_t)head * nseg * stride + o;
    int sg = 0;
    if (seg_decay) {   // gates: a factor per segment
        const float *fs = seg_decay + (size_t)head * nseg;
        for (; sg < nseg - 1; ++sg) {
            dst[base + sg * stride] = acc;
            acc = fmaf(__ldg(fs + sg), acc, src[base + sg * stride]);
        }
        dst[base + (size_t)(nseg - 1) * stride] = acc;
        return;
    }
    for (; sg + 4 <= nseg - 1; sg += 4) {
        const float s0 = src[base + (sg + 0) * stride], s1 = src[base + (sg + 1) * stride];
        const float s2 = src[base + (sg + 2) * stride], s3 = src[base + (sg + 3) * stride];
        dst[base + (sg + 0) * stride] = acc; acc = fmaf(f, acc, s0);
        dst[base + (sg + 1) * stride] = acc; acc = fmaf(f, acc, s1);
        dst[base + (sg + 2) * stride] = acc; acc = fmaf(f, acc, s2);
        dst[base + (sg + 3) * stride] = acc; acc = fmaf(f, acc, s3);
    }
    for (; sg < nseg - 1; ++sg) {
        dst[base + sg * stride] = acc;
        acc = fmaf(f, acc, src[base + sg * stride]);
    }
    dst[base + (size_t)(nseg - 1) * stride] = acc;
}

// ------------------------------------------------------------------ host side
// Split the sequence only when the heads alone leave SMs idle: then aim for
// about four waves of (head, segment) items, at least one block per segment.
// (A short-then-long split of one wave of heads, to fill the SMs it leaves
// idle, measured slower on B8 H16 N8192 and is not used.)
void choose_segments(int BH, int N, int &nseg, int &seg_chunks) {
    const int nch = (N + kC - 1) / kC;
    const int sms = num_sms();
    nseg = 1;
    seg_chunks = nch > 0 ? nch : 1;
    if (nch <= 1 || 5 * BH >= 3 * sms) return;
    int target = (4 * sms + BH - 1) / BH;
    if (target > nch) target = nch;
    seg_chunks = (nch + target - 1) / target;
    nseg = (nch + seg_chunks - 1) / seg_chunks;
}

size_t segment_workspace(int BH, int N, int d, int dv) {
    int nseg, seg_chunks;
    choose_segments(BH, N, nseg, seg_chunks);
    if (nseg <= 1) return sizeof(WsHeader);
    return sizeof(WsHeader) + 2 * sizeof(float) * (size_t)BH * nseg * ((size_t)d * dv + d);
}

// Per-token gates: the per-block tables of gate products (kGateTab floats per
// block, see DecayPow) and the per-head flag of a gate outside [2^-1/2, 1]
// (the flags start at zero).  One warp per (head, block): lane l takes the
// block's gates 4l .. 4l+3, multiplies them in order, and a warp scan
// multiplies in the products of the lanes below it.
constexpr int kGateWarps = 4;
__global__ void __launch_bounds__(kGateWarps * 32)
gate_tables_kernel(const float *__restrict__ gate, int N, int nblocks, float *__restrict__ tab,
                   unsigned int *__restrict__ skip)
{
    const int lane = threadIdx.x & 31;
    const int blk = blockIdx.x * kGateWarps + (threadIdx.x >> 5), head = blockIdx.y;
    if (blk >= nblocks) return;
    const int t0 = blk * kC + 4 * lane;
    float gv[4];
    bool bad = false;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int t = t0 + k;
        gv[k] = t < N ? gate[(size_t)head * N + t] : 1.f;
        bad |= !(gv[k] >= kGateMin && gv[k] <= 1.f);   // NaN counts as outside
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&skip[head], 1u);
    float loc[4];
    loc[0] = gv[0];
#pragma unroll
    for (int k = 1; k < 4; ++k) loc[k] = loc[k - 1] * gv[k];
    float x = loc[3];   // inclusive scan of the lanes' products
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x *= y;
    }
    float ex = __shfl_up_sync(0xffffffffu, x, 1);
    if (lane == 0) ex = 1.f;
    float *tb = tab + ((size_t)head * nblocks + blk) * kGateTab;
    if (lane == 0) {
        tb[0] = 1.f;
        tb[kGateInv] = 1.f;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float P = ex * loc[k];
        tb[4 * lane + k + 1] = P;
        tb[kGateInv + 4 * lane + k + 1] = 1.f / P;
    }
}

template <int D, int DV, int DK>
cudaError_t launch_dv(const FwdArgs &a) {
    constexpr bool DECAY = DK == 1;
    using Lay = Layout<D, DV, DK>;
    CUtensorMap qm, km, vm;
    const int BH = a.BH();
    if (!encode_3d(&qm, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, kC,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&km, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, kC,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&vm, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, a.N, BH, 64, kC,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    TcParams p{};
    p.y = a.y;
    p.N = a.N;
    p.BH = BH;
    p.eps = a.eps;
    p.S_in = a.S_in;
    p.z_in = a.z_in;
    p.S_out = a.S_out;
    p.z_out = a.z_out;
    choose_segments(BH, a.N, p.nseg, p.seg_chunks);
    // the segment states: after the header, or with gates after their tables
    size_t split_base = sizeof(WsHeader);
    if (DK == 2) {
        p.gate_blocks = (a.N + kC - 1) / kC;
        p.gate_tab = reinterpret_cast<const float *>(static_cast<const char *>(a.ws) +
                                                     gated_tables_offset(BH));
        p.gate_skip = reinterpret_cast<const unsigned int *>(static_cast<const char *>(a.ws) +
                                                             sizeof(WsHeader));
        split_base = gated_split_offset(BH, a.N);
    }
    if (DECAY) {
        p.gamma = a.gamma;
        p.H = a.H;
    }
    WsHeader *hdr = static_cast<WsHeader *>(a.ws);
    p.err = &hdr->error;
    p.err_where = &hdr->error_where;
    const long long lim = debug_fault().wait_limit_ns;
    p.limit_ns = lim > 0 ? (unsigned long long)lim : 1000000000ull;
    p.drop_item = debug_fault().drop_load_item;
    const int items = BH * p.nseg;
    if (p.nseg > 1) {
        // states of every segment but each head's last, then their exclusive
        // prefixes, which become the initial states of the (head, segment) items
        const size_t nS = (size_t)D * DV, cnt = (size_t)items;
        p.state_segs = p.nseg - 1;
        float *S_seg = reinterpret_cast<float *>(static_cast<char *>(a.ws) + split_base);
        float *z_seg = S_seg + cnt * nS;
        float *S_pre = z_seg + cnt * D;
        float *z_pre = S_pre + cnt * nS;
        if (DK == 2) p.seg_decay = z_pre + cnt * D;   // the segments' products of gates
        cudaError_t e;
        if (DK == 0 && D == 64) {
            // phase 1 of the fused non-causal kernel: one MMA per 16 tokens and
            // up to four K/V stages, which streams at the SM's share of HBM
            e = launch_segment_states_nc(a, p.nseg, p.seg_chunks, S_seg, z_seg);
        } else {
            using SL = StateLayout<D, DV, DK == 1>;
            auto skern = causal_state_kernel<D, DV, DK>;
            e = cudaFuncSetAttribute(skern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     SL::request);
            if (e != cudaSuccess) return e;
            skern<<<BH * p.state_segs, kStateThreads, SL::request, a.stream>>>(km, vm, p, S_seg,
                                                                                 z_seg);
            e = cudaGetLastError();
        }
        if (e != cudaSuccess) return e;
        const dim3 sgrid(BH, (D * DV + D + kScanThreads - 1) / kScanThreads);
        e = launch_overlapped(scan_states_kernel, sgrid, dim3(kScanThreads), 0, a.stream,
                              (const float *)S_seg, (const float *)z_seg, S_pre, z_pre, a.S_in,
                              a.z_in, p.nseg, D, DV, DECAY ? a.gamma : (const float *)nullptr,
                              a.H, p.seg_chunks * kC, (const float *)p.seg_decay);
        if (e != cudaSuccess) return e;
        p.S_in = S_pre;
        p.z_in = z_pre;
    }
    auto kern = causal_tc_kernel<D, DV, DK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::request);
    if (e != cudaSuccess) return e;
    if (p.nseg > 1)
        return launch_overlapped(kern, dim3(items), dim3(kThreads), Lay::request, a.stream, qm, km,
                                 vm, p);
    kern<<<items, kThreads, Lay::request, a.stream>>>(qm, km, vm, p);
    return cudaGetLastError();
}

}  // namespace

bool causal_tc_supported(const FwdArgs &a) {
    return a.dt == LA_DTYPE_BF16 && (a.d == 64 || a.d == 128) && (a.dv == 64 || a.dv == 128);
}

size_t causal_tc_workspace(int BH, int N, int d, int dv) { return segment_workspace(BH, N, d, dv); }

int causal_tc_launches(int BH, int N) {
    int nseg, seg_chunks;
    choose_segments(BH, N, nseg, seg_chunks);
    return nseg > 1 ? 3 : 1;
}

template <int DK>
cudaError_t launch_tc_dims(const FwdArgs &a) {
    if (a.d == 64 && a.dv == 64) return launch_dv<64, 64, DK>(a);
    if (a.d == 64 && a.dv == 128) return launch_dv<64, 128, DK>(a);
    if (a.d == 128 && a.dv == 64) return launch_dv<128, 64, DK>(a);
    if (a.d == 128 && a.dv == 128) return launch_dv<128, 128, DK>(a);
    return cudaErrorInvalidValue;
}

cudaError_t launch_causal_tc(const FwdArgs &a) {
    return a.gamma ? launch_tc_dims<1>(a) : launch_tc_dims<0>(a);
}

bool gated_tc_supported(const FwdArgs &a) {
    return causal_tc_supported(a) && a.gate != nullptr && a.gate_dim == 1 && a.phi == LA_PHI_ELU1;
}

size_t gated_tables_offset(int BH) {
    return sizeof(WsHeader) + ((size_t)BH * sizeof(unsigned int) + 255) / 256 * 256;
}

size_t gated_split_offset(int BH, int N) {
    const size_t nb = (size_t)(N + kC - 1) / kC;
    return (gated_tables_offset(BH) + sizeof(float) * (size_t)BH * nb * kGateTab + 255) / 256 * 256;
}

// header | flags | tables | (sequence split: S_seg, z_seg, S_pre, z_pre, the
// segments' products of gates)
size_t gated_tc_workspace(int BH, int N, int d, int dv) {
    int nseg, seg_chunks;
    choose_segments(BH, N, nseg, seg_chunks);
    size_t bytes = gated_split_offset(BH, N);
    if (nseg > 1)
        bytes += sizeof(float) * (size_t)BH * nseg * (2 * ((size_t)d * dv + d) + 1);
    return bytes;
}

size_t gated_tc_clear_bytes(int BH) { return gated_tables_offset(BH); }

cudaError_t launch_gated_tc(const FwdArgs &a) {
    const int BH = a.BH(), nb = (a.N + kC - 1) / kC;
    char *ws = static_cast<char *>(a.ws);
    gate_tables_kernel<<<dim3((nb + kGateWarps - 1) / kGateWarps, BH), kGateWarps * 32, 0,
                         a.stream>>>(a.gate, a.N, nb,
                                     reinterpret_cast<float *>(ws + gated_tables_offset(BH)),
                                     reinterpret_cast<unsigned int *>(ws + sizeof(WsHeader)));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_tc_dims<2>(a);
}

}  // namespace la

#ifdef LA_TRACE
extern "C" LA_API void la_trace_fetch(unsigned long long *dst) {
    cudaDeviceSynchronize();
    cudaMemcpyFromSymbol(dst, la_trace_buf, sizeof(unsigned long long) * 256 * 32);
}
#endif
