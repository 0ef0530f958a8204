// noncausal_tc.cu -- non-causal elu(x)+1 linear attention on the sm_103a
// tensor cores (tcgen05 MMA, TMEM accumulators, TMA tiles, mbarriers), one
// fused kernel.
//
// Method ("Linear Attention/es", "Reformulación con núcleos"): the sums
//   S = sum_j phi(k_j) v_j^T  [d x dv],   z = sum_j phi(k_j)  [d]
// do not depend on the query, so they are formed once per head and every
// query reads them: y_i = phi(q_i)^T S / max(phi(q_i)^T z, eps).
//
// One launch.  A work item is a (head, range of 128-token blocks); the items
// of a head first reduce their ranges of K and V, then meet, then each forms
// the head's whole state and evaluates its own range of queries:
//   phase 1  partial S_r, z_r of the range on the tensor cores, in the split
//            form of tc_state.cuh (S = 1 u^T + R, z = n 1 + zeta, per-key split
//            constants c'), written to the workspace;
//   meet     each item publishes its partial (a per-head counter, release),
//            then waits for all of the head's partials (acquire, bounded in
//            time);
//   image    S = sum_r S_r and z = sum_r z_r in range order (every item adds
//            in the same order, so the result does not depend on scheduling),
//            written into shared memory as the MMA operand image: S_hi, S_lo
//            (bf16 pairs in the 128-byte-swizzled MN-major layout), z_hi, z_lo,
//            with colsum(S) and sum z kept in fp32; item 0 of the head writes
//            the optional S_out, z_out;
//   phase 2  per 128-query block: A = psi_c(Q) (the residual features
//            phi(q) - c_i, in place over the TMA tile), Y = A S_hi + A S_lo,
//            den = A [z_hi | z_lo] in TMEM (with dv = 64 as one N = 192 MMA per
//            16 features: the MMAs' instruction count bounds these short
//            phases), and the epilogue
//            y_i = (c_i colsum(S) + Y_i) / max(c_i sum z + den_i, eps),
//            using phi(q_i) = c_i 1 + a_i.
// With more than one range per head the items wait for one another, so the
// launch is cooperative (every item resident at once); with one range per
// head nothing waits.  In its state-only mode the kernel runs phase 1 alone:
// the causal path's sequence split uses it for the states of its segments
// (d = 64, no decay), each (head, segment) item exporting its own sums.
//
// Precision: the residual features enter the tensor cores as bf16 (the same
// features c + bf16(phi(x) - c) as the causal path, split_const in
// tc_common.cuh); S and z are fp32 sums split into bf16 hi + lo pairs, so the
// rounding of the state costs about 2^-17 of its value; colsum(S) and sum z
// are fp32.  Outputs are float32.
//
// Warp roles (448 threads):
//   warp 0      TMA producer: K, V (phase 1, 2 to 4 stages), Q (phase 2, 3 or
//               6 stages)
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2..9  phase 1: psi_c(k) in place, two threads per key row (half of
//               its features each); warps 2..5 export the partial state
//   warps 2..5  phase 2: psi_c(q) in place, one query row per thread
//   warps 6..13 phase 2: normaliser epilogue (thread = TMEM lane) in two groups
//               that take alternate blocks, each row's split constant taken
//               from its first eight features in global memory (the tile has
//               been overwritten by then)
// One warp per scheduler leaves the epilogue latency-bound; two groups on
// alternate blocks double its throughput.
// Shared memory holds the phase-1 and phase-2 buffers in one region (they are
// never live together).  Every wait is bounded in time; a wait that runs out
// records LA_ERR_TIMEOUT in the workspace header and the item unwinds.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "la_internal.h"
#include "tc_common.cuh"
#include "tc_state.cuh"

namespace la {
namespace {

constexpr int kFThreads = 448;
constexpr int kFWarpB = 6;       // first epilogue warp (two groups of four warps)
constexpr int kFWorkEnd = 10;    // phase-1 row workers: warps 2..9
constexpr int kMaxS1 = 4;        // phase-1 stages at most
constexpr int kMaxQS = 6;        // Q stages at most
constexpr int kImgThreads = 256; // threads that form S (a multiple of dv)
constexpr int kZThreads = 64;    // threads that form z (threads 256..319)
constexpr int kBarE1 = 3;        // named barrier of the second epilogue group

// Operand image of one head in shared memory:
//   [hi]   S_hi: dv/64 boxes of [d rows][64 columns] bf16, 128-byte swizzle
//   [lo]   S_lo = bf16(S - S_hi), same layout
//   dv = 64 ("merged"): [zb] one more box of the same layout, column 0 = z_hi,
//          column 1 = z_lo, the rest 0, so [S_hi | S_lo | zb] is one N = 192
//          operand and one MMA per 16 features forms both halves of Y and of
//          the denominator;
//   dv = 128: [zt] [16 x d] bf16, K-major, no swizzle: row 0 = z_hi, row 1 = z_lo,
//          rest 0, a separate N = 16 operand.
template <int D, int DV>
struct OpImage {
    static constexpr bool kMerged = DV == 64;
    static constexpr int kHi = 0;
    static constexpr int kLo = D * DV * 2;
    static constexpr int kZt = 2 * D * DV * 2;   // zb (merged) or zt
    static constexpr int bytes = kMerged ? kZt + D * 128 : kZt + 16 * D * 2;
    static_assert(kZt % 1024 == 0, "swizzle alignment");
};

// Byte offset of element (k, n) in the [16 x D] no-swizzle K-major operand.
__host__ __device__ __forceinline__ uint32_t ztile_off(int n, int k, int D) {
    return (uint32_t)((n >> 3) * (D * 16) + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2);
}

struct FSmall {
    alignas(16) float colsum[128];           // colsum(S), fp32
    alignas(16) float cpart[4][128];         // partial column sums while they are formed
    alignas(16) float u[128];                // phase 1: u of the partial state
    alignas(16) float e_inv[2][kC];          // per epilogue group: 1 / max(den, eps) per row
    alignas(16) float cq[2][kC];             // per epilogue group: split constant per row
    alignas(16) float n_part[4];
    alignas(16) float zpart[2];
    float zsum;
    uint64_t kv_full[kMaxS1], kv_empty[kMaxS1], phik_done[kMaxS1], init_done, st_done;
    uint64_t q_full[kMaxQS], q_empty[kMaxQS], psi_done[kMaxQS];
    uint64_t acc_full[2], acc_empty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(offsetof(FSmall, kv_full) % 8 == 0, "mbarriers need 8-byte alignment");

template <int D, int DV>
struct FLayout {
    static constexpr int kK = kC * D * 2, kV = kC * DV * 2, kOnes = 16 * kC * 2, kQ = kC * D * 2;
    // phase 1, d = 64 ("ext"): each K stage is the K box and an extension box
    // [C tokens x 64] whose first column holds the keys' split constants, so
    // the M = 128 operand is [psi_c(K)^T ; c'^T]; each V stage is the V boxes
    // and a ones box (first column 1), so N = dv + 64.  One MMA per 16 tokens
    // then accumulates R, zeta (the ones column), u (row 64) and n (row 64,
    // the ones column) together.
    // phase 1, d = 128: K, V (2 stages each), the [1|s] operands (2 stages),
    // a 16 KB pad that the padded M = 128 operand (dv = 64) may read; three
    // MMAs per 16 tokens (R, zeta and u).
    // With d = dv = 64 the V stages share one ones box: they lie below it in
    // reverse order, V stage s (s + 1) boxes below, and each stage's operand
    // descriptor takes that distance as the stride to its ones box.
    static constexpr bool kExt = D == 64;
    static constexpr bool kSharedOnes = kExt && DV == 64;
    static constexpr int kS1 = (D == 64 && DV == 64) ? 4 : ((D == 128 && DV == 64) ? 3 : 2);
    static constexpr int kKs = kExt ? 2 * kK : kK;                         // K stage stride
    static constexpr int kVs = (kExt && !kSharedOnes) ? kV + 16384 : kV;  // V stage stride
    static constexpr int oK = 0, oV = oK + kS1 * kKs, oOnesBox = oV + kS1 * kVs;
    static constexpr int oOnes = oOnesBox + (kSharedOnes ? 16384 : 0), oPad = oOnes + kS1 * kOnes;
    static constexpr int p1 = kExt ? oOnes : oPad + 16384;
    __host__ __device__ static constexpr int v_stage(int s) {
        return kSharedOnes ? oV + (kS1 - 1 - s) * kV : oV + s * kVs;
    }
    __host__ __device__ static constexpr uint32_t v_lbo(int s) {   // stride between V's 64-column boxes
        return kSharedOnes ? (uint32_t)((s + 1) * kV) : (uint32_t)(kC * 128);
    }
    // phase 2: Q (kQS stages), the operand image
    static constexpr int kQS = D == 64 ? 6 : 3;
    static constexpr int oQ = 0, oOp = kQS * kQ;
    static constexpr int p2 = oOp + OpImage<D, DV>::bytes;
    static constexpr int oSmall = ((p1 > p2 ? p1 : p2) + 1023) / 1024 * 1024;
    static constexpr int bytes = oSmall + (int)sizeof(FSmall);
    static constexpr int request = bytes + 1024;
    // TMEM: phase 1 R [0, dv), zeta [128, 144), u [144, 160); phase 2 two
    // accumulators of kYCols columns: merged [Y_hi | Y_lo | den_hi, den_lo ...],
    // else Y_0, Y_1 [0, 2 dv) and the denominators [2 dv, 2 dv + 32)
    static constexpr bool kMerged = OpImage<D, DV>::kMerged;
    static constexpr uint32_t kYCols = kMerged ? 192 : DV;
    static constexpr uint32_t colDen = kMerged ? 128 : 2 * DV;   // merged: within each accumulator
    static constexpr uint32_t tmem_cols = kMerged ? 512 : ((2 * DV + 32 <= 256) ? 256 : 512);
    // two CTAs per SM when both TMEM and shared memory allow it
    static constexpr int min_blocks = (tmem_cols <= 256 && request <= 113 * 1024) ? 2 : 1;
    static_assert(oOp % 1024 == 0 && oOnes % 1024 == 0, "swizzled operands need 1024-byte alignment");
    static_assert(kS1 <= kMaxS1 && kQS <= kMaxQS, "stage counts");
    static_assert(request <= 232448, "shared memory per CTA");
};

struct FParams {
    float *y;
    const __nv_bfloat16 *q;        // the queries themselves (split constants of the epilogue)
    int N;
    int nranges;                   // ranges per head (work items = heads * nranges)
    int range_chunks;              // 128-token blocks per range (the last one may be shorter)
    float eps;
    float *S_part, *z_part;        // workspace: [BH][nranges][d][dv], [BH][nranges][d]
    int slot_stride;               // item (head, range) exports to slot head * slot_stride + range
    int state_only;                // 1: phase 1 and its export only (the causal path's segment states)
    unsigned int *counters;        // workspace: [BH] partials published (zero at the call's start)
    float *S_out, *z_out;
    unsigned int *err;
    unsigned int *err_where;
    unsigned long long limit_ns;
    int drop_item;                 // test hook: this item's first Q copy is never issued (-1: off)
};

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_gpu_add(unsigned int *p, unsigned int v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <int D, int DV>
__global__ void __launch_bounds__(kFThreads, FLayout<D, DV>::min_blocks)
noncausal_fused_kernel(const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const FParams p)
{
    using Lay = FLayout<D, DV>;
    using Img = OpImage<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    FSmall &S = *reinterpret_cast<FSmall *>(sm + Lay::oSmall);
    uint8_t *sK = sm + Lay::oK, *sV = sm + Lay::oV, *sOnes = sm + Lay::oOnes;
    uint8_t *sQ = sm + Lay::oQ, *sOp = sm + Lay::oOp;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int item = blockIdx.x;
    const int head = item / p.nranges, rng = item - head * p.nranges;
    const int tok0 = rng * p.range_chunks * kC;
    const int nloc = min(p.N - tok0, p.range_chunks * kC);
    const int nchunks = (nloc + kC - 1) / kC;
    const Guard g{&S.abort_flag, p.err, p.err_where, p.limit_ns};
    // segment states: the item reads only K and V, and the prefix scan that
    // consumes them waits for this whole grid, so it may be scheduled now
    if (p.state_only) griddep_launch_dependents();

    if (tid == 0) {
        S.abort_flag = 0;
        for (int s = 0; s < Lay::kS1; ++s) {
            mbar_init(&S.kv_full[s], 1);
            mbar_init(&S.kv_empty[s], 1);
            mbar_init(&S.phik_done[s], kWG);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&S.acc_full[s], 1);
            mbar_init(&S.acc_empty[s], kWG);
        }
        mbar_init(&S.init_done, kWG);
        mbar_init(&S.st_done, 1);
        for (int s = 0; s < Lay::kQS; ++s) {
            mbar_init(&S.q_full[s], 1);
            mbar_init(&S.q_empty[s], 1);
            mbar_init(&S.psi_done[s], kWG);
        }
        mbar_init(&S.drain, 1);
        fence_mbar_init();
        prefetch_tmap(&qmap);
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
    }
    if (warp == 1) {
        tmem_alloc(&S.tmem_base, Lay::tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem_base;

    // ======================================================== phase 1: partial state
    if (warp == 0) {
        if (lane == 0) {   // K and V blocks of this range
            constexpr uint32_t kvbytes = kC * (D + DV) * 2;
            int last_kv[kMaxS1] = {-1, -1, -1, -1};
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % Lay::kS1, t0 = tok0 + c * kC;
                if (c >= Lay::kS1 && !mbar_wait(&S.kv_empty[s], ((c / Lay::kS1) - 1) & 1, g, 80)) break;
                mbar_arrive_expect_tx(&S.kv_full[s], kvbytes);
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load_3d(sK + s * Lay::kKs + bx * kC * 128, &kmap, &S.kv_full[s], bx * 64, t0, head);
                for (int bx = 0; bx < DV / 64; ++bx)
                    tma_load_3d(sm + Lay::v_stage(s) + bx * kC * 128, &vmap, &S.kv_full[s], bx * 64, t0, head);
                last_kv[s] = c;
            }
            if (*g.abort)
                for (int s = 0; s < Lay::kS1; ++s)
                    if (last_kv[s] >= 0)
                        drain_wait(&S.kv_full[s], (last_kv[s] / Lay::kS1) & 1, g.limit_ns);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // R += B^T V, zeta += B^T 1, u += V^T s
            constexpr uint32_t iR = idesc_bf16(128, DV, 1, 1);
            constexpr uint32_t iZ = idesc_bf16(128, 16, 1, 0);
            bool ok = mbar_wait(&S.init_done, 0, g, 81);
            for (int c = 0; ok && c < nchunks; ++c) {
                const int s = c % Lay::kS1;
                if (!mbar_wait(&S.kv_full[s], (c / Lay::kS1) & 1, g, 82)) break;
                if (!mbar_wait(&S.phik_done[s], (c / Lay::kS1) & 1, g, 83)) break;
                tc_fence_after();
                const uint32_t kb = smem_u32(sK + s * Lay::kKs), vb = smem_u32(sm + Lay::v_stage(s));
                const uint32_t vlbo = Lay::v_lbo(s);
                const uint32_t ob = smem_u32(sOnes + s * Lay::kOnes);
                constexpr uint32_t iE = idesc_bf16(128, DV + 64, 1, 1);   // ext: [R | zeta ...]
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks) {
                    const uint64_t ad = smem_desc(kb + ks * 2048, kC * 128, 1024, kSwizzle128B);
                    const uint64_t vd = smem_desc(vb + ks * 2048, vlbo, 1024, kSwizzle128B);
                    if (Lay::kExt) {
                        mma_ss(tb + kStColR, ad, vd, iE, 1);
                    } else {
                        const uint64_t od = smem_desc(ob + ks * 256, 128, 2048, kSwizzleNone);
                        mma_ss(tb + kStColR, ad, vd, iR, 1);
                        mma_ss(tb + kStColZ, ad, od, iZ, 1);
                        mma_ss(tb + kStColU, vd, od, iZ, 1);
                    }
                }
                mma_commit(&S.kv_empty[s]);
            }
            mma_commit(&S.st_done);
            drain_wait(&S.st_done, 0, g.limit_ns);
        }
    } else if (warp < kFWorkEnd) {
        // warps 2..9: two threads per key row, each with half of its features
        // (h = 0: warps 2..5, h = 1: warps 6..9); warp w's TMEM lane quarter
        // is w & 3, the quarter of its rows
        const int wq = warp & 3, row = wq * 32 + lane, h = (warp - 2) >> 2;
        const int wtid = tid - 64;   // 0..255
        const uint32_t lb = (uint32_t)(wq * 32) << 16;
        if (Lay::kExt) {
            // extension boxes zero (their first column is rewritten per block);
            // ones boxes: first column 1, rest 0
            for (int e = wtid; e < Lay::kS1 * kC * 8; e += 2 * kWG) {
                const int st = e / (kC * 8), r = (e / 8) % kC, ch = e % 8;
                *reinterpret_cast<uint4 *>(sK + st * Lay::kKs + Lay::kK + sw128_off(r, ch * 8)) =
                    make_uint4(0u, 0u, 0u, 0u);
                if (!Lay::kSharedOnes || st == 0)
                    *reinterpret_cast<uint4 *>(sm + Lay::v_stage(st) + Lay::v_lbo(st) * (DV / 64) +
                                               sw128_off(r, ch * 8)) =
                        ch == 0 ? make_uint4(pack_bf16x2(1.f, 0.f), 0u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
            }
        } else {
            // [1|s] operands: row 0 = ones, rows 1, 2 rewritten per block, rest 0;
            // a zeroed pad region
            for (int e = wtid; e < Lay::kS1 * 16 * kC; e += 2 * kWG) {
                const int st = e / (16 * kC), n = (e / kC) % 16, k = e % kC;
                *reinterpret_cast<__nv_bfloat16 *>(sOnes + st * Lay::kOnes + (n >> 3) * 2048 +
                                                   (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2) =
                    __float2bfloat16_rn(n == 0 ? 1.f : 0.f);
            }
            for (int e = wtid; e < 16384 / 16; e += 2 * kWG)
                reinterpret_cast<uint4 *>(sm + Lay::oPad)[e] = make_uint4(0u, 0u, 0u, 0u);
        }
        if (h == 0) {   // zero accumulators
            uint32_t zero[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) zero[m] = 0u;
            if (Lay::kExt) {
#pragma unroll
                for (int grp = 0; grp < DV / 16 + 4; ++grp)
                    tmem_st16(tb + lb + kStColR + grp * 16, zero);
            } else {
#pragma unroll
                for (int grp = 0; grp < DV / 16; ++grp) tmem_st16(tb + lb + kStColR + grp * 16, zero);
                tmem_st16(tb + lb + kStColZ, zero);
                tmem_st16(tb + lb + kStColU, zero);
            }
            tmem_wait_st();
        }
        fence_proxy_async();
        tc_fence_before();
        named_bar(kBarB, 2 * kWG);   // both halves' operand writes are done
        if (h == 0) mbar_arrive(&S.init_done);
        bool ok = true;
        float nrow = 0.f;   // this key row's share of n (h = 0)
        for (int c = 0; c < nchunks; ++c) {
            const int s = c % Lay::kS1;
            const int L = min(kC, nloc - c * kC);
            ok = wait_warp(&S.kv_full[s], (c / Lay::kS1) & 1, g, 84);
            uint8_t *kt = sK + s * Lay::kKs;
            // the key's split constant from its first eight features (in h = 0's
            // half): both halves read them; h = 0 writes their residuals back
            // only after the group barrier below, once h = 1 has read them
            uint4 first = make_uint4(0u, 0u, 0u, 0u);
            if (ok) first = *reinterpret_cast<const uint4 *>(kt + sw128_off(row, 0));
            const float ck = split_const(first);
            const SplitC kk = split_pairs(ck);
            uint4 held = make_uint4(0u, 0u, 0u, 0u);
            if (ok) {
                constexpr int kChunks = D / 16;   // 8-feature chunks per half
                const int f0 = h * kChunks;
                uint4 raw[kChunks];
#pragma unroll
                for (int f = 0; f < kChunks; ++f)
                    raw[f] = *reinterpret_cast<const uint4 *>(
                        kt + ((f0 + f) >> 3) * (kC * 128) + sw128_off(row, ((f0 + f) & 7) * 8));
#pragma unroll
                for (int f = 0; f < kChunks; ++f) {
                    uint32_t w[4] = {raw[f].x, raw[f].y, raw[f].z, raw[f].w};
#pragma unroll
                    for (int hw = 0; hw < 4; ++hw) w[hw] = feat_bf16x2(w[hw], kk);
                    raw[f] = make_uint4(w[0], w[1], w[2], w[3]);
                }
#pragma unroll
                for (int f = 0; f < kChunks; ++f) {
                    if (f0 + f == 0)
                        held = raw[f];
                    else
                        *reinterpret_cast<uint4 *>(kt + ((f0 + f) >> 3) * (kC * 128) +
                                                   sw128_off(row, ((f0 + f) & 7) * 8)) = raw[f];
                }
                fence_proxy_async();
            }
            if (group_any<kBarB, 2 * kWG>(!ok)) { ok = false; break; }
            if (h == 0) {
                *reinterpret_cast<uint4 *>(kt + sw128_off(row, 0)) = held;
                // the key's constant (a bf16 value; 0 on padding rows): ext, the
                // first column of the extension box (u, n from row 64 of the
                // accumulator); else rows 1, 2 of the [1|s] operand (u += V^T c')
                const float cj = row < L ? ck : 0.f;
                if (Lay::kExt) {
                    *reinterpret_cast<uint4 *>(kt + Lay::kK + sw128_off(row, 0)) =
                        make_uint4(pack_bf16x2(cj, 0.f), 0u, 0u, 0u);
                } else {
                    uint8_t *op = sOnes + s * Lay::kOnes + (row >> 3) * 128 + (row & 7) * 2;
                    *reinterpret_cast<__nv_bfloat16 *>(op + 16) = __float2bfloat16_rn(cj);
                    *reinterpret_cast<__nv_bfloat16 *>(op + 32) = __float2bfloat16_rn(0.f);
                }
                nrow += cj;
                fence_proxy_async();
                mbar_arrive(&S.phik_done[s]);
            }
        }
        if (h == 0) {
            ok = ok && wait_warp(&S.st_done, 0, g, 85);
            if (ok) {   // partial state of the range: S = 1 u^T + R, z = n 1 + zeta
                tc_fence_after();
                uint32_t zv[4], uv[4];
                if (Lay::kExt) {
                    // zeta in the ones column; row 64 holds u (and n in the ones column)
                    tmem_ld4(tb + lb + kStColR + DV, zv);
                    tmem_wait_ld();
                    if (wq == 2) {   // the warp of lanes 64..95 (TMEM loads are warp-wide)
#pragma unroll 1
                        for (int grp = 0; grp < DV / 16; ++grp) {
                            uint32_t rv[16];
                            tmem_ld16(tb + lb + kStColR + grp * 16, rv);
                            tmem_wait_ld();
                            if (lane == 0)
#pragma unroll
                                for (int m = 0; m < 16; ++m) S.u[grp * 16 + m] = u2f(rv[m]);
                        }
                        if (lane == 0) {
                            S.n_part[0] = u2f(zv[0]);
                            S.n_part[1] = S.n_part[2] = S.n_part[3] = 0.f;
                        }
                    }
                } else {
                    tmem_ld4(tb + lb + kStColZ, zv);
                    tmem_ld4(tb + lb + kStColU, uv);
                    tmem_wait_ld();
                    S.u[row] = u2f(uv[1]) + u2f(uv[2]);
                    const float ns = warp_sum_f(nrow);
                    if (lane == 0) S.n_part[wq] = ns;
                }
                named_bar(kBarA, kWG);
                const size_t slot = (size_t)head * p.slot_stride + rng;
                float *dst = p.S_part + slot * D * DV;
#pragma unroll 1
                for (int grp = 0; grp < DV / 16; ++grp) {
                    uint32_t rv[16];
                    tmem_ld16(tb + lb + kStColR + grp * 16, rv);
                    tmem_wait_ld();
                    if (row < D)
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 4)
                            *reinterpret_cast<float4 *>(dst + (size_t)row * DV + grp * 16 + jj) =
                                make_float4(u2f(rv[jj]) + S.u[grp * 16 + jj],
                                            u2f(rv[jj + 1]) + S.u[grp * 16 + jj + 1],
                                            u2f(rv[jj + 2]) + S.u[grp * 16 + jj + 2],
                                            u2f(rv[jj + 3]) + S.u[grp * 16 + jj + 3]);
                }
                const float n = (S.n_part[0] + S.n_part[1]) + (S.n_part[2] + S.n_part[3]);
                if (row < D) p.z_part[slot * D + row] = u2f(zv[0]) + n;
                __threadfence();   // the partial is visible GPU-wide before it is published
            }
        }
    }
    tc_fence_before();
    __syncthreads();   // phase 1 is over in this item; its TMEM columns are free again
    tc_fence_after();
    // the first Q tiles fly in while the items meet and the image is formed
    // (the Q stages lie below the image in shared memory)
    static_assert(Lay::oQ + Lay::kQS * Lay::kQ <= Lay::oOp, "Q stages below the image");
    const bool drop = item == p.drop_item;   // test hook: block 0 never arrives
    int c_last = -1;                          // producer: last block whose copy was issued
    auto load_q = [&](int c) {
        const int s = c % Lay::kQS;
        mbar_arrive_expect_tx(&S.q_full[s], kC * D * 2);
        if (c == 0 && drop) return;
        for (int bx = 0; bx < D / 64; ++bx)
            tma_load_3d(sQ + s * Lay::kQ + bx * kC * 128, &qmap, &S.q_full[s], bx * 64,
                        tok0 + c * kC, head);
        c_last = c;
    };
    // The item publishes its partial before it issues the Q copies: a release
    // waits for the thread's earlier memory operations, copies included.
    const bool so = p.state_only != 0;   // the item ends with its exported partial
    const bool meet = !so && !S.abort_flag && p.nranges > 1;
    if (meet && tid == 0) red_release_gpu_add(&p.counters[head], 1u);
    if (!so && !S.abort_flag && warp == 0 && lane == 0)
        for (int c = 0; c < min(nchunks, Lay::kQS); ++c) load_q(c);

    // ======================================================== meet
    if (meet) {
        if (tid == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(&p.counters[head]) < (unsigned)p.nranges) {
                if (globaltimer_ns() - t0 > g.limit_ns) {
                    guard_fail(g, 4u /* LA_ERR_TIMEOUT */, 86);
                    break;
                }
                __nanosleep(256);
            }
        }
        __syncthreads();
    }

    // ======================================================== image of the head's state
    const bool run2 = !so && !S.abort_flag;
    if (run2) {
        if (tid < kImgThreads) {   // S: thread t keeps column t % dv, rows t / dv + k (256 / dv)
            constexpr int kRowStep = kImgThreads / DV;
            constexpr int kPer = D / kRowStep;   // rows per thread
            constexpr int kBatch = kPer < 16 ? kPer : 16;
            const int b = tid % DV, j0 = tid / DV;
            const float *src = p.S_part + (size_t)head * p.nranges * D * DV + (size_t)j0 * DV + b;
            float cs = 0.f;
#pragma unroll 1
            for (int i0 = 0; i0 < kPer; i0 += kBatch) {
                // every partial's rows of this batch are in flight together
                float acc[kBatch];
#pragma unroll
                for (int i = 0; i < kBatch; ++i) acc[i] = 0.f;
#pragma unroll 2
                for (int r = 0; r < p.nranges; ++r) {
                    float x[kBatch];
#pragma unroll
                    for (int i = 0; i < kBatch; ++i)
                        x[i] = __ldcg(src + (size_t)r * D * DV + (size_t)(i0 + i) * kRowStep * DV);
#pragma unroll
                    for (int i = 0; i < kBatch; ++i) acc[i] += x[i];
                }
#pragma unroll
                for (int i = 0; i < kBatch; ++i) {
                    const int a = j0 + (i0 + i) * kRowStep;
                    const float v = acc[i];
                    if (rng == 0 && p.S_out) p.S_out[((size_t)head * D + a) * DV + b] = v;
                    const float vh = bf16_round(v);
                    const uint32_t off = (uint32_t)(b >> 6) * (D * 128) + sw128_off(a, b & 63);
                    *reinterpret_cast<__nv_bfloat16 *>(sOp + Img::kHi + off) = __float2bfloat16_rn(vh);
                    *reinterpret_cast<__nv_bfloat16 *>(sOp + Img::kLo + off) =
                        __float2bfloat16_rn(v - vh);
                    cs += v;
                }
            }
            S.cpart[j0][b] = cs;
            named_bar(kBarB, kImgThreads);
            if (tid < DV) {   // the column's partial sums in a fixed order
                float t = 0.f;
#pragma unroll
                for (int j = 0; j < kRowStep; ++j) t += S.cpart[j][b];
                S.colsum[b] = t;
            }
        } else if (tid < kImgThreads + kZThreads) {   // z (threads 256..319)
            const int t = tid - kImgThreads;
            const float *src = p.z_part + (size_t)head * p.nranges * D;
            float zs = 0.f;
            for (int a = t; a < D; a += kZThreads) {
                float zv = 0.f;
                for (int r = 0; r < p.nranges; ++r) zv += __ldcg(src + (size_t)r * D + a);
                if (rng == 0 && p.z_out) p.z_out[(size_t)head * D + a] = zv;
                const float zh = bf16_round(zv);
                if (Img::kMerged) {   // row a of zb: [z_hi, z_lo, 0 ...]
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        *reinterpret_cast<uint4 *>(sOp + Img::kZt + sw128_off(a, ch * 8)) =
                            ch == 0 ? make_uint4(pack_bf16x2(zh, zv - zh), 0u, 0u, 0u)
                                    : make_uint4(0u, 0u, 0u, 0u);
                } else {
#pragma unroll
                    for (int n = 0; n < 16; ++n)
                        *reinterpret_cast<__nv_bfloat16 *>(sOp + Img::kZt + ztile_off(n, a, D)) =
                            __float2bfloat16_rn(n == 0 ? zh : (n == 1 ? zv - zh : 0.f));
                }
                zs += zv;
            }
            zs = warp_sum_f(zs);   // fixed butterfly order: deterministic
            if (lane == 0) S.zpart[t >> 5] = zs;
            named_bar(kBarA, kZThreads);
            if (t == 0) S.zsum = S.zpart[0] + S.zpart[1];
        }
        fence_proxy_async();   // the image is read by the MMAs (async proxy)
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ======================================================== phase 2: the queries
    if (run2) {
        if (warp == 0) {
            if (lane == 0) {   // the rest of the Q tiles of this range
                for (int c = Lay::kQS; c < nchunks; ++c) {
                    if (!mbar_wait(&S.q_empty[c % Lay::kQS], ((c / Lay::kQS) - 1) & 1, g, 90))
                        break;
                    load_q(c);
                }
            }
        } else if (warp == 1) {
            if (lane == 0) {   // Y_b = A (S_hi + S_lo), den_b = A [z_hi | z_lo]
                constexpr uint32_t iY = idesc_bf16(128, DV, 0, 1);   // A K-major, B MN-major
                constexpr uint32_t iZ = idesc_bf16(128, 16, 0, 0);   // A K-major, B K-major
                const uint32_t hb = smem_u32(sOp + Img::kHi), lb2 = smem_u32(sOp + Img::kLo);
                const uint32_t zb = smem_u32(sOp + Img::kZt);
                constexpr uint32_t iM = idesc_bf16(128, 192, 0, 1);   // merged: [S_hi | S_lo | zb]
                for (int c = 0; c < nchunks; ++c) {
                    const int s = c % Lay::kQS, b = c & 1;
                    if (!mbar_wait(&S.psi_done[s], (c / Lay::kQS) & 1, g, 91)) break;
                    if (c >= 2 && !mbar_wait(&S.acc_empty[b], ((c >> 1) - 1) & 1, g, 92)) break;
                    tc_fence_after();
                    const uint32_t qb = smem_u32(sQ + s * FLayout<D, DV>::kQ);
                    const uint32_t dY = tb + (uint32_t)(b * Lay::kYCols), dZ = tb + Lay::colDen + 16u * b;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint64_t ad = smem_desc(qb + (ks >> 2) * (kC * 128) + (ks & 3) * 32,
                                                      16, 1024, kSwizzle128B);
                        const uint64_t hd = smem_desc(hb + ks * 2048, D * 128, 1024, kSwizzle128B);
                        if (Lay::kMerged) {
                            mma_ss(dY, ad, hd, iM, ks > 0);
                        } else {
                            const uint64_t ld = smem_desc(lb2 + ks * 2048, D * 128, 1024, kSwizzle128B);
                            const uint64_t zd = smem_desc(zb + ks * 256, 128, D * 16, kSwizzleNone);
                            mma_ss(dY, ad, hd, iY, ks > 0);
                            mma_ss(dY, ad, ld, iY, 1);
                            mma_ss(dZ, ad, zd, iZ, ks > 0);
                        }
                    }
                    mma_commit(&S.q_empty[s]);
                    mma_commit(&S.acc_full[b]);
                }
            }
        } else if (warp < kFWarpB) {
            // psi_c(q) in place (bf16) over the swizzled Q tile, one row per thread
            const int row = (warp & 3) * 32 + lane;
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % Lay::kQS;
                const bool ok = wait_warp(&S.q_full[s], (c / Lay::kQS) & 1, g, 94);
                if (ok) {
                    uint8_t *qt = sQ + s * FLayout<D, DV>::kQ;
                    // the query's split constant, read before the row is overwritten
                    const SplitC kq = split_pairs(
                        split_const(*reinterpret_cast<const uint4 *>(qt + sw128_off(row, 0))));
#pragma unroll 1
                    for (int f0 = 0; f0 < D / 8; f0 += 8) {
                        uint4 raw[8];
#pragma unroll
                        for (int f = 0; f < 8; ++f)
                            raw[f] = *reinterpret_cast<const uint4 *>(
                                qt + ((f0 + f) >> 3) * (kC * 128) + sw128_off(row, ((f0 + f) & 7) * 8));
#pragma unroll
                        for (int f = 0; f < 8; ++f) {
                            uint32_t w[4] = {raw[f].x, raw[f].y, raw[f].z, raw[f].w};
#pragma unroll
                            for (int h = 0; h < 4; ++h) w[h] = feat_bf16x2(w[h], kq);
                            raw[f] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
#pragma unroll
                        for (int f = 0; f < 8; ++f)
                            *reinterpret_cast<uint4 *>(qt + ((f0 + f) >> 3) * (kC * 128) +
                                                       sw128_off(row, ((f0 + f) & 7) * 8)) = raw[f];
                    }
                    fence_proxy_async();
                    mbar_arrive(&S.psi_done[s]);
                }
                if (group_any<kBarA>(!ok)) break;
            }
        } else {
            // normaliser epilogue per block
            const int wq = warp & 3, row = wq * 32 + lane;
            const float zsum = S.zsum;
            const int tq = lane >> 2, tcol = (lane & 3) * 2;
            constexpr int kParts = 2 * (DV / 32);   // (16-lane half, 32-column block) pairs
            // two groups of four warps take alternate blocks: group e the blocks
            // c = e (mod 2), whose accumulator is b = e
            const int e = (warp - kFWarpB) >> 2;
            bool ok = true;
            for (int c = e; ok && c < nchunks; c += 2) {
                const int b = e;
                // this row's first eight features (rows past the range: c = 1),
                // loaded while the block's MMAs run
                uint4 first = make_uint4(0u, 0u, 0u, 0u);
                if (c * kC + row < nloc)
                    first = *reinterpret_cast<const uint4 *>(
                        p.q + ((size_t)head * p.N + tok0 + c * kC + row) * D);
                ok = wait_warp(&S.acc_full[b], (c >> 1) & 1, g, 96);
                if (ok) {
                    tc_fence_after();
                    uint32_t dz[4];
                    tmem_ld4(tb + ((uint32_t)(wq * 32) << 16) +
                                 (Lay::kMerged ? b * Lay::kYCols + Lay::colDen : Lay::colDen + 16u * b),
                             dz);
                    const float cr = split_const(first);
                    tmem_wait_ld();
                    __syncwarp();
                    S.cq[e][row] = cr;
                    S.e_inv[e][row] = 1.f / fmaxf(fmaf(cr, zsum, u2f(dz[0]) + u2f(dz[1])), p.eps);
                    __syncwarp();
                    const int t0 = c * kC;
                    float *ychunk = p.y + ((size_t)head * p.N + tok0 + t0) * DV;
                    auto part_addr = [&](int part) {
                        return tb + ((uint32_t)(wq * 32 + 16 * (part & 1)) << 16) +
                               (uint32_t)(b * Lay::kYCols) + (part >> 1) * 32;
                    };
                    // 16x256b shape: 4 neighbouring lanes hold 8 consecutive columns
                    // of one row, so each warp store covers whole 32-byte sectors
                    auto outputs = [&](int part, const uint32_t (&vc)[16]) {
                        const int half = part & 1, cblk = part >> 1;
                        const int rA = wq * 32 + 16 * half + tq, rB = rA + 8;
                        const uint64_t invA = f2pack(S.e_inv[e][rA], S.e_inv[e][rA]);
                        const uint64_t invB = f2pack(S.e_inv[e][rB], S.e_inv[e][rB]);
                        const uint64_t cA = f2pack(S.cq[e][rA], S.cq[e][rA]);
                        const uint64_t cB = f2pack(S.cq[e][rB], S.cq[e][rB]);
                        const bool okA = t0 + rA < nloc, okB = t0 + rB < nloc;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int col = cblk * 32 + 8 * k + tcol;
                            const uint64_t cs = *reinterpret_cast<const uint64_t *>(S.colsum + col);
                            float2 oA, oB;
                            f2unpack(f2mul(f2add(f2mul(cA, cs), f2pack(u2f(vc[4 * k]), u2f(vc[4 * k + 1]))),
                                           invA), oA.x, oA.y);
                            f2unpack(f2mul(f2add(f2mul(cB, cs), f2pack(u2f(vc[4 * k + 2]), u2f(vc[4 * k + 3]))),
                                           invB), oB.x, oB.y);
                            if (okA) *reinterpret_cast<float2 *>(ychunk + (size_t)rA * DV + col) = oA;
                            if (okB) *reinterpret_cast<float2 *>(ychunk + (size_t)rB * DV + col) = oB;
                        }
                    };
                    uint32_t vA[16], vB[16];
                    if (Lay::kMerged) {   // Y = Y_hi + Y_lo (the lo half 64 columns on)
#pragma unroll 1
                        for (int part = 0; part < kParts; ++part) {
                            tmem_ld_16x256b_x4(part_addr(part), vA);
                            tmem_ld_16x256b_x4(part_addr(part) + 64, vB);
                            tmem_wait_ld();
#pragma unroll
                            for (int m = 0; m < 16; ++m) vA[m] = f2u(u2f(vA[m]) + u2f(vB[m]));
                            outputs(part, vA);
                        }
                    } else {
                        tmem_ld_16x256b_x4(part_addr(0), vA);
                        tmem_wait_ld();
#pragma unroll 1
                        for (int part = 0; part < kParts; part += 2) {
                            tmem_ld_16x256b_x4(part_addr(part + 1), vB);   // kParts is even
                            outputs(part, vA);
                            tmem_wait_ld();
                            if (part + 2 < kParts) tmem_ld_16x256b_x4(part_addr(part + 2), vA);
                            outputs(part + 1, vB);
                            if (part + 2 < kParts) tmem_wait_ld();
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(&S.acc_empty[b]);
                }
                if (e == 0 ? group_any<kBarB>(!ok) : group_any<kBarE1>(!ok)) break;
            }
        }
        if (warp == 1 && lane == 0) {   // every MMA issued has completed once `drain` flips
            mma_commit(&S.drain);
            drain_wait(&S.drain, 0, g.limit_ns);
        }
    }
    if (warp == 0 && lane == 0 && *g.abort) {   // no copy may still be landing when the item exits
        for (int s = 0; s < Lay::kQS; ++s) {
            if (c_last < 0) break;
            const int c = c_last - ((c_last - s) % Lay::kQS + Lay::kQS) % Lay::kQS;
            if (c < 0 || (c == 0 && drop)) continue;
            drain_wait(&S.q_full[s], (c / Lay::kQS) & 1, g.limit_ns);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tb, Lay::tmem_cols);
    }
}

// ------------------------------------------------------------------ host side
// Items of the fused kernel that the current device holds at once (its SMs
// times the kernel's resident CTAs per SM), cached per device and size.
template <int D, int DV>
int fused_capacity() {
    constexpr int kMaxDev = 64;
    static int cache[kMaxDev];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) dev = -1;
    if (dev >= 0) {
        std::lock_guard<std::mutex> lock(mu);
        if (cache[dev] > 0) return cache[dev];
    }
    int nb = 0;
    using Lay = FLayout<D, DV>;
    auto kern = noncausal_fused_kernel<D, DV>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::request) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kFThreads, Lay::request) !=
            cudaSuccess ||
        nb < 1)
        nb = 1;
    const int cap = nb * num_sms();
    if (dev >= 0) {
        std::lock_guard<std::mutex> lock(mu);
        cache[dev] = cap;
    }
    return cap;
}

int capacity_for(int d, int dv) {
    if (d == 64 && dv == 64) return fused_capacity<64, 64>();
    if (d == 64 && dv == 128) return fused_capacity<64, 128>();
    if (d == 128 && dv == 64) return fused_capacity<128, 64>();
    return fused_capacity<128, 128>();
}

// Ranges per head: enough items to fill the GPU once, all resident together
// (a cooperative launch); one range per head when the heads alone fill it.
void nc_split(int BH, int N, int d, int dv, int &nranges, int &range_chunks) {
    const int nch = (N + kC - 1) / kC;
    const int cap = capacity_for(d, dv);
    int want = BH >= cap ? 1 : cap / BH;
    if (want > nch) want = nch;
    if (want < 1) want = 1;
    range_chunks = (nch + want - 1) / want;
    if (range_chunks < 1) range_chunks = 1;
    nranges = (nch + range_chunks - 1) / range_chunks;
    if (nranges < 1) nranges = 1;
}

// [header][counters: BH u32, padded to 256][S_part][z_part]
size_t counters_bytes(int BH) { return ((size_t)BH * 4 + 255) / 256 * 256; }

template <int D, int DV>
cudaError_t launch_fused(const FwdArgs &a) {
    using Lay = FLayout<D, DV>;
    const int BH = a.BH();
    CUtensorMap qm, km, vm;
    if (!encode_3d(&qm, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, kC,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&km, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, kC,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&vm, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, a.N, BH, 64, kC,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    WsHeader *hdr = static_cast<WsHeader *>(a.ws);
    const long long lim = debug_fault().wait_limit_ns;
    FParams p{};
    p.y = a.y;
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.N = a.N;
    p.eps = a.eps;
    nc_split(BH, a.N, D, DV, p.nranges, p.range_chunks);
    char *ws = static_cast<char *>(a.ws);
    p.counters = reinterpret_cast<unsigned int *>(ws + sizeof(WsHeader));
    p.S_part = reinterpret_cast<float *>(ws + sizeof(WsHeader) + counters_bytes(BH));
    p.z_part = p.S_part + (size_t)BH * p.nranges * D * DV;
    p.slot_stride = p.nranges;
    p.state_only = 0;
    p.S_out = a.S_out;
    p.z_out = a.z_out;
    p.err = &hdr->error;
    p.err_where = &hdr->error_where;
    p.limit_ns = lim > 0 ? (unsigned long long)lim : 1000000000ull;
    p.drop_item = debug_fault().drop_load_item;
    auto kern = noncausal_fused_kernel<D, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::request);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(BH * p.nranges);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = Lay::request;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // the items of a head wait for one another
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.nranges > 1 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, qm, km, vm, p);
}

}  // namespace

bool noncausal_tc_supported(const FwdArgs &a) {
    return a.dt == LA_DTYPE_BF16 && (a.d == 64 || a.d == 128) && (a.dv == 64 || a.dv == 128);
}

size_t noncausal_tc_workspace(int BH, int N, int d, int dv) {
    int nranges, range_chunks;
    nc_split(BH, N, d, dv, nranges, range_chunks);
    return sizeof(WsHeader) + counters_bytes(BH) +
           sizeof(float) * (size_t)BH * nranges * ((size_t)d * dv + d);
}

size_t noncausal_tc_clear_bytes(int BH) { return sizeof(WsHeader) + counters_bytes(BH); }

// The causal path's sequence split (d = 64, no decay): the states of every
// segment but each head's last, by phase 1 of the fused kernel alone.  Item
// (head, segment) reduces its segment's K and V and exports the plain state
// to slot head * nseg + segment of S_seg, z_seg; nothing waits across items.
template <int D, int DV>
cudaError_t launch_states(const FwdArgs &a, int nseg, int seg_chunks, float *S_seg, float *z_seg) {
    using Lay = FLayout<D, DV>;
    const int BH = a.BH();
    CUtensorMap qm, km, vm;
    if (!encode_3d(&qm, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, kC,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&km, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, D, a.N, BH, 64, kC,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_3d(&vm, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, DV, a.N, BH, 64, kC,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    WsHeader *hdr = static_cast<WsHeader *>(a.ws);
    const long long lim = debug_fault().wait_limit_ns;
    FParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.N = a.N;
    p.eps = a.eps;
    p.nranges = nseg - 1;
    p.range_chunks = seg_chunks;
    p.slot_stride = nseg;
    p.state_only = 1;
    p.S_part = S_seg;
    p.z_part = z_seg;
    p.err = &hdr->error;
    p.err_where = &hdr->error_where;
    p.limit_ns = lim > 0 ? (unsigned long long)lim : 1000000000ull;
    p.drop_item = -1;
    auto kern = noncausal_fused_kernel<D, DV>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::request);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    kern<<<BH * p.nranges, kFThreads, Lay::request, a.stream>>>(qm, km, vm, p);
    return cudaGetLastError();
}

cudaError_t launch_segment_states_nc(const FwdArgs &a, int nseg, int seg_chunks, float *S_seg,
                                     float *z_seg) {
    if (a.d == 64 && a.dv == 64) return launch_states<64, 64>(a, nseg, seg_chunks, S_seg, z_seg);
    if (a.d == 64 && a.dv == 128) return launch_states<64, 128>(a, nseg, seg_chunks, S_seg, z_seg);
    return cudaErrorInvalidValue;
}

cudaError_t launch_noncausal_tc(const FwdArgs &a) {
    if (a.d == 64 && a.dv == 64) return launch_fused<64, 64>(a);
    if (a.d == 64 && a.dv == 128) return launch_fused<64, 128>(a);
    if (a.d == 128 && a.dv == 64) return launch_fused<128, 64>(a);
    if (a.d == 128 && a.dv == 128) return launch_fused<128, 128>(a);
    return cudaErrorInvalidValue;
}

}  // namespace la
