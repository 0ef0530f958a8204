// noncausal_tc.cu -- non-causal elu(x)+1 linear attention on the sm_103a
// tensor cores (tcgen05 MMA, TMEM accumulators, TMA tiles, mbarriers).
//
// Method ("Linear Attention/es", "Reformulación con núcleos"): the sums
//   S = sum_j phi(k_j) v_j^T  [d x dv],   z = sum_j phi(k_j)  [d]
// do not depend on the query, so they are formed once per head and every
// query reads them: y_i = phi(q_i)^T S / max(phi(q_i)^T z, eps).
//
// Three launches, none of which waits on another CTA:
//   1. causal_state_kernel (shared with the causal path): per (head, segment)
//      item, the segment's S_s and z_s from K and V on the tensor cores;
//   2. noncausal_prepare_kernel: per head, S = sum_s S_s and z = sum_s z_s in a
//      fixed segment order (so the result does not depend on scheduling),
//      the optional S_out / z_out, and a ready-to-copy image of the query
//      kernel's operands: S as bf16 hi + lo pairs in the 128-byte-swizzled
//      layout the MMA reads, z likewise, and sum_i z_i;
//   3. noncausal_query_kernel: per (head, range of 128-query blocks), one bulk
//      copy brings the head's operand image into shared memory, then for every
//      block  A = psi_c(Q) [128 x d] (the residual features phi(q) - c_i, in
//      place over the TMA tile) times S_hi and S_lo into a TMEM accumulator,
//      A times z_hi, z_lo into two more columns, and the epilogue
//        y_i = (c_i colsum(S) + a_i^T S) / max(c_i sum z + a_i^T z, eps),
//      using phi(q_i) = c_i 1 + a_i, so phi(q_i)^T S = c_i 1^T S + a_i^T S.
// Precision: the residual features enter the tensor cores as bf16 (the same
// features c + bf16(phi(x) - c), with the same per-token split constants, as
// the causal path; split_const in tc_common.cuh); S and z are fp32 sums split
// into bf16 hi + lo pairs, so the rounding of the state costs about 2^-17 of
// its value; colsum(S) and sum z are fp32.  Outputs are float32.
//
// Query kernel warp roles (320 threads):
//   warp 0      TMA producer (operand image once, then Q tiles, 3 stages)
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2..5  group A: psi_c(q) in place in shared memory, one token row per thread
//   warps 6..9  group B (thread = TMEM lane): normaliser epilogue, 16-byte stores;
//               each thread takes its row's split constant from the row's first
//               eight features in global memory (just read by the TMA, so an
//               L2 hit), since the tile itself has been overwritten by then
// Two TMEM accumulators (blocks c and c+1) let the epilogue of one block
// overlap the MMA of the next.  Every wait is bounded in time; a wait that
// runs out records LA_ERR_TIMEOUT in the workspace header and the CTA unwinds.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>

#include "la_internal.h"
#include "tc_common.cuh"
#include "tc_state.cuh"

namespace la {
namespace {

constexpr int kQThreads = 320;
constexpr int kQWarpB = 6;       // first warp of group B
constexpr int kQStages = 3;      // Q tiles in flight

// Operand image of one head, identical in global memory (written by the
// prepare kernel) and in shared memory (one bulk copy):
//   [hi]   S_hi: dv/64 boxes of [d rows][64 columns] bf16, 128-byte swizzle
//   [lo]   S_lo = bf16(S - S_hi), same layout
//   [zt]   [16 x d] bf16, K-major, no swizzle: row 0 = z_hi, row 1 = z_lo, rest 0
//   [zsum] sum_i z_i (fp32), padded to 16 bytes
template <int D, int DV>
struct OpImage {
    static constexpr int kHi = 0;
    static constexpr int kLo = D * DV * 2;
    static constexpr int kZt = 2 * D * DV * 2;
    static constexpr int kZsum = kZt + 16 * D * 2;
    static constexpr int bytes = kZsum + 16;
    static constexpr int stride = (bytes + 1023) / 1024 * 1024;   // per head in the workspace
    static_assert(bytes % 16 == 0 && kZt % 1024 == 0, "bulk copy and swizzle alignment");
};

// Byte offset of element (k, n) in the [16 x D] no-swizzle K-major operand.
__host__ __device__ __forceinline__ uint32_t ztile_off(int n, int k, int D) {
    return (uint32_t)((n >> 3) * (D * 16) + (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2);
}

// ------------------------------------------------------------------ prepare
// Grid (heads, D*DV/512 + 1), 128 threads.  Blocks y < D*DV/512: one float4
// of S per thread, summed over the segments in order; the last block: z.
constexpr int kPrepThreads = 128;

template <int D, int DV>
__global__ void __launch_bounds__(kPrepThreads)
noncausal_prepare_kernel(const float *__restrict__ S_seg, const float *__restrict__ z_seg,
                         int nseg, uint8_t *__restrict__ img_all, float *__restrict__ S_out,
                         float *__restrict__ z_out)
{
    using Img = OpImage<D, DV>;
    constexpr int kSBlocks = D * DV / (4 * kPrepThreads);
    griddep_launch_dependents();
    griddep_wait();   // S_seg, z_seg come from the state pass
    const int head = blockIdx.x, tid = threadIdx.x;
    uint8_t *img = img_all + (size_t)head * Img::stride;
    if ((int)blockIdx.y < kSBlocks) {
        const int e4 = blockIdx.y * kPrepThreads + tid;   // float4 index in [D][DV]
        const int a = (e4 * 4) / DV, b = (e4 * 4) % DV;
        const float4 *src = reinterpret_cast<const float4 *>(S_seg + (size_t)head * nseg * D * DV) + e4;
        const size_t st = (size_t)D * DV / 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int s = 0;
        for (; s + 4 <= nseg; s += 4) {
            const float4 x0 = src[(s + 0) * st], x1 = src[(s + 1) * st];
            const float4 x2 = src[(s + 2) * st], x3 = src[(s + 3) * st];
            acc.x += x0.x; acc.y += x0.y; acc.z += x0.z; acc.w += x0.w;
            acc.x += x1.x; acc.y += x1.y; acc.z += x1.z; acc.w += x1.w;
            acc.x += x2.x; acc.y += x2.y; acc.z += x2.z; acc.w += x2.w;
            acc.x += x3.x; acc.y += x3.y; acc.z += x3.z; acc.w += x3.w;
        }
        for (; s < nseg; ++s) {
            const float4 x = src[s * st];
            acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
        }
        if (S_out) reinterpret_cast<float4 *>(S_out + (size_t)head * D * DV)[e4] = acc;
        const float v[4] = {acc.x, acc.y, acc.z, acc.w};
        uint32_t hi[2], lo[2];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            hi[m] = pack_bf16x2(v[2 * m], v[2 * m + 1]);
            lo[m] = pack_bf16x2(v[2 * m] - bf16_lo_f(hi[m]), v[2 * m + 1] - bf16_hi_f(hi[m]));
        }
        // four consecutive columns stay inside one 16-byte swizzle chunk
        const uint32_t off = (uint32_t)(b >> 6) * (D * 128) + sw128_off(a, b & 63);
        *reinterpret_cast<uint2 *>(img + Img::kHi + off) = make_uint2(hi[0], hi[1]);
        *reinterpret_cast<uint2 *>(img + Img::kLo + off) = make_uint2(lo[0], lo[1]);
    } else {
        __shared__ float wsum[kPrepThreads / 32];
        float z = 0.f;
        if (tid < D) {
            const float *src = z_seg + (size_t)head * nseg * D + tid;
            for (int s = 0; s < nseg; ++s) z += src[(size_t)s * D];
            if (z_out) z_out[(size_t)head * D + tid] = z;
            const float zh = bf16_round(z);
#pragma unroll
            for (int n = 0; n < 16; ++n)
                *reinterpret_cast<__nv_bfloat16 *>(img + Img::kZt + ztile_off(n, tid, D)) =
                    __float2bfloat16_rn(n == 0 ? zh : (n == 1 ? z - zh : 0.f));
        }
        const float ws = warp_sum_f(z);   // fixed butterfly order: deterministic
        if ((tid & 31) == 0) wsum[tid >> 5] = ws;
        __syncthreads();
        if (tid == 0) {
            float t = 0.f;
            for (int w = 0; w < kPrepThreads / 32; ++w) t += wsum[w];
            *reinterpret_cast<float4 *>(img + Img::kZsum) = make_float4(t, 0.f, 0.f, 0.f);
        }
    }
}

// ------------------------------------------------------------------ query kernel
struct QParams {
    float *y;
    const __nv_bfloat16 *q;        // the queries themselves (split constants of the epilogue)
    int D;
    const uint8_t *img;            // operand images, OpImage::stride bytes per head
    int N;
    int nq;                        // query ranges per head (work items = heads * nq)
    int q_chunks;                  // 128-query blocks per range (the last one may be shorter)
    float eps;
    unsigned int *err;
    unsigned int *err_where;
    unsigned long long limit_ns;
    int drop_item;                 // test hook: this item's first Q copy is never issued (-1: off)
};

struct QSmall {
    alignas(16) float colsum[128];     // colsum(S), fp32
    alignas(16) float cpart[128];      // second half of the column sums while they are formed
    alignas(16) float e_inv[kC];       // 1 / max(den, eps) per row of the current block
    alignas(16) float cq[kC];          // split constant per row of the current block
    float zsum;
    uint64_t q_full[kQStages], q_empty[kQStages], psi_done[kQStages];
    uint64_t op_full, acc_full[2], acc_empty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(offsetof(QSmall, q_full) % 8 == 0, "mbarriers need 8-byte alignment");

template <int D, int DV>
struct QLayout {
    static constexpr int kQ = kC * D * 2;
    static constexpr int oQ = 0;                                   // kQStages stages
    static constexpr int oOp = kQStages * kQ;                      // 1024-aligned
    static constexpr int oSmall = oOp + OpImage<D, DV>::stride;
    static constexpr int bytes = oSmall + (int)sizeof(QSmall);
    static constexpr int request = bytes + 1024;
    // TMEM: accumulators Y_0, Y_1 [0, 2 dv), denominators [2 dv, 2 dv + 32)
    static constexpr uint32_t colDen = 2 * DV;
    static constexpr uint32_t tmem_cols = (2 * DV + 32 <= 256) ? 256 : 512;
    // two CTAs per SM when both TMEM and shared memory allow it
    static constexpr int min_blocks = (tmem_cols <= 256 && request <= 113 * 1024) ? 2 : 1;
    static_assert(oOp % 1024 == 0, "swizzled operands need 1024-byte alignment");
};

template <int D, int DV>
__global__ void __launch_bounds__(kQThreads, QLayout<D, DV>::min_blocks)
noncausal_query_kernel(const __grid_constant__ CUtensorMap qmap, const QParams p)
{
    using Lay = QLayout<D, DV>;
    using Img = OpImage<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    QSmall &S = *reinterpret_cast<QSmall *>(sm + Lay::oSmall);
    uint8_t *sQ = sm + Lay::oQ, *sOp = sm + Lay::oOp;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int item = blockIdx.x;
    const int head = item / p.nq, qr = item - head * p.nq;
    const int tok0 = qr * p.q_chunks * kC;
    const int nloc = min(p.N - tok0, p.q_chunks * kC);
    const int nchunks = (nloc + kC - 1) / kC;
    const Guard g{&S.abort_flag, p.err, p.err_where, p.limit_ns};

    if (tid == 0) {
        S.abort_flag = 0;
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&S.q_full[s], 1);
            mbar_init(&S.q_empty[s], 1);
            mbar_init(&S.psi_done[s], kWG);
        }
        mbar_init(&S.op_full, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&S.acc_full[b], 1);
            mbar_init(&S.acc_empty[b], kWG);
        }
        mbar_init(&S.drain, 1);
        fence_mbar_init();
        prefetch_tmap(&qmap);
    }
    if (warp == 1) {
        tmem_alloc(&S.tmem_base, Lay::tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem_base;

    if (warp == 0) {
        if (lane == 0) {   // Q tiles of this range and, once it exists, the operand image
            // The first kQStages tiles read only q, so they are issued before
            // waiting for the kernels that write the image (this kernel may
            // start while they run: programmatic dependent launch).
            const int npre = min(nchunks, kQStages);
            const bool drop = item == p.drop_item;   // test hook: block 0 never arrives
            int c_last = -1;                          // last block whose copy was issued
            auto load_q = [&](int c) {
                const int s = c % kQStages;
                mbar_arrive_expect_tx(&S.q_full[s], kC * D * 2);
                if (c == 0 && drop) return;
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load_3d(sQ + s * Lay::kQ + bx * kC * 128, &qmap, &S.q_full[s], bx * 64,
                                tok0 + c * kC, head);
                c_last = c;
            };
            for (int c = 0; c < npre; ++c) load_q(c);
            griddep_wait();
            mbar_arrive_expect_tx(&S.op_full, Img::bytes);
            bulk_load(sOp, p.img + (size_t)head * Img::stride, Img::bytes, &S.op_full);
            for (int c = npre; c < nchunks; ++c) {
                if (!mbar_wait(&S.q_empty[c % kQStages], ((c / kQStages) - 1) & 1, g, 70)) break;
                load_q(c);
            }
            if (*g.abort) {   // no copy may still be landing when the CTA exits
                drain_wait(&S.op_full, 0, g.limit_ns);
                // copies were issued for every block up to c_last (block 0
                // excepted when dropped); the newest one on each stage:
                for (int s = 0; s < kQStages; ++s) {
                    if (c_last < 0) break;
                    const int c = c_last - ((c_last - s) % kQStages + kQStages) % kQStages;
                    if (c < 0 || (c == 0 && drop)) continue;
                    drain_wait(&S.q_full[s], (c / kQStages) & 1, g.limit_ns);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {   // Y_b = psi(Q) (S_hi + S_lo), den_b = psi(Q) [z_hi | z_lo]
            constexpr uint32_t iY = idesc_bf16(128, DV, 0, 1);   // A K-major, B MN-major
            constexpr uint32_t iZ = idesc_bf16(128, 16, 0, 0);   // A K-major, B K-major
            const uint32_t hb = smem_u32(sOp + Img::kHi), lb2 = smem_u32(sOp + Img::kLo);
            const uint32_t zb = smem_u32(sOp + Img::kZt);
            griddep_wait();   // bounded waits below start once the image exists
            bool ok = mbar_wait(&S.op_full, 0, g, 71);
            for (int c = 0; ok && c < nchunks; ++c) {
                const int s = c % kQStages, b = c & 1;
                if (!mbar_wait(&S.psi_done[s], (c / kQStages) & 1, g, 72)) break;
                if (c >= 2 && !mbar_wait(&S.acc_empty[b], ((c >> 1) - 1) & 1, g, 73)) break;
                tc_fence_after();
                const uint32_t qb = smem_u32(sQ + s * Lay::kQ);
                const uint32_t dY = tb + (uint32_t)(b * DV), dZ = tb + Lay::colDen + 16u * b;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t ad =
                        smem_desc(qb + (ks >> 2) * (kC * 128) + (ks & 3) * 32, 16, 1024, kSwizzle128B);
                    const uint64_t hd = smem_desc(hb + ks * 2048, D * 128, 1024, kSwizzle128B);
                    const uint64_t ld = smem_desc(lb2 + ks * 2048, D * 128, 1024, kSwizzle128B);
                    const uint64_t zd = smem_desc(zb + ks * 256, 128, D * 16, kSwizzleNone);
                    mma_ss(dY, ad, hd, iY, ks > 0);
                    mma_ss(dY, ad, ld, iY, 1);
                    mma_ss(dZ, ad, zd, iZ, ks > 0);
                }
                mma_commit(&S.q_empty[s]);
                mma_commit(&S.acc_full[b]);
            }
            mma_commit(&S.drain);
            drain_wait(&S.drain, 0, g.limit_ns);
        }
    } else if (warp < kQWarpB) {
        // group A: psi(q) in place (bf16) over the swizzled Q tile, one row per thread
        const int row = (warp & 3) * 32 + lane;
        for (int c = 0; c < nchunks; ++c) {
            const int s = c % kQStages;
            // tiles from kQStages on wait for the MMA, hence for the image
            if (c == kQStages) griddep_wait();
            const bool ok = wait_warp(&S.q_full[s], (c / kQStages) & 1, g, 74);
            if (ok) {
                uint8_t *qt = sQ + s * Lay::kQ;
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
                        for (int h = 0; h < 4; ++h)
                            w[h] = feat_bf16x2(w[h], kq);
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
        // group B: column sums of S once, then the normaliser epilogue per block
        const int wq = warp & 3, row = wq * 32 + lane, wtid = tid - kQWarpB * 32;
        griddep_wait();
        bool ok = wait_warp(&S.op_full, 0, g, 75);
        ok = !group_any<kBarB>(!ok);   // all four warps agree before the named barriers below
        if (ok) {
            constexpr int P = kWG / DV;   // threads per column (1 or 2)
            const int b = wtid % DV, part = wtid / DV;
            const uint8_t *hi = sOp + Img::kHi + (b >> 6) * (D * 128);
            const uint8_t *lo = sOp + Img::kLo + (b >> 6) * (D * 128);
            float cs = 0.f;
#pragma unroll 4
            for (int a = part; a < D; a += P) {
                const uint32_t off = sw128_off(a, b & 63);
                cs += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(hi + off)) +
                      __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(lo + off));
            }
            if (part == 1) S.cpart[b] = cs;
            named_bar(kBarB, kWG);
            if (part == 0) S.colsum[b] = (P == 2) ? cs + S.cpart[b] : cs;
            named_bar(kBarB, kWG);
        }
        const float zsum = *reinterpret_cast<const float *>(sOp + Img::kZsum);
        const int tq = lane >> 2, tcol = (lane & 3) * 2;
        constexpr int kParts = 2 * (DV / 32);   // (16-lane half, 32-column block) pairs
        for (int c = 0; ok && c < nchunks; ++c) {
            const int b = c & 1;
            // this row's first eight features (rows past the range: c = 1),
            // loaded while the block's MMAs run
            uint4 first = make_uint4(0u, 0u, 0u, 0u);
            if (c * kC + row < nloc)
                first = *reinterpret_cast<const uint4 *>(
                    p.q + ((size_t)head * p.N + tok0 + c * kC + row) * p.D);
            ok = wait_warp(&S.acc_full[b], (c >> 1) & 1, g, 76);
            if (ok) {
                tc_fence_after();
                uint32_t dz[4];
                tmem_ld4(tb + ((uint32_t)(wq * 32) << 16) + Lay::colDen + 16u * b, dz);
                const float cr = split_const(first);
                tmem_wait_ld();
                __syncwarp();
                S.cq[row] = cr;
                S.e_inv[row] = 1.f / fmaxf(fmaf(cr, zsum, u2f(dz[0]) + u2f(dz[1])), p.eps);
                __syncwarp();
                const int t0 = c * kC;
                float *ychunk = p.y + ((size_t)head * p.N + tok0 + t0) * DV;
                auto part_addr = [&](int part) {
                    return tb + ((uint32_t)(wq * 32 + 16 * (part & 1)) << 16) + (uint32_t)(b * DV) +
                           (part >> 1) * 32;
                };
                // 16x256b shape: 4 neighbouring lanes hold 8 consecutive columns of
                // one row, so each warp store covers whole 32-byte sectors
                auto outputs = [&](int part, const uint32_t (&vc)[16]) {
                    const int half = part & 1, cblk = part >> 1;
                    const int rA = wq * 32 + 16 * half + tq, rB = rA + 8;
                    const float invA = S.e_inv[rA], invB = S.e_inv[rB];
                    const float cA = S.cq[rA], cB = S.cq[rB];
                    const bool okA = t0 + rA < nloc, okB = t0 + rB < nloc;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int col = cblk * 32 + 8 * k + tcol;
                        const float2 cs = *reinterpret_cast<const float2 *>(S.colsum + col);
                        const float2 oA = make_float2(fmaf(cA, cs.x, u2f(vc[4 * k])) * invA,
                                                      fmaf(cA, cs.y, u2f(vc[4 * k + 1])) * invA);
                        const float2 oB = make_float2(fmaf(cB, cs.x, u2f(vc[4 * k + 2])) * invB,
                                                      fmaf(cB, cs.y, u2f(vc[4 * k + 3])) * invB);
                        if (okA) *reinterpret_cast<float2 *>(ychunk + (size_t)rA * DV + col) = oA;
                        if (okB) *reinterpret_cast<float2 *>(ychunk + (size_t)rB * DV + col) = oB;
                    }
                };
                uint32_t vA[16], vB[16];
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
                tc_fence_before();
                mbar_arrive(&S.acc_empty[b]);
            }
            if (group_any<kBarB>(!ok)) break;
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
// Both the state pass and the query pass split each head's blocks into
// ranges so that about two waves of (head, range) items cover the SMs.
void nc_split(int BH, int N, int &nranges, int &range_chunks) {
    const int nch = (N + kC - 1) / kC;
    const int sms = num_sms();
    int want = (2 * sms + BH - 1) / BH;
    if (want > nch) want = nch;
    if (want < 1) want = 1;
    range_chunks = (nch + want - 1) / want;
    if (range_chunks < 1) range_chunks = 1;
    nranges = (nch + range_chunks - 1) / range_chunks;
    if (nranges < 1) nranges = 1;
}

size_t image_stride(int d, int dv) {
    const size_t bytes = 4 * (size_t)d * dv + 32 * (size_t)d + 16;
    return (bytes + 1023) / 1024 * 1024;
}

// [header][S_seg: heads*nseg*d*dv][z_seg: heads*nseg*d][pad to 1024][images: heads*stride]
size_t images_offset(int BH, int nseg, int d, int dv) {
    const size_t o = sizeof(WsHeader) + 4 * (size_t)BH * nseg * ((size_t)d * dv + d);
    return (o + 1023) / 1024 * 1024;
}

template <int D, int DV>
cudaError_t launch_nc(const FwdArgs &a) {
    using SL = StateLayout<D, DV>;
    using QL = QLayout<D, DV>;
    static_assert(OpImage<D, DV>::stride % 1024 == 0, "image stride");
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
    const unsigned long long limit_ns = lim > 0 ? (unsigned long long)lim : 1000000000ull;

    TcParams sp{};
    sp.N = a.N;
    sp.BH = BH;
    sp.eps = a.eps;
    nc_split(BH, a.N, sp.nseg, sp.seg_chunks);
    sp.err = &hdr->error;
    sp.err_where = &hdr->error_where;
    sp.limit_ns = limit_ns;
    sp.drop_item = -1;
    char *ws = static_cast<char *>(a.ws);
    float *S_seg = reinterpret_cast<float *>(ws + sizeof(WsHeader));
    float *z_seg = S_seg + (size_t)BH * sp.nseg * D * DV;
    uint8_t *img = reinterpret_cast<uint8_t *>(ws + images_offset(BH, sp.nseg, D, DV));

    auto skern = causal_state_kernel<D, DV>;
    cudaError_t e = cudaFuncSetAttribute(skern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SL::request);
    if (e != cudaSuccess) return e;
    skern<<<BH * sp.nseg, kStateThreads, SL::request, a.stream>>>(km, vm, sp, S_seg, z_seg);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    // the prepare and query kernels may start while their predecessor runs;
    // each waits for it (griddep_wait) before touching what it writes
    const dim3 pgrid(BH, D * DV / (4 * kPrepThreads) + 1);
    e = launch_overlapped(noncausal_prepare_kernel<D, DV>, pgrid, dim3(kPrepThreads), 0, a.stream,
                          (const float *)S_seg, (const float *)z_seg, sp.nseg, img, a.S_out,
                          a.z_out);
    if (e != cudaSuccess) return e;

    QParams qp{};
    qp.y = a.y;
    qp.q = static_cast<const __nv_bfloat16 *>(a.q);
    qp.D = D;
    qp.img = img;
    qp.N = a.N;
    qp.eps = a.eps;
    nc_split(BH, a.N, qp.nq, qp.q_chunks);
    qp.err = &hdr->error;
    qp.err_where = &hdr->error_where;
    qp.limit_ns = limit_ns;
    qp.drop_item = debug_fault().drop_load_item;
    auto qkern = noncausal_query_kernel<D, DV>;
    if ((e = cudaFuncSetAttribute(qkern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  QL::request)) != cudaSuccess)
        return e;
    return launch_overlapped(qkern, dim3(BH * qp.nq), dim3(kQThreads), QL::request, a.stream, qm,
                             qp);
}

}  // namespace

bool noncausal_tc_supported(const FwdArgs &a) {
    return a.dt == LA_DTYPE_BF16 && (a.d == 64 || a.d == 128) && (a.dv == 64 || a.dv == 128);
}

size_t noncausal_tc_workspace(int BH, int N, int d, int dv) {
    int nseg, seg_chunks;
    nc_split(BH, N, nseg, seg_chunks);
    return images_offset(BH, nseg, d, dv) + (size_t)BH * image_stride(d, dv);
}

cudaError_t launch_noncausal_tc(const FwdArgs &a) {
    if (a.d == 64 && a.dv == 64) return launch_nc<64, 64>(a);
    if (a.d == 64 && a.dv == 128) return launch_nc<64, 128>(a);
    if (a.d == 128 && a.dv == 64) return launch_nc<128, 64>(a);
    if (a.d == 128 && a.dv == 128) return launch_nc<128, 128>(a);
    return cudaErrorInvalidValue;
}

}  // namespace la
