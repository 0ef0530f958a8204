// tc_state.cuh -- tensor-core pass that reduces K and V of (head, segment)
// items to their states S_s = sum_j phi(k_j) v_j^T and z_s = sum_j phi(k_j)
// ("Linear Attention/es", "Reformulación con núcleos": the sums do not depend
// on the query).  Used for the sequence-axis split of the causal path and as
// the first pass of the non-causal path.
#pragma once

#include "tc_common.cuh"

namespace la {
namespace {

// For long sequences with few heads the sequence axis is split into segments
// ("Linear Attention/es", "Entrenamiento: forma paralela": the cumulative sums
// can be formed with a prefix scan).  Three launches, with no waits between
// CTAs:
//   1. per (head, segment), the segment's own state S_s = sum phi(k_j) v_j^T,
//      z_s = sum phi(k_j) from K and V (tensor cores): causal_state_kernel
//      below, or at d = 64 without a decay phase 1 of the fused non-causal
//      kernel (noncausal_tc.cu), which issues one MMA per 16 tokens;
//   2. scan_states_kernel: per head, exclusive prefixes P_s = S_in + sum_{s'<s} S_s';
//   3. causal_tc_kernel: every (head, segment) runs from its prefix.
// The state pass reuses the split form of the main kernel (per-key split
// constants c'_j, residual features b_j = bf16(phi(k_j) - c'_j)): R = B^T V,
// zeta = B^T 1 and u = V^T c' accumulate in TMEM, and the plain state is
// S = 1 u^T + R, z = n 1 + zeta with n = sum_j c'_j.
// With a per-head decay (DECAY) the segment's state is the decayed sum
// S_s = sum_j gamma^(end-1-j) phi(k_j) v_j^T (z alike), as the causal
// kernel's: key j of a block of L tokens carries s_j = gamma^(L-1-j), the
// TMEM sums are held divided by a running scale G that shrinks by gamma^L per
// block (keys enter multiplied by s_j / G; the export multiplies by G), and
// they are rescaled in TMEM only when G would fall below 2^-48.  With
// per-token gates (DK = 2) gamma^m becomes the product of the block's first m
// gates, read from the per-block tables of the gated path, and the pass also
// records each segment's product of gates for the prefix scan.
constexpr int kStateThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2..5 psi(k) / export
constexpr uint32_t kStColR = 0, kStColZ = 128, kStColU = 144, kStTmemCols = 256;

template <int D, int DV, bool DECAY = false>
struct StateLayout {
    static constexpr int kK = kC * D * 2;
    static constexpr int kV = kC * DV * 2;
    // [16 x C] operand per stage: row 0 = ones (zeta += B^T 1), rows 1, 2 =
    // the key weights as bf16 hi, lo (u += V^T s): s_j = c'_j, the key's split
    // constant (0 for padding rows), times gamma^(L-1-j) / G with a decay
    static constexpr int kOnes = 16 * kC * 2;
    static constexpr int oK = 0;                   // 2 stages
    static constexpr int oV = oK + 2 * kK;         // 2 stages
    static constexpr int oOnes = oV + 2 * kV;      // 2 stages
    static constexpr int oPad = oOnes + 2 * kOnes; // 16 KB the padded M = 128 operands may touch
    static constexpr int oSmall = oPad + 16384;
    static constexpr int oDecay = oSmall + 2048;   // decay only: StateDecay
    static constexpr int bytes = oDecay + (DECAY ? 1024 : 0);
    static constexpr int request = bytes + 1024;
};

struct StateSmall {
    alignas(16) float u[128];
    alignas(16) float n_part[4];      // per-warp sums of the keys' constants (decayed, over G)
    uint64_t kv_full[2], kv_empty[2], phik_done[2], init_done, st_done;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(StateSmall) <= 2048, "state small area");

struct StateDecay {
    alignas(16) float gpow[kC + 1];   // gamma^m
};
static_assert(sizeof(StateDecay) <= 1024, "state decay area");

// Where the state pass keeps the slow path of its bounded waits (the W of
// mbar_wait), as measured on the long-sequence workloads (d = 64).
template <int D, bool DECAY>
struct StateWaitPolicy {
    static constexpr int value = D == 64 ? (DECAY ? 1 : 2) : 0;
};

template <int D, int DV, int DK = 0>
__global__ void __launch_bounds__(kStateThreads)
causal_state_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const TcParams p, float *__restrict__ S_seg, float *__restrict__ z_seg)
{
    constexpr bool DECAY = DK != 0;   // a fixed decay (1) or gates (2)
    constexpr int kW = StateWaitPolicy<D, DECAY>::value;
    using Lay = StateLayout<D, DV, DK == 1>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
    StateSmall &S = *reinterpret_cast<StateSmall *>(sm + Lay::oSmall);
    StateDecay &X = *reinterpret_cast<StateDecay *>(sm + Lay::oDecay);   // DECAY only
    uint8_t *sK = sm + Lay::oK, *sV = sm + Lay::oV, *sOnes = sm + Lay::oOnes;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // work item = (head, segment) over the segments this pass reduces (the
    // causal split needs all but the last); its state goes to slot
    // head * nseg + seg
    const int item = blockIdx.x;
    const int nss = p.state_segs > 0 ? p.state_segs : p.nseg;
    const int head = item / nss, seg = item - head * nss;
    const int slot = head * p.nseg + seg;
    int tok0, nloc;
    segment_range(p, seg, tok0, nloc);
    const int nchunks = (nloc + kC - 1) / kC;
    const Guard g{&S.abort_flag, p.err, p.err_where, p.limit_ns};
    // reads only K and V: the consumer of S_seg waits for this whole grid
    griddep_launch_dependents();
    // decay: heads left to the CUDA-core kernel need no segment states (the
    // chunk kernel skips them too); the whole CTA leaves before any barrier
    if (DK == 1 && !decay_on_tensor_cores(p.gamma[head % p.H])) return;
    if (DK == 2 && p.gate_skip[head] != 0u) return;
    // gates: this segment's first block's table of gate products
    const float *gtab =
        DK == 2 ? p.gate_tab + ((size_t)head * p.gate_blocks + tok0 / kC) * kGateTab : nullptr;
    // the block's decay over its first m tokens
    auto pw = [&](int c, int m) { return DK == 2 ? __ldg(gtab + (size_t)c * kGateTab + m) : X.gpow[m]; };

    if (tid == 0) {
        S.abort_flag = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(&S.kv_full[s], 1);
            mbar_init(&S.kv_empty[s], 1);
            mbar_init(&S.phik_done[s], kWG);
        }
        mbar_init(&S.init_done, kWG);
        mbar_init(&S.st_done, 1);
        fence_mbar_init();
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
    }
    if (DK == 1 && tid < kC + 1) X.gpow[tid] = powf(p.gamma[head % p.H], (float)tid);
    if (warp == 1) {
        tmem_alloc(&S.tmem_base, kStTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = S.tmem_base;

    if (warp == 0) {
        if (lane == 0) {   // TMA: K and V blocks of this segment
            constexpr uint32_t kvbytes = kC * (D + DV) * 2;
            int last_kv[2] = {-1, -1};
            for (int c = 0; c < nchunks; ++c) {
                const int s = c & 1, t0 = tok0 + c * kC;
                if (c >= 2 && !mbar_wait<kW>(&S.kv_empty[s], ((c >> 1) - 1) & 1, g, 60)) break;
                mbar_arrive_expect_tx(&S.kv_full[s], kvbytes);
                for (int bx = 0; bx < D / 64; ++bx)
                    tma_load_3d(sK + s * Lay::kK + bx * kC * 128, &kmap, &S.kv_full[s], bx * 64, t0, head);
                for (int bx = 0; bx < DV / 64; ++bx)
                    tma_load_3d(sV + s * Lay::kV + bx * kC * 128, &vmap, &S.kv_full[s], bx * 64, t0, head);
                last_kv[s] = c;
            }
            if (*g.abort)
                for (int s = 0; s < 2; ++s)
                    if (last_kv[s] >= 0) drain_wait(&S.kv_full[s], (last_kv[s] >> 1) & 1, g.limit_ns);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // MMA: R += B^T V, zeta += B^T 1, u += V^T s (rows of the [1|s] operand)
            constexpr uint32_t iR = idesc_bf16(128, DV, 1, 1);
            constexpr uint32_t iZ = idesc_bf16(128, 16, 1, 0);
            bool ok = mbar_wait<kW>(&S.init_done, 0, g, 61);
            for (int c = 0; ok && c < nchunks; ++c) {
                const int s = c & 1;
                if (!mbar_wait<kW>(&S.kv_full[s], (c >> 1) & 1, g, 62)) break;
                if (!mbar_wait<kW>(&S.phik_done[s], (c >> 1) & 1, g, 63)) break;
                tc_fence_after();
                const uint32_t kb = smem_u32(sK + s * Lay::kK), vb = smem_u32(sV + s * Lay::kV);
                const uint32_t ob = smem_u32(sOnes + s * Lay::kOnes);
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks) {
                    const uint64_t ad = smem_desc(kb + ks * 2048, kC * 128, 1024, kSwizzle128B);
                    const uint64_t vd = smem_desc(vb + ks * 2048, kC * 128, 1024, kSwizzle128B);
                    const uint64_t od = smem_desc(ob + ks * 256, 128, 2048, kSwizzleNone);
                    mma_ss(tb + kStColR, ad, vd, iR, 1);
                    mma_ss(tb + kStColZ, ad, od, iZ, 1);
                    mma_ss(tb + kStColU, vd, od, iZ, 1);
                }
                mma_commit(&S.kv_empty[s]);
            }
            mma_commit(&S.st_done);
            drain_wait(&S.st_done, 0, g.limit_ns);
        }
    } else {
        const int wq = warp & 3, row = wq * 32 + lane, wtid = tid - 64;
        const uint32_t lb = (uint32_t)(wq * 32) << 16;
        // constant operands (row 0 = ones; rows 1, 2 are rewritten per block,
        // rows 3..15 stay 0) and a zeroed pad region
        for (int e = wtid; e < 2 * 16 * kC; e += kWG) {
            const int st = e / (16 * kC), n = (e / kC) % 16, k = e % kC;
            *reinterpret_cast<__nv_bfloat16 *>(sOnes + st * Lay::kOnes + (n >> 3) * 2048 +
                                               (k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2) =
                __float2bfloat16_rn(n == 0 ? 1.f : 0.f);
        }
        for (int e = wtid; e < 16384 / 16; e += kWG)
            reinterpret_cast<uint4 *>(sm + Lay::oPad)[e] = make_uint4(0u, 0u, 0u, 0u);
        {   // zero accumulators
            uint32_t zero[16];
#pragma unroll
            for (int m = 0; m < 16; ++m) zero[m] = 0u;
#pragma unroll
            for (int grp = 0; grp < DV / 16; ++grp) tmem_st16(tb + lb + kStColR + grp * 16, zero);
            tmem_st16(tb + lb + kStColZ, zero);
            tmem_st16(tb + lb + kStColU, zero);
            tmem_wait_st();
        }
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(&S.init_done);
        bool ok = true;
        DecayScale ks(DK == 1 ? X.gpow[1] : (DK == 2 ? 0.5f : 1.f));   // X.gpow[1] = gamma
        float segf = 1.f;   // gates: the segment's product of gates (thread wtid 0)
        float nrow = 0.f;   // this token row's share of n (with a decay: decayed, over G)
        for (int c = 0; c < nchunks; ++c) {
            const int s = c & 1;
            const int L = min(kC, nloc - c * kC);
            float sc = 1.f;
            if (DECAY) {
                const float Gp = ks.G, gL = pw(c, L);
                ks.step(gL);
                segf *= gL;
                nrow *= gL * Gp / ks.G;   // the count is carried over the new scale too
                if (ks.renorm && c > 0) {
                    // the previous block's MMAs must be done before the sums are rescaled
                    ok = wait_warp<kW>(&S.kv_empty[(c - 1) & 1], ((c - 1) >> 1) & 1, g, 66);
                    if (!ok) break;
                    tc_fence_after();
                    const float f = gL * Gp / ks.G0;
#pragma unroll 1
                    for (int grp = 0; grp < DV / 16 + 2; ++grp) {
                        const uint32_t col = grp < DV / 16 ? kStColR + grp * 16
                                                           : (grp == DV / 16 ? kStColZ : kStColU);
                        uint32_t rv[16];
                        tmem_ld16(tb + lb + col, rv);
                        tmem_wait_ld();
#pragma unroll
                        for (int m = 0; m < 16; ++m) rv[m] = f2u(u2f(rv[m]) * f);
                        tmem_st16(tb + lb + col, rv);
                    }
                    tmem_wait_st();
                }
                const float kw = DK == 2 ? gL * __ldg(gtab + (size_t)c * kGateTab + kGateInv + row + 1)
                                         : X.gpow[L - 1 - row];
                sc = row < L ? kw / ks.G : 0.f;
            }
            ok = wait_warp<kW>(&S.kv_full[s], (c >> 1) & 1, g, 64);
            if (!ok) break;
            uint8_t *kt = sK + s * Lay::kK;
            // the key's split constant from its first eight features (padding
            // rows read zeros: c' = 1), read before the row is overwritten
            const float ck = split_const(*reinterpret_cast<const uint4 *>(kt + sw128_off(row, 0)));
            const SplitC kk = split_pairs(ck);
#pragma unroll 1
            for (int f0 = 0; f0 < D / 8; f0 += 8) {
                uint4 raw[8];
#pragma unroll
                for (int f = 0; f < 8; ++f)
                    raw[f] = *reinterpret_cast<const uint4 *>(
                        kt + ((f0 + f) >> 3) * (kC * 128) + sw128_off(row, ((f0 + f) & 7) * 8));
#pragma unroll
                for (int f = 0; f < 8; ++f) {
                    uint32_t w[4] = {raw[f].x, raw[f].y, raw[f].z, raw[f].w};
#pragma unroll
                    for (int h = 0; h < 4; ++h)
                        w[h] = DECAY ? feat_scaled_bf16x2(w[h], kk, sc) : feat_bf16x2(w[h], kk);
                    raw[f] = make_uint4(w[0], w[1], w[2], w[3]);
                }
#pragma unroll
                for (int f = 0; f < 8; ++f)
                    *reinterpret_cast<uint4 *>(kt + ((f0 + f) >> 3) * (kC * 128) +
                                               sw128_off(row, ((f0 + f) & 7) * 8)) = raw[f];
            }
            {   // rows 1, 2: the key weight s_j = c'_j sc as a bf16 pair (u += V^T s;
                // sc = 1 without a decay); 0 on padding rows
                const float sj = row < L ? sc * ck : 0.f;
                const float sh = bf16_round(sj), sl = bf16_round(sj - sh);
                uint8_t *op = sOnes + s * Lay::kOnes + (row >> 3) * 128 + (row & 7) * 2;
                *reinterpret_cast<__nv_bfloat16 *>(op + 16) = __float2bfloat16_rn(sh);
                *reinterpret_cast<__nv_bfloat16 *>(op + 32) = __float2bfloat16_rn(sl);
                nrow += sh + sl;
            }
            fence_proxy_async();
            if (DECAY) tc_fence_before();   // after a rescale of the TMEM sums
            mbar_arrive(&S.phik_done[s]);
        }
        ok = ok && wait_warp<kW>(&S.st_done, 0, g, 65);
        if (ok) {   // plain state of the segment: S = 1 u^T + R, z = n 1 + zeta
            tc_fence_after();
            uint32_t zv[4], uv[4];
            tmem_ld4(tb + lb + kStColZ, zv);
            tmem_ld4(tb + lb + kStColU, uv);
            tmem_wait_ld();
            // u = v^T [s_hi + s_lo] (columns 1, 2); with a decay the sums are held over G
            const float G = DECAY ? ks.G : 1.f;
            S.u[row] = G * (u2f(uv[1]) + u2f(uv[2]));
            const float ns = warp_sum_f(nrow);
            if (lane == 0) S.n_part[wq] = ns;
            named_bar(kBarA, kWG);
            float *dst = S_seg + (size_t)slot * D * DV;
#pragma unroll 1
            for (int grp = 0; grp < DV / 16; ++grp) {
                uint32_t rv[16];
                tmem_ld16(tb + lb + kStColR + grp * 16, rv);
                tmem_wait_ld();
                if (row < D)
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 4)
                        *reinterpret_cast<float4 *>(dst + (size_t)row * DV + grp * 16 + jj) =
                            make_float4(fmaf(u2f(rv[jj]), G, S.u[grp * 16 + jj]),
                                        fmaf(u2f(rv[jj + 1]), G, S.u[grp * 16 + jj + 1]),
                                        fmaf(u2f(rv[jj + 2]), G, S.u[grp * 16 + jj + 2]),
                                        fmaf(u2f(rv[jj + 3]), G, S.u[grp * 16 + jj + 3]));
            }
            // n = sum of the keys' constants (nloc when every constant is 1)
            const float n = G * ((S.n_part[0] + S.n_part[1]) + (S.n_part[2] + S.n_part[3]));
            if (row < D) z_seg[(size_t)slot * D + row] = fmaf(u2f(zv[0]), G, n);
            if (DK == 2 && wtid == 0) p.seg_decay[slot] = segf;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tb, kStTmemCols);
    }
}

}  // namespace
}  // namespace la
