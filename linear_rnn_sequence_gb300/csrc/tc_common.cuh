// tc_common.cuh -- helpers shared by the tensor-core kernels (causal and
// non-causal): the psi feature function, swizzled shared-memory addressing,
// warp-uniform bounded waits, group barriers, TMA tensor-map encoding.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>
#include <utility>

#include "la_internal.h"
#include "tc_ptx.cuh"

namespace la {
namespace {

using namespace tc;

constexpr int kC = 128;          // tokens per block (MMA M)
constexpr int kWG = 128;         // threads per row-worker group
constexpr int kBarA = 1, kBarB = 2;  // named barrier ids of the two row-worker groups

struct TcParams {
    float *y;
    int N, BH;
    int nseg;                      // segments per head (work items = BH * nseg)
    int seg_chunks;                // blocks per segment (the last one may be shorter)
    float eps;
    const float *S_in, *z_in;
    float *S_out, *z_out;
    unsigned int *err;             // workspace header error word
    unsigned int *err_where;
    unsigned long long limit_ns;
    int drop_item;                 // test hook: this item's first K/V copy is never issued (-1: off)
    const float *gamma;            // per-head decay [H] (causal kernel with DECAY only)
    int H;
    // per-token gates (causal kernel with gates only): per-block tables of the
    // gate products, gate_blocks blocks per head, and a per-head flag that is
    // nonzero when a gate lies outside the kernel's range
    const float *gate_tab;
    const unsigned int *gate_skip;
    int gate_blocks;
    float *seg_decay;              // gates with a sequence split: each segment's product of gates
    int state_segs;                // segments per head the state pass reduces (0: all)
};

// Per-token gates: one table per 128-token block, [P_0 .. P_128 | pad | 1/P_0 .. 1/P_128 | pad]
// with P_m = g_t0 g_t0+1 ... g_t0+m-1 the product of the block's first m gates.
constexpr int kGateInv = kC + 4;          // offset of the inverses
constexpr int kGateTab = 2 * kGateInv;    // floats per block
// Gates the tensor-core kernels take: [2^-1/2, 1], so that the products over a
// block stay at or above 2^-64, the range the fixed decay is held to.
constexpr float kGateMin = 0.70710677f;

// Token range of segment seg of a head (segments of seg_chunks blocks).
__device__ __forceinline__ void segment_range(const TcParams &p, int seg, int &tok0, int &nloc) {
    tok0 = seg * p.seg_chunks * kC;
    nloc = min(p.N - tok0, p.seg_chunks * kC);
}

// Decay: the TMEM state (the causal kernel's R, zeta, u, r; the segment
// sums of the state pass) is held divided by a scale G that
// shrinks by gamma^L with every block, so a block's update only adds to it
// (its keys enter multiplied by 1/G) and the export multiplies by G.  When
// gamma^L G would fall below 2^-48, the state is instead rescaled in TMEM
// before the block and G restarts at G0.  G0 = 3/4 (1 when gamma = 1): the
// first keys after a restart then carry scales near 4/3 rather than just
// above 1, where bf16(scale * x) would round most bf16 values x back to x and
// drop the scale from their psi part in the same direction for every
// feature.  Each role steps its own copy through the blocks in order; the
// copies agree bit for bit.
struct DecayScale {
    float G0;              // restart value
    float G;               // scale of the state after the current block
    bool renorm = false;   // the state is rescaled in TMEM before the current block
    __device__ __forceinline__ explicit DecayScale(float gamma)
        : G0(gamma == 1.f ? 1.f : 0.75f), G(G0) {}
    __device__ __forceinline__ void step(float gL) {
        const float cand = gL * G;
        renorm = cand < 0x1p-48f;
        G = renorm ? G0 : cand;
    }
};


// Packed fp32 pairs (two floats in one 64-bit register; the f32x2 arithmetic
// of sm_100 and later does both lanes in one instruction).
__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ float f2sum(uint64_t v) {
    float a, b;
    f2unpack(v, a, b);
    return a + b;
}

__device__ __forceinline__ float bf16_round(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

// ---- the features the tensor cores see ------------------------------------
// phi(x) = elu(x) + 1 is split per token as phi(x) = c + (phi(x) - c): the
// constant c is carried exactly (it is a bf16 value) and only the residual
// phi(x) - c enters the MMAs as bf16.  For inputs of order one or below,
// phi is close to 1 and c = 1 (the residual is then elu(x) itself); for a
// token whose features are mostly strongly negative (phi << 1) a residual
// taken against 1 would cancel almost all of phi, so c is then the mean of
// phi over the token's first eight features.  The kernels compute the exact
// attention of the features c + bf16(phi(x) - c).
constexpr float kLog2e = 1.4426950408889634f;
// e^x - 1 is replaced by x above this argument: for -2^-8 < x < 0 the two
// differ by less than x^2 / 2, under half a bf16 unit of x, while the fp32
// e^x - 1 loses relative accuracy there
constexpr float kExpArgMax = -0.00390625f;

// Split constant of a token from its first eight features (one 16-byte
// chunk of the bf16 row): 1 when the mean of phi over them is at least 1/2,
// else that mean rounded to bf16.  Every role that needs a token's constant
// computes it from the same eight values with the same operations.  When
// all eight inputs are at least ln(1/2), every phi is at least 1/2 and the
// constant is 1 without any exponential; the warp takes the full rule only
// when one of its rows needs it (a warp-wide vote: all lanes must call this
// together), so a row's constant does not depend on its warp's other rows.
constexpr float kLnHalf = -0.693147180559945f;
__device__ __forceinline__ float split_const(uint4 raw) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    float mn = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        mn = fminf(mn, fminf(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u)));
    if (!__any_sync(0xffffffffu, !(mn >= kLnHalf))) return 1.f;
    uint64_t acc = f2pack(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // phi(x) = max(x + 1, e^min(x, 0)), on packed pairs
        const float x0 = __uint_as_float(w[i] << 16), x1 = __uint_as_float(w[i] & 0xFFFF0000u);
        float t0, t1, a0, a1;
        f2unpack(f2mul(f2pack(fminf(x0, 0.f), fminf(x1, 0.f)), f2pack(kLog2e, kLog2e)), t0, t1);
        f2unpack(f2add(f2pack(x0, x1), f2pack(1.f, 1.f)), a0, a1);
        acc = f2add(acc, f2pack(fmaxf(a0, ex2_ftz(t0)), fmaxf(a1, ex2_ftz(t1))));
    }
    const float m = f2sum(acc) * 0.125f;
    return m >= 0.5f ? 1.f : bf16_round(m);
}

// The per-token constants as packed pairs: (1 - c, 1 - c) and (-c, -c).
struct SplitC {
    uint64_t omc2, nc2;
};
__device__ __forceinline__ SplitC split_pairs(float c) {
    return {f2pack(1.f - c, 1.f - c), f2pack(-c, -c)};
}

// phi(x) - c of both bf16 halves of w, rounded to bf16x2:
//   max(x + 1 - c, e^min(x, -2^-8) - c).
// For x <= -2^-8 the exponential term is the larger (e^x >= 1 + x); for
// x > -2^-8 it is e^-2^-8 - c, below x + 1 - c.  Branch-free, so lanes with
// inputs of either sign stay converged.  e^x = 2^(x log2 e) in the
// flush-to-zero form (a flushed result means e^x < 2^-126).  The multiply
// and the adds run on the packed pair.  With c = 1 this is elu(x).
__device__ __forceinline__ uint32_t feat_bf16x2(uint32_t w, const SplitC &k) {
    const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xFFFF0000u);
    float t0, t1, e0, e1, a0, a1;
    f2unpack(f2mul(f2pack(fminf(x0, kExpArgMax), fminf(x1, kExpArgMax)),
                   f2pack(kLog2e, kLog2e)), t0, t1);
    f2unpack(f2add(f2pack(ex2_ftz(t0), ex2_ftz(t1)), k.nc2), e0, e1);
    f2unpack(f2add(f2pack(x0, x1), k.omc2), a0, a1);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(fmaxf(a1, e1)), "f"(fmaxf(a0, e0)));
    return r;
}

// The same, also adding the two residuals (before their bf16 rounding) to
// the packed row sum acc.  The row sums feed the constant parts of the
// weights (c beta_j and c' alpha_i); taking them before the rounding moves a
// weight by a constant per row or per key of about sqrt(d) 2^-9 |phi - c|,
// some 1e-5 of the weight, and saves the unpacking of the rounded pair.
__device__ __forceinline__ uint32_t feat_bf16x2_sum(uint32_t w, const SplitC &k, uint64_t &acc) {
    const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xFFFF0000u);
    float t0, t1, e0, e1, a0, a1;
    f2unpack(f2mul(f2pack(fminf(x0, kExpArgMax), fminf(x1, kExpArgMax)),
                   f2pack(kLog2e, kLog2e)), t0, t1);
    f2unpack(f2add(f2pack(ex2_ftz(t0), ex2_ftz(t1)), k.nc2), e0, e1);
    f2unpack(f2add(f2pack(x0, x1), k.omc2), a0, a1);
    const float r0 = fmaxf(a0, e0), r1 = fmaxf(a1, e1);
    acc = f2add(acc, f2pack(r0, r1));
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(r1), "f"(r0));
    return r;
}

// sc * (phi(x) - c) for both bf16 halves of w, rounded once to bf16x2 (the
// decayed kernels weight key j by sc = gamma^(L-1-j) / G before the tensor
// cores see it).
__device__ __forceinline__ uint32_t feat_scaled_bf16x2(uint32_t w, const SplitC &k, float sc) {
    const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xFFFF0000u);
    float t0, t1, e0, e1, a0, a1;
    f2unpack(f2mul(f2pack(fminf(x0, kExpArgMax), fminf(x1, kExpArgMax)),
                   f2pack(kLog2e, kLog2e)), t0, t1);
    f2unpack(f2add(f2pack(ex2_ftz(t0), ex2_ftz(t1)), k.nc2), e0, e1);
    f2unpack(f2add(f2pack(x0, x1), k.omc2), a0, a1);
    f2unpack(f2mul(f2pack(fmaxf(a0, e0), fmaxf(a1, e1)), f2pack(sc, sc)), e0, e1);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(e1), "f"(e0));
    return r;
}

// sc * (phi(x) - c) as feat_scaled_bf16x2, also adding the scaled residuals
// (before their bf16 rounding) to the packed row sum acc (see feat_bf16x2_sum).
__device__ __forceinline__ uint32_t feat_scaled_bf16x2_sum(uint32_t w, const SplitC &k, float sc,
                                                           uint64_t &acc) {
    const float x0 = __uint_as_float(w << 16), x1 = __uint_as_float(w & 0xFFFF0000u);
    float t0, t1, e0, e1, a0, a1;
    f2unpack(f2mul(f2pack(fminf(x0, kExpArgMax), fminf(x1, kExpArgMax)),
                   f2pack(kLog2e, kLog2e)), t0, t1);
    f2unpack(f2add(f2pack(ex2_ftz(t0), ex2_ftz(t1)), k.nc2), e0, e1);
    f2unpack(f2add(f2pack(x0, x1), k.omc2), a0, a1);
    const uint64_t m = f2mul(f2pack(fmaxf(a0, e0), fmaxf(a1, e1)), f2pack(sc, sc));
    acc = f2add(acc, m);
    f2unpack(m, e0, e1);
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(e1), "f"(e0));
    return r;
}

__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// acc (two fp32 lanes) += the two bf16 halves of p.
__device__ __forceinline__ uint64_t acc_bf16x2(uint64_t acc, uint32_t p) {
    return f2add(acc, f2pack(__uint_as_float(p << 16), __uint_as_float(p & 0xFFFF0000u)));
}

// Byte offset of element (row, col) in a [rows x 64] bf16 box with 128-byte
// swizzle, the layout TMA writes (16-byte chunk index XOR row % 8).
__device__ __forceinline__ uint32_t sw128_off(int row, int col) {
    return (uint32_t)row * 128u + ((((uint32_t)col >> 3) ^ ((uint32_t)row & 7u)) << 4) +
           (((uint32_t)col & 7u) << 1);
}


__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
__device__ __forceinline__ float warp_sum_f(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Warp-uniform bounded wait: every lane polls, the warp agrees on the result.
template <int W = 0>
__device__ __forceinline__ bool wait_warp(uint64_t *bar, uint32_t parity, const Guard &g,
                                          unsigned int where) {
    const bool ok = mbar_wait<W>(bar, parity, g, where);
    return __all_sync(0xffffffffu, ok);
}

// Wait used only while unwinding after an abort: ignores the abort flag but
// still gives up after the time limit.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) break;
}

// Group barrier that also agrees on "someone gave up": returns true if any of
// the group's COUNT threads passes failed = true.
template <int BAR, int COUNT = kWG>
__device__ __forceinline__ bool group_any(bool failed) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)failed), "n"(BAR), "n"(COUNT)
        : "memory");
    return r != 0;
}


// ------------------------------------------------------------------ host helpers
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// 3-D map over [heads][rows][inner] with a box of [1][box_rows][box_inner].
bool encode_3d(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esz, int inner,
               int rows, int heads, int box_inner, int box_rows, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)heads};
    const cuuint64_t strides[2] = {(cuuint64_t)inner * esz, (cuuint64_t)rows * inner * esz};
    const cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launch `kern` with programmatic stream serialization: it may start while
// the previous kernel in the stream is still running, and must call
// griddep_wait before it reads anything that kernel writes.
template <typename... Params, typename... Args>
cudaError_t launch_overlapped(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 152;
    return n;
}

}  // namespace
}  // namespace la
