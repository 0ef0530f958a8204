// simt_tiles.cuh -- shared pieces of the fp32 CUDA-core token-recurrent
// kernels (the causal forward with or without decay, and the gradients):
// register tiles of a d x dv state whose reductions stay inside a warp,
// warp reduce-scatter, vector shared-memory access, and a chunk of q/k/v/dy
// staged from HBM through registers.
#pragma once

#include <cstdint>

#include "la_device.cuh"

namespace la {
namespace tiles {

constexpr int kBC = 32;   // tokens per staged chunk

// psi(x) = elu(x) = phi(x) - 1.
__device__ __forceinline__ float psi_f(float x) { return x > 0.f ? x : __expf(x) - 1.f; }

// Tiling of a ROWS x COLS matrix over NT threads: warp w owns rows
// [w RPW, (w+1) RPW) and lane l owns columns [l CPL, (l+1) CPL) of each.
template <int NT, int ROWS, int COLS>
struct WarpRows {
    static constexpr int NW = NT / 32;
    static constexpr int RPW = ROWS / NW, CPL = COLS / 32;
    static_assert(RPW >= 2 && RPW <= 8 && (RPW & (RPW - 1)) == 0 && RPW * NW == ROWS &&
                  CPL >= 1 && CPL <= 4 && CPL * 32 == COLS, "tile");
    // the row whose finished sum lane `lane` holds after reduce_scatter<RPW>
    __device__ static int row_of(int lane) {
        int r = 0;
#pragma unroll
        for (int m = RPW, o = 16; m > 1; m >>= 1, o >>= 1)
            if (lane & o) r += m >> 1;
        return r;
    }
    // lanes that write the finished rows (one per row)
    __device__ static bool writer(int lane) { return (lane & (32 / RPW - 1)) == 0; }
};

// Packed fp32 pairs: two floats in one 64-bit register.  The f32x2
// arithmetic of sm_100 and later does both lanes in one instruction, each
// lane rounded exactly as the scalar operation would be.  The register tiles
// pair rows 2i and 2i + 1 of a column.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpk2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {   // a b + c
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 x) { *reinterpret_cast<float4 *>(p) = x; }

// n consecutive floats (n in {1, 2, 4, 8}, p aligned to min(n, 4) floats)
template <int n>
__device__ __forceinline__ void ldn(const float *p, float (&o)[n]) {
    if constexpr (n >= 4) {
#pragma unroll
        for (int i = 0; i < n; i += 4) {
            const float4 x = ld4(p + i);
            o[i] = x.x; o[i + 1] = x.y; o[i + 2] = x.z; o[i + 3] = x.w;
        }
    } else if constexpr (n == 2) {
        const float2 x = *reinterpret_cast<const float2 *>(p);
        o[0] = x.x; o[1] = x.y;
    } else {
        o[0] = *p;
    }
}

template <int n>
__device__ __forceinline__ void stn(float *p, const float (&x)[n]) {
    if constexpr (n >= 4) {
#pragma unroll
        for (int i = 0; i < n; i += 4) st4(p + i, make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]));
    } else if constexpr (n == 2) {
        *reinterpret_cast<float2 *>(p) = make_float2(x[0], x[1]);
    } else {
        *p = x[0];
    }
}

// Sum M per-lane values over the 32 lanes of a warp.  Each halving step
// trades half of the values with the partner lane, so the warp spends
// M - 1 + log2(32 / M) shuffles; lane l returns the total of value
// WarpRows::row_of(l).
template <int M>
__device__ __forceinline__ float reduce_scatter(const float (&x)[M], int lane) {
    float cur[M];
#pragma unroll
    for (int j = 0; j < M; ++j) cur[j] = x[j];
#pragma unroll
    for (int m = M, o = 16; m > 1; m >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < m / 2; ++j) {
            const float send = up ? cur[j] : cur[j + m / 2];
            const float keep = up ? cur[j + m / 2] : cur[j];
            cur[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
#pragma unroll
    for (int o = 16 / M; o > 0; o >>= 1) cur[0] += __shfl_xor_sync(0xffffffffu, cur[0], o);
    return cur[0];
}

template <typename T> struct Vec;
template <> struct Vec<float> {
    static constexpr int n = 4;
    __device__ static void unpack(uint4 u, float *o) {
        o[0] = __uint_as_float(u.x); o[1] = __uint_as_float(u.y);
        o[2] = __uint_as_float(u.z); o[3] = __uint_as_float(u.w);
    }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int n = 8;
    __device__ static void unpack(uint4 u, float *o) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[2 * i] = __uint_as_float(w[i] << 16);
            o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
};

// One chunk (kBC rows of width W) of a row-major global array, held in
// registers between its load and its store into shared memory as fp32.
template <int W, typename T, int NT>
struct ChunkLoad {
    static constexpr int n = Vec<T>::n;
    static constexpr int kVecs = kBC * W / n;
    static constexpr int kPer = (kVecs + NT - 1) / NT;
    uint4 r[kPer];
    // rows [0, L) of the chunk starting at src; the rest read as zero
    __device__ __forceinline__ void load(const T *src, int L) {
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = (threadIdx.x + i * NT) * n;
            r[i] = (e < kBC * W && e / W < L) ? __ldg(reinterpret_cast<const uint4 *>(src + e))
                                              : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    // dst[kBC][W] = op(x) on rows [0, L), 0 on the others
    template <typename Op>
    __device__ __forceinline__ void store(float *dst, int L, Op op) const {
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = (threadIdx.x + i * NT) * n;
            if (e >= kBC * W) continue;
            float x[n];
            Vec<T>::unpack(r[i], x);
            const bool valid = e / W < L;
#pragma unroll
            for (int j = 0; j < n; ++j) x[j] = valid ? op(x[j]) : 0.f;
#pragma unroll
            for (int j = 0; j < n; j += 4) st4(dst + e + j, make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]));
        }
    }
};

struct Ident { __device__ float operator()(float x) const { return x; } };
struct Phi { __device__ float operator()(float x) const { return phi_f(x); } };
struct Psi { __device__ float operator()(float x) const { return psi_f(x); } };

}  // namespace tiles
}  // namespace la
