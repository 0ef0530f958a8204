// decode.cu -- one recurrent decode step per head, in place on the fp32 state.
//
// "Linear Attention/es", "Forma recurrente e inferencia autorregresiva":
//   S <- S + phi(k) v^T,  z <- z + phi(k),  y = phi(q)^T S / max(phi(q)^T z, eps)
// (update first, then read, as in "La formulación recurrente paso a paso").
// With a per-head decay gamma (RetNet in "Variantes y extensiones":
// S <- gamma S + phi(k) v^T, and z alike) the stored state is scaled first;
// with a gate (gated linear attention, same section) row a of S and z[a] are
// scaled by the step's gate g (one value, or one per feature row).  The
// feature map is elu + 1 or the identity ("Mapas de características").
//
// The step is bound by HBM: per head it reads and writes d*dv*4 bytes of S
// and does 2*d*dv FMAs.  One CTA of 8 warps owns one head.  Warp w owns the
// d/8 rows [w*d/8, (w+1)*d/8) of S; lane l owns the dv/32 contiguous columns
// starting at l*dv/32, so each warp moves whole 128..512-byte rows with 4..16
// byte vector accesses.  All of a warp's row loads are issued before any is
// used to keep d/8 * dv*4/ (32 lanes) bytes per lane in flight.  The dot
// products over d are finished with a per-warp partial in shared memory
// (columns) and a warp-shuffle reduction (the denominator).
#include "la_device.cuh"
#include "la_internal.h"

namespace la {
namespace {

template <int VEC> struct FVec;
template <> struct FVec<1> {
    float x[1];
    __device__ __forceinline__ void load(const float *p) { x[0] = __ldcs(p); }
    __device__ __forceinline__ void store(float *p) const { __stcs(p, x[0]); }
};
template <> struct FVec<2> {
    float x[2];
    __device__ __forceinline__ void load(const float *p) {
        float2 t = __ldcs(reinterpret_cast<const float2 *>(p));
        x[0] = t.x; x[1] = t.y;
    }
    __device__ __forceinline__ void store(float *p) const {
        __stcs(reinterpret_cast<float2 *>(p), make_float2(x[0], x[1]));
    }
};
template <> struct FVec<4> {
    float x[4];
    __device__ __forceinline__ void load(const float *p) {
        float4 t = __ldcs(reinterpret_cast<const float4 *>(p));
        x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
    }
    __device__ __forceinline__ void store(float *p) const {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(x[0], x[1], x[2], x[3]));
    }
};

constexpr int kDecodeWarps = 8;

// MODE: 0 plain, 1 per-head decay gamma[H], 2 gate[head][gate_dim]
template <int D, int DV, typename T, int MODE>
__global__ void __launch_bounds__(kDecodeWarps * 32)
decode_step_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   float *__restrict__ y, float *__restrict__ S, float *__restrict__ z, float eps,
                   const float *__restrict__ gamma, int H, int phi, int gate_dim)
{
    constexpr bool DECAY = MODE != 0;
    constexpr int NW = kDecodeWarps;
    constexpr int RPW = D / NW;   // rows of S per warp
    constexpr int VEC = DV / 32;  // columns per lane
    static_assert(RPW >= 1 && VEC >= 1, "unsupported size");
    __shared__ float fq_s[D], fk_s[D], v_s[DV];
    __shared__ float ypart[NW][DV];
    __shared__ float dpart[NW];

    const int head = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long qk_off = (long)head * D, v_off = (long)head * DV;
    float *Sh = S + (long)head * D * DV;
    // the multiplier of row a of the stored state
    const float *gh = MODE == 2 ? gamma + (long)head * gate_dim : nullptr;
    const float g1 = MODE == 1 ? gamma[head % H] : (MODE == 2 ? gh[0] : 1.f);
    auto gate_of = [&](int a) { return MODE == 2 && gate_dim > 1 ? gh[a] : g1; };

    // Issue the state loads first: they are the whole cost of the step.
    FVec<VEC> s[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) s[r].load(Sh + (long)(warp * RPW + r) * DV + lane * VEC);

    // phi(q), phi(k), v to shared; z update and the denominator phi(q)^T z_new.
    float dp = 0.f;
    for (int i = tid; i < D; i += NW * 32) {
        const float fq = feature_f(to_f(q[qk_off + i]), phi);
        const float fk = feature_f(to_f(k[qk_off + i]), phi);
        fq_s[i] = fq;
        fk_s[i] = fk;
        const float zn = DECAY ? fmaf(gate_of(i), z[qk_off + i], fk) : z[qk_off + i] + fk;
        z[qk_off + i] = zn;
        dp = fmaf(fq, zn, dp);
    }
    for (int i = tid; i < DV; i += NW * 32) v_s[i] = to_f(v[v_off + i]);
    dp = warp_sum(dp);
    if (lane == 0) dpart[warp] = dp;
    __syncthreads();

    float vv[VEC], acc[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) { vv[c] = v_s[lane * VEC + c]; acc[c] = 0.f; }
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int a = warp * RPW + r;
        const float fk = fk_s[a], fq = fq_s[a], g = DECAY ? gate_of(a) : 1.f;
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
            const float sn = fmaf(fk, vv[c], DECAY ? g * s[r].x[c] : s[r].x[c]);
            s[r].x[c] = sn;
            acc[c] = fmaf(fq, sn, acc[c]);
        }
        s[r].store(Sh + (long)a * DV + lane * VEC);
    }
#pragma unroll
    for (int c = 0; c < VEC; ++c) ypart[warp][lane * VEC + c] = acc[c];
    __syncthreads();

    if (tid < DV) {
        float den = 0.f, num = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) { den += dpart[w]; num += ypart[w][tid]; }
        y[v_off + tid] = num / fmaxf(den, eps);
    }
}

template <int D, int DV, typename T, int MODE>
cudaError_t launch_typed(const DecodeArgs &a) {
    decode_step_kernel<D, DV, T, MODE><<<a.B * a.H, kDecodeWarps * 32, 0, a.stream>>>(
        (const T *)a.q, (const T *)a.k, (const T *)a.v, a.y, a.S, a.z, a.eps,
        MODE == 2 ? a.gate : a.gamma, a.H, a.phi, a.gate_dim);
    return cudaGetLastError();
}

template <int D, int DV, typename T>
cudaError_t launch_mode(const DecodeArgs &a) {
    if (a.gate) return launch_typed<D, DV, T, 2>(a);
    return a.gamma ? launch_typed<D, DV, T, 1>(a) : launch_typed<D, DV, T, 0>(a);
}

template <int D, int DV>
cudaError_t launch_dv(const DecodeArgs &a) {
    return a.dt == LA_DTYPE_BF16 ? launch_mode<D, DV, __nv_bfloat16>(a)
                                 : launch_mode<D, DV, float>(a);
}

template <int D>
cudaError_t launch_d(const DecodeArgs &a) {
    switch (a.dv) {
    case 32: return launch_dv<D, 32>(a);
    case 64: return launch_dv<D, 64>(a);
    case 128: return launch_dv<D, 128>(a);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs &a) {
    switch (a.d) {
    case 32: return launch_d<32>(a);
    case 64: return launch_d<64>(a);
    case 128: return launch_d<128>(a);
    }
    return cudaErrorInvalidValue;
}

}  // namespace la
