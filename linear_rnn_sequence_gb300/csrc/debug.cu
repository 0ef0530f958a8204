// debug.cu -- test-only entry point that applies the tensor-core kernels'
// bf16 feature function (feat_bf16x2 in tc_common.cuh: phi(x) - c, rounded to
// bf16, with c = 1 giving elu(x)) to an array, so that the function every
// tensor-core kernel feeds to the MMAs can be checked on its own against an
// fp64 reference, over every bf16 input.
#include "tc_common.cuh"

namespace la {
namespace {

constexpr int kFeatThreads = 256;

__global__ void __launch_bounds__(kFeatThreads)
feature_kernel(const uint16_t *__restrict__ x, uint16_t *__restrict__ out, long long n, float c)
{
    const SplitC k = split_pairs(c);
    const long long pairs = (n + 1) / 2;
    for (long long i = blockIdx.x * (long long)kFeatThreads + threadIdx.x; i < pairs;
         i += (long long)gridDim.x * kFeatThreads) {
        const long long e = 2 * i;
        const uint32_t lo = x[e], hi = e + 1 < n ? x[e + 1] : 0u;
        const uint32_t r = feat_bf16x2(lo | (hi << 16), k);
        out[e] = static_cast<uint16_t>(r & 0xFFFFu);
        if (e + 1 < n) out[e + 1] = static_cast<uint16_t>(r >> 16);
    }
}

}  // namespace
}  // namespace la

extern "C" la_status la_debug_feature_bf16(const void *x, void *out, long long n, float c,
                                           void *stream) {
    if (n < 0 || (n > 0 && (!x || !out))) return LA_ERR_INVALID_ARG;
    if (!(c >= 0.f && c <= 1.f)) return LA_ERR_INVALID_ARG;
    if (n == 0) return LA_OK;
    const long long pairs = (n + 1) / 2;
    long long blocks = (pairs + la::kFeatThreads - 1) / la::kFeatThreads;
    if (blocks > 4096) blocks = 4096;
    la::feature_kernel<<<(unsigned)blocks, la::kFeatThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(x), static_cast<uint16_t *>(out), n, c);
    return cudaGetLastError() == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}
