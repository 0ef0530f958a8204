// noalloc.cu -- a non-causal forward for callers that cannot allocate device
// memory: its scratch space is a fixed array compiled into the library.
//
// Who needs it: code that is handed only its input and output buffers and may
// not create any others, for example an operator or plugin inside another
// framework that owns all device memory, or a latency-critical path that
// must avoid cudaMalloc (which can synchronise the whole device).  Such a
// caller cannot provide the workspace la_forward_noncausal asks for.
//
// The scratch array below holds the split-N partial sums of S and z.  It is
// placed in device memory when the library is loaded on a GPU and stays there
// until the process exits (LA_NOALLOC_SCRATCH_BYTES on every GPU that loads
// the library).  Every call shares it; calls that can overlap on the GPU race
// on it, so the caller must order them (one stream, or explicit waits).
// Nothing in it has to start at zero: each call writes every partial it later
// reads, and clears the run-time status word at its start.  That word (a
// bounded wait that ran out) is read back with la_noalloc_status, since the
// caller holds no pointer to the array.
#include <mutex>

#include "la_internal.h"

namespace la {
namespace {

constexpr size_t kScratchBytes = LA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices];  // device address of the array, per device

// The array's name is only a host-side handle; the kernels need its device
// address, looked up once per device with that device current.
la_status scratch_address(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return LA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return LA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return LA_OK;
}

}  // namespace
}  // namespace la

extern "C" la_status la_forward_noncausal_noalloc(const void *q, const void *k, const void *v,
                                                  float *y, int B, int H, int N, int d, int dv,
                                                  la_dtype dt, float eps, float *S_out,
                                                  float *z_out, void *stream) {
    const size_t need = la_noncausal_workspace_bytes(B, H, N, d, dv, dt);
    if (need > la::kScratchBytes) return LA_ERR_WORKSPACE;  // too large for the fixed scratch
    void *scratch = nullptr;
    const la_status st = la::scratch_address(&scratch);
    if (st != LA_OK) return st;
    return la_forward_noncausal(q, k, v, y, B, H, N, d, dv, dt, eps, S_out, z_out, scratch,
                                la::kScratchBytes, stream);
}

extern "C" la_status la_noalloc_status(void *stream) {
    void *scratch = nullptr;
    const la_status st = la::scratch_address(&scratch);
    if (st != LA_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LA_ERR_CUDA;
    la::WsHeader h;
    if (cudaMemcpy(&h, scratch, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
        return LA_ERR_CUDA;
    return h.error == 0 ? LA_OK : static_cast<la_status>(h.error);
}
