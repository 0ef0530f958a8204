// la_internal.h -- internal declarations shared by the CUDA translation units
// of liblinattn.so.  Not part of the public ABI (that is include/linattn.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "linattn.h"

namespace la {

// Everything a forward launch needs; pointers are device pointers.
struct FwdArgs {
    const void *q, *k, *v;
    float *y;
    int B, H, N, d, dv;
    la_dtype dt;
    float eps;
    const float *S_in, *z_in;   // nullable (zero initial state)
    float *S_out, *z_out;       // nullable
    void *ws;                   // workspace (may be null when none is needed)
    size_t ws_bytes;
    cudaStream_t stream;
    const float *gamma = nullptr;   // per-head decay [H] (device), null: none
    // decay only: heads whose gamma passes decay_on_tensor_cores were already
    // computed by the tensor-core kernel; the CUDA-core kernel skips them
    bool skip_tc_heads = false;
    int phi = 0;                    // feature map: 0 elu + 1, 1 identity (CUDA-core kernels)
    const float *gate = nullptr;    // per-token gate [B][H][N][gate_dim] (device), null: none
    int gate_dim = 1;               // 1 or d
    // gates: per-head flags of the gated tensor-core path (0: that kernel took
    // the head, and the CUDA-core kernel skips it); null: every head here
    const unsigned int *gate_skip = nullptr;
    int BH() const { return B * H; }
};

// The decayed tensor-core kernel scales block-local weights by gamma^-128 and
// gamma^-(i+1); with gamma >= 2^-1/2 these stay below 2^64, far inside the
// fp32 and bf16 range.  Smaller decays (and values outside [0, 1], NaN)
// take the CUDA-core kernel, which multiplies the state token by token.
__host__ __device__ inline bool decay_on_tensor_cores(float gamma) {
    return gamma >= 0.70710678f && gamma <= 1.f;
}

struct DecodeArgs {
    const void *q, *k, *v;
    float *y, *S, *z;
    int B, H, d, dv;
    la_dtype dt;
    float eps;
    cudaStream_t stream;
    const float *gamma = nullptr;   // per-head decay [H] (device), null: none
    int phi = 0;                    // feature map: 0 elu + 1, 1 identity
    const float *gate = nullptr;    // per-step gate [B][H][gate_dim] (device), null: none
    int gate_dim = 1;               // 1 or d
};

// Gradients of the causal form; pointers are device pointers.
struct BwdArgs {
    const void *q, *k, *v;
    const float *dy;
    float *dq, *dk, *dv_grad;
    int B, H, N, d, dv;
    la_dtype dt;
    float eps;
    const float *S_in, *z_in;      // nullable (zero initial state)
    float *grad_S_in, *grad_z_in;  // nullable
    void *ws;
    size_t ws_bytes;
    cudaStream_t stream;
    const float *gamma = nullptr;  // per-head decay [H] (device), null: none
};

// Workspace header written at the start of every workspace (256 bytes).
struct WsHeader {
    unsigned int error;         // 0 = ok, else an la_status value (LA_ERR_TIMEOUT)
    unsigned int error_where;   // diagnostic: which segment gave up
    unsigned int reserved;
    unsigned int pad[61];
};
static_assert(sizeof(WsHeader) == 256, "workspace header must be 256 bytes");

// Process-wide test hook state (see la_debug_set_fault).
struct DebugFault {
    int drop_load_item = -1;      // work item whose first tile copy is never issued
    long long wait_limit_ns = 0;  // <= 0: default limit of every bounded wait
};
DebugFault &debug_fault();

// ---- launchers (return cudaSuccess or the launch error) ------------------
cudaError_t launch_decode_simt(const DecodeArgs &a);
cudaError_t launch_causal_simt(const FwdArgs &a);
size_t noncausal_simt_workspace(int BH, int N, int d, int dv);
cudaError_t launch_noncausal_simt(const FwdArgs &a);

// tcgen05 / TMA path (bf16 inputs, d and dv in {64, 128}).
bool causal_tc_supported(const FwdArgs &a);
size_t causal_tc_workspace(int BH, int N, int d, int dv);
int causal_tc_launches(int BH, int N);   // kernels one causal call launches
cudaError_t launch_causal_tc(const FwdArgs &a);
// the gated form on the tensor cores (gate_dim 1, elu + 1, bf16, d and dv in
// {64, 128}): workspace = header | per-head flags | per-block gate tables |
// the sequence split's segment states
bool gated_tc_supported(const FwdArgs &a);
size_t gated_tables_offset(int BH);
size_t gated_split_offset(int BH, int N);
size_t gated_tc_workspace(int BH, int N, int d, int dv);
size_t gated_tc_clear_bytes(int BH);   // header and flags, cleared before each call
cudaError_t launch_gated_tc(const FwdArgs &a);
bool noncausal_tc_supported(const FwdArgs &a);
size_t noncausal_tc_workspace(int BH, int N, int d, int dv);
size_t noncausal_tc_clear_bytes(int BH);   // workspace bytes to zero before each call
cudaError_t launch_noncausal_tc(const FwdArgs &a);
// States of every segment but each head's last for the causal sequence split
// (d = 64, bf16, no decay), into slot head * nseg + segment of S_seg, z_seg.
cudaError_t launch_segment_states_nc(const FwdArgs &a, int nseg, int seg_chunks, float *S_seg,
                                     float *z_seg);

// gated recurrence and feature maps (CUDA cores, fp32)
cudaError_t launch_causal_gated(const FwdArgs &a);        // tensor cores where they apply
cudaError_t launch_causal_gated_simt(const FwdArgs &a);   // CUDA cores (skips a.gate_skip's heads)
cudaError_t launch_random_features(const void *x, float *out, long long rows, int d, int m,
                                   la_dtype dt, const float *W, cudaStream_t stream);

// gradients of the causal form (CUDA cores, fp32)
size_t causal_backward_workspace(int BH, int N, int d, int dv);
cudaError_t launch_causal_backward(const BwdArgs &a);

}  // namespace la
