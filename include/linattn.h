/*
 * linattn.h -- C ABI of liblinattn.so: elu(x)+1 kernelized linear attention
 * on one NVIDIA GB300 GPU (sm_103a).
 *
 * The method ("Linear Attention/es", section "Reformulación con núcleos"):
 *
 *     y_i = phi(q_i)^T S / max(phi(q_i)^T z, eps),
 *     S   = sum_j phi(k_j) v_j^T  (d x dv),   z = sum_j phi(k_j)  (d),
 *     phi(x) = elu(x) + 1 = x + 1 (x > 0), e^x (x <= 0)
 *
 * ("Mapas de características"; "Linear Transformer (Transformers are RNNs)",
 * section "La función ELU + 1").  The sums run over all j (non-causal) or over
 * j <= i (causal: "Forma recurrente e inferencia autorregresiva", where the
 * state is updated with token i before it is read).  The denominator is
 * clamped from below by eps, as the worked PyTorch examples on the "Linear
 * Transformer" page do with clamp_min.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Pointers   All tensor pointers are DEVICE pointers (cudaMalloc'd or
 *             equivalent) owned by the caller.  The library allocates no
 *             device memory and keeps no state between calls except a small
 *             host-side cache of TMA tensor maps (none outlives the process).
 *  Layout     Contiguous row-major:
 *               q, k : [B][H][N][d]   (decode: [B][H][d])   dtype `dt`
 *               v    : [B][H][N][dv]  (decode: [B][H][dv])  dtype `dt`
 *               y    : [B][H][N][dv]  (decode: [B][H][dv])  float32
 *               S    : [B][H][d][dv]  float32,  z : [B][H][d] float32
 *             q, k, v and y must be 16-byte aligned; S and z 16-byte aligned.
 *  Output     y is float32 for both input dtypes.  (A bfloat16 output could
 *             not meet the stated accuracy: rounding y alone to bf16 moves the
 *             largest early-token outputs by up to 2^-9 of their size, far more
 *             than 2e-2 of the RMS of y for long causal sequences.)
 *  Sizes      B, H >= 1; N >= 0 (N = 0 is a no-op that still writes the
 *             final state when asked; q, k, v, y may then be NULL);
 *             d, dv in {32, 64, 128}.  Other d / dv
 *             return LA_ERR_UNSUPPORTED.  B*H*N*max(d,dv) must fit in 2^31.
 *  eps        must be finite and > 0, else LA_ERR_INVALID_ARG.
 *  Streams    `stream` is a cudaStream_t (NULL = legacy default stream).  All
 *             work is enqueued asynchronously; the call returns after the
 *             launches.  Launch failures return LA_ERR_CUDA.
 *  Aliasing   y must not alias q, k, v, S or z.  S_in may equal S_out and
 *             z_in may equal z_out (read fully before written per head).
 *  Errors     Argument checks happen on the host before anything is
 *             launched; on any error nothing is enqueued.  The only error a
 *             kernel can raise at run time is a bounded wait that ran out
 *             (LA_ERR_TIMEOUT), recorded in the workspace and reported by
 *             la_workspace_status().
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__) || defined(__clang__)
#define LA_API __attribute__((visibility("default")))
#else
#define LA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad size, bad eps */
    LA_ERR_UNSUPPORTED = 2,   /* d or dv outside {32, 64, 128}, unknown dtype  */
    LA_ERR_CUDA = 3,          /* a CUDA runtime / driver call failed           */
    LA_ERR_TIMEOUT = 4,       /* a bounded inter-CTA wait ran out (see above)  */
    LA_ERR_WORKSPACE = 5      /* workspace missing or smaller than required    */
} la_status;

typedef enum {
    LA_DTYPE_F32 = 0,         /* float32 q, k, v                               */
    LA_DTYPE_BF16 = 1         /* bfloat16 q, k, v                              */
} la_dtype;

/* The element-wise feature maps of "Mapas de características". */
typedef enum {
    LA_PHI_ELU1 = 0,          /* phi(x) = elu(x) + 1 (the canonical map)       */
    LA_PHI_IDENTITY = 1       /* phi(x) = x (bilinear attention)               */
} la_phi;

/* Human-readable name of a status code (static string, never NULL). */
LA_API const char *la_status_string(la_status s);

/* Library version string, e.g. "linattn 0.1 sm_103a". */
LA_API const char *la_version(void);

/*
 * Workspace size in bytes for la_forward_causal and la_forward_causal_decay
 * with these sizes (0 when the chosen kernels need none).  The workspace holds a small header (run-time
 * status) and, when the heads alone cannot fill the GPU, the per-segment
 * states and their prefixes for the sequence-axis split ("Entrenamiento:
 * forma paralela": cumulative sums by a prefix scan).  The split depends on
 * the current device's SM count, so query with the device current that will
 * run the call.  It must be device memory, 256-byte aligned, and may be
 * reused by later calls on the same stream.
 */
LA_API size_t la_causal_workspace_bytes(int B, int H, int N, int d, int dv, la_dtype dt);

/*
 * Workspace size in bytes for la_forward_noncausal with these sizes (0 for
 * N == 0 or unsupported sizes).  It holds the run-time status header and
 * the partial sums of S and z over ranges of the sequence (bf16 inputs with
 * d, dv in {64, 128}: also one arrival counter per head, which the call
 * clears with the header; other cases: the split-N partial sums).  Like the
 * causal workspace it depends on the dtype and on the current device's SM
 * count; it must be device memory, 256-byte aligned, and may be reused by
 * later calls on the same stream.
 */
LA_API size_t la_noncausal_workspace_bytes(int B, int H, int N, int d, int dv, la_dtype dt);

/*
 * Causal forward ("Linear Attention/es", "Forma recurrente e inferencia
 * autorregresiva" for the definition, computed blockwise as in
 * "Entrenamiento: forma paralela"):
 *   for each (b, h) and t = 0..N-1:
 *     S_t = S_{t-1} + phi(k_t) v_t^T,  z_t = z_{t-1} + phi(k_t),
 *     y_t = phi(q_t)^T S_t / max(phi(q_t)^T z_t, eps)
 * starting from (S_in, z_in), or from zero when both are NULL (one NULL and
 * one not is LA_ERR_INVALID_ARG).  When S_out / z_out are non-NULL the final
 * (S_N, z_N) is written there (both or neither).
 */
LA_API la_status la_forward_causal(const void *q, const void *k, const void *v, float *y,
                            int B, int H, int N, int d, int dv, la_dtype dt, float eps,
                            const float *S_in, const float *z_in,
                            float *S_out, float *z_out,
                            void *workspace, size_t workspace_bytes, void *stream);

/*
 * Causal forward with a per-head decay ("Linear Attention/es", "Variantes y
 * extensiones", RetNet: the unbounded cumulative sum is replaced by
 *   S_t = gamma_h S_{t-1} + phi(k_t) v_t^T,  z_t = gamma_h z_{t-1} + phi(k_t),
 *   y_t = phi(q_t)^T S_t / max(phi(q_t)^T z_t, eps),
 * one gamma per head for the multi-scale retention the section mentions; z
 * is decayed like S so that y stays a normalised average).  gamma is a DEVICE
 * array of H floats in [0, 1], 4-byte aligned, shared by the B batch rows;
 * its values are not checked (a value outside [0, 1] gives a meaningless
 * result, not an error).  Arguments, layouts, the initial / final state and
 * the workspace (size: la_causal_workspace_bytes; its status header and, for
 * split sequences, the decayed segment states and their prefixes; NULL when
 * that size is 0) as in la_forward_causal.
 * bf16 inputs with d, dv in {64, 128}: heads with gamma in [2^-1/2, 1] run on
 * the tensor cores, 128-token blocks as in la_forward_causal with key j of a
 * block of L tokens weighted by gamma^(L-1-j), the block's weights by
 * gamma^-L, and the carried state decayed by gamma^L per block (same
 * precision scheme and bound as la_forward_causal; long sequences with few
 * heads are split into segments the same way, with decayed segment states
 * and prefixes); a second kernel then computes the other heads on the CUDA
 * cores.  Otherwise (float32 inputs,
 * d or dv = 32) every head runs on the CUDA cores, token by token in fp32.
 * The split needs no host read of gamma.  NULL gamma: LA_ERR_INVALID_ARG.
 */
LA_API la_status la_forward_causal_decay(const void *q, const void *k, const void *v, float *y,
                                         int B, int H, int N, int d, int dv, la_dtype dt,
                                         float eps, const float *gamma, const float *S_in,
                                         const float *z_in, float *S_out, float *z_out,
                                         void *workspace, size_t workspace_bytes,
                                         void *stream);

/*
 * One decode step with a per-head decay, in place on (S, z):
 *   S <- gamma_h S + phi(k) v^T,  z <- gamma_h z + phi(k),
 *   y = phi(q)^T S / max(phi(q)^T z, eps).
 * gamma as in la_forward_causal_decay; the rest as in la_decode_step.
 */
LA_API la_status la_decode_step_decay(const void *q, const void *k, const void *v, float *y,
                                      float *S, float *z, int B, int H, int d, int dv,
                                      la_dtype dt, float eps, const float *gamma, void *stream);

/*
 * Workspace size in bytes for la_forward_causal_gated with a gate of
 * gate_dim values per token (1 or d); 0 for unsupported arguments.  For bf16
 * inputs with d, dv in {64, 128}, gate_dim = 1 and LA_PHI_ELU1 (the
 * tensor-core path) it holds the run-time status header, one flag per head,
 * per-128-token-block tables of gate products (1,056 bytes per block and
 * head) and, when few heads make the call split the sequence into segments,
 * the segments' states and products of gates, so it depends on the current
 * device's SM count; otherwise the header alone (256 bytes), which also serves
 * a call without a gate.  Device memory, 256-byte aligned, reusable by later
 * calls on the same stream.
 */
LA_API size_t la_causal_gated_workspace_bytes(int B, int H, int N, int d, int dv, la_dtype dt,
                                              la_phi phi, int gate_dim);

/*
 * Gated causal forward ("Linear Attention/es", "Variantes y extensiones":
 * gated linear attention replaces RetNet's scalar decay by a data-dependent
 * gate; the pages print no equation, and the update is read as the decay's
 * with the decay taken per token):
 *   S_t = diag(g_t) S_{t-1} + phi(k_t) v_t^T,  z_t = g_t * z_{t-1} + phi(k_t),
 *   y_t = phi(q_t)^T S_t / max(phi(q_t)^T z_t, eps),
 * g_t in [0, 1] given per token: gate is a DEVICE float32 array
 * [B][H][N][gate_dim], 4-byte aligned, with gate_dim = 1 (one gate per token;
 * row a of S and z[a] all scale by it) or gate_dim = d (one per token and
 * feature row of S); gate = NULL means no gate (g_t = 1), which with phi =
 * LA_PHI_IDENTITY gives the identity-map swap of "Mapas de características"
 * (the layer becomes a bilinear attention).  phi: LA_PHI_ELU1 or
 * LA_PHI_IDENTITY (else LA_ERR_UNSUPPORTED); with the identity map the
 * denominator can be <= 0, and the clamp then gives num / eps.  Layouts,
 * sizes, the initial / final state and the errors as in la_forward_causal.
 * Workspace: la_causal_gated_workspace_bytes (header size when gate is NULL),
 * overlapping no other buffer.
 *
 * Where it applies (bf16, d and dv in {64, 128}, gate_dim = 1, LA_PHI_ELU1),
 * the heads whose gates all lie in [2^-1/2, 1] run on the tensor cores, as
 * the decayed form of la_forward_causal_decay does, with the bf16 tolerance;
 * the device decides per head from the gate values, and the other heads
 * (closed gates, NaN, ...) run on the CUDA cores.  Everything else runs on
 * the CUDA cores, token by token in float32, one CTA per head.  A wait of the
 * tensor-core path that runs out records LA_ERR_TIMEOUT in the workspace
 * header (la_workspace_status).
 */
LA_API la_status la_forward_causal_gated(const void *q, const void *k, const void *v, float *y,
                                         int B, int H, int N, int d, int dv, la_dtype dt,
                                         float eps, la_phi phi, const float *gate, int gate_dim,
                                         const float *S_in, const float *z_in, float *S_out,
                                         float *z_out, void *workspace, size_t workspace_bytes,
                                         void *stream);

/*
 * One gated decode step in place on (S, z):
 *   S <- diag(g) S + phi(k) v^T,  z <- g * z + phi(k),  y = phi(q)^T S / max(phi(q)^T z, eps),
 * gate a DEVICE float32 array [B][H][gate_dim] (gate_dim 1 or d; NULL: no
 * gate), phi as in la_forward_causal_gated; the rest as in la_decode_step.
 */
LA_API la_status la_decode_step_gated(const void *q, const void *k, const void *v, float *y,
                                      float *S, float *z, int B, int H, int d, int dv,
                                      la_dtype dt, float eps, la_phi phi, const float *gate,
                                      int gate_dim, void *stream);

/*
 * Workspace size in bytes for la_forward_noncausal_phi: that of
 * la_forward_noncausal for LA_PHI_ELU1; for LA_PHI_IDENTITY the status
 * header and the split-N partial sums of the CUDA-core path.  0 for
 * unsupported arguments.
 */
LA_API size_t la_noncausal_phi_workspace_bytes(int B, int H, int N, int d, int dv, la_dtype dt,
                                               la_phi phi);

/*
 * Non-causal forward with a choice of element-wise feature map ("Mapas de
 * características"): la_forward_noncausal for LA_PHI_ELU1; for
 * LA_PHI_IDENTITY the same sums with phi(x) = x, on the CUDA cores in
 * float32.  Workspace: la_noncausal_phi_workspace_bytes.
 */
LA_API la_status la_forward_noncausal_phi(const void *q, const void *k, const void *v, float *y,
                                          int B, int H, int N, int d, int dv, la_dtype dt,
                                          float eps, la_phi phi, float *S_out, float *z_out,
                                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * Positive random features ("Mapas de características", Performer: phi(x)
 * proportional to exp(W x - ||x||^2 / 2), W random projections; the constant
 * is taken as 1 / sqrt(m), so that phi(q) . phi(k) averages exp(q . k)
 * estimates over the m rows of W):
 *   phi_out[r][f] = exp(W[f] . x[r] - ||x[r]||^2 / 2) / sqrt(m)
 * x: DEVICE [rows][d] of dtype dt (aligned to its element size); W: DEVICE
 * float32 [m][d], drawn by the caller (the library draws no random numbers);
 * phi_out: DEVICE float32 [rows][m], 4-byte aligned, overlapping neither.
 * 1 <= d <= 128, 1 <= m <= 256, else LA_ERR_INVALID_ARG.  The features then
 * go to the attention calls as float32 inputs with LA_PHI_IDENTITY and
 * d = m (m in {32, 64, 128}).  Computed in float32 on the CUDA cores.
 */
LA_API la_status la_random_features(const void *x, float *phi_out, long long rows, int d, int m,
                                    la_dtype dt, const float *W, void *stream);

/*
 * Workspace size in bytes for la_backward_causal (0 for N == 0 or
 * unsupported sizes).  It holds the run-time status header, per-segment
 * forward and reverse state sums for the sequence-axis split, and two floats
 * per token (1 / max(den_t, eps) and dL/d den_t).  It depends on the current
 * device's SM count; it must be device memory, 256-byte aligned, and may be
 * reused by later calls on the same stream.
 */
LA_API size_t la_causal_backward_workspace_bytes(int B, int H, int N, int d, int dv,
                                                 la_dtype dt);

/*
 * Gradients of the causal forward (training through the recurrence:
 * "Linear Attention/es", "Entrenamiento: forma paralela").  Given
 * dy = dL/dy (float32, [B][H][N][dv]) for the output y of la_forward_causal
 * on the same q, k, v, eps and initial state, writes
 *   grad_q = dL/dq, grad_k = dL/dk   float32 [B][H][N][d]
 *   grad_v = dL/dv                   float32 [B][H][N][dv]
 * and, when grad_S_in / grad_z_in are non-NULL (both or neither), the
 * gradients with respect to the initial state, float32 [B][H][d][dv] and
 * [B][H][d] (also when S_in / z_in are NULL: the initial state is then the
 * zero state).  By the chain rule through the recurrence, with
 * D_t = max(den_t, eps) and g_t = dy_t / D_t:
 *   e_t            = -(dy_t . y_t) / D_t  when den_t >= eps, else 0
 *   dL/dphi(q_t)   = S_t g_t + z_t e_t
 *   dL/dphi(k_t)   = sum_{s>=t} phi(q_s) (g_s . v_t + e_s)
 *   dL/dv_t        = sum_{s>=t} g_s (phi(q_s) . phi(k_t))
 * and dL/dx = dL/dphi(x) * phi'(x), phi'(x) = 1 (x > 0), e^x (x <= 0).
 * y is not an input: the kernels recompute what they need.  Everything runs
 * in float32 on the CUDA cores.  All tensor pointers are device pointers,
 * 16-byte aligned; no output may overlap an input, the workspace or another
 * output.  Errors as la_forward_causal.
 */
LA_API la_status la_backward_causal(const void *q, const void *k, const void *v,
                                    const float *dy, float *grad_q, float *grad_k,
                                    float *grad_v, int B, int H, int N, int d, int dv,
                                    la_dtype dt, float eps, const float *S_in,
                                    const float *z_in, float *grad_S_in, float *grad_z_in,
                                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * Gradients of la_forward_causal_decay: as la_backward_causal for the
 * decayed recurrence S_t = gamma_h S_{t-1} + phi(k_t) v_t^T (z alike), with
 * gamma as in la_forward_causal_decay (DEVICE array of H floats in [0, 1],
 * 4-byte aligned; NULL: LA_ERR_INVALID_ARG).  The reverse state then obeys
 * Sh_t = phi(q_t) g_t^T + gamma_h Sh_{t+1}, and dL/dS_in = gamma_h Sh_1.
 * The gradient with respect to gamma is not computed.  Workspace: the size
 * la_causal_backward_workspace_bytes returns.
 */
LA_API la_status la_backward_causal_decay(const void *q, const void *k, const void *v,
                                          const float *dy, float *grad_q, float *grad_k,
                                          float *grad_v, int B, int H, int N, int d, int dv,
                                          la_dtype dt, float eps, const float *gamma,
                                          const float *S_in, const float *z_in,
                                          float *grad_S_in, float *grad_z_in, void *workspace,
                                          size_t workspace_bytes, void *stream);

/*
 * Device staging memory, in bytes, that la_forward_causal_host needs for
 * these sizes (0 for N == 0 or unsupported sizes).  Like the workspace size,
 * it depends on the current device's SM count.
 */
LA_API size_t la_causal_host_buffer_bytes(int B, int H, int N, int d, int dv, la_dtype dt);

/*
 * la_forward_causal on HOST buffers (no counterpart on the pages: it is the
 * path for callers whose q, k, v and y live in host memory).  q, k, v, y (and
 * the optional S_out, z_out, both or neither) are host pointers with the same
 * layouts as in la_forward_causal; the initial state is zero.  The call
 * copies the inputs to the device, runs the forward and copies y (and the
 * final state) back, pipelined over groups of heads: the upload of one group,
 * the kernels of the previous one and the download of the one before run at
 * once, on two streams the call creates and destroys plus `stream`, which the
 * work is ordered after.  It returns when the results are in host memory.
 * Page-locked host memory gives asynchronous full-speed copies; pageable
 * memory works but its copies are staged by the CUDA runtime and do not overlap.
 * dev_buf is caller-owned device memory of at least
 * la_causal_host_buffer_bytes(...) bytes, 256-byte aligned; its contents are
 * scratch.  Errors: as la_forward_causal (checked per group), LA_ERR_WORKSPACE
 * for a missing, short or misaligned dev_buf, LA_ERR_TIMEOUT when a bounded
 * wait of any group ran out (the outputs are then undefined).
 */
LA_API la_status la_forward_causal_host(const void *q, const void *k, const void *v, float *y,
                                        int B, int H, int N, int d, int dv, la_dtype dt,
                                        float eps, float *S_out, float *z_out, void *dev_buf,
                                        size_t dev_buf_bytes, void *stream);

/*
 * Non-causal forward ("Linear Attention/es", "Reformulación con núcleos"):
 *   S = sum_j phi(k_j) v_j^T, z = sum_j phi(k_j) over all N tokens, then
 *   y_i = phi(q_i)^T S / max(phi(q_i)^T z, eps) for every i.
 * S_out / z_out (both or neither) receive S and z.  N must be >= 1.
 */
LA_API la_status la_forward_noncausal(const void *q, const void *k, const void *v, float *y,
                               int B, int H, int N, int d, int dv, la_dtype dt, float eps,
                               float *S_out, float *z_out,
                               void *workspace, size_t workspace_bytes, void *stream);

/*
 * One recurrent decode step per (b, h), in place on the state ("Forma
 * recurrente e inferencia autorregresiva"; constant memory, no growing
 * cache):  S += phi(k) v^T,  z += phi(k),  y = phi(q)^T S / max(phi(q)^T z, eps).
 * q, k: [B][H][d]; v: [B][H][dv]; y: [B][H][dv] float32; S, z float32 in/out.
 */
LA_API la_status la_decode_step(const void *q, const void *k, const void *v, float *y,
                         float *S, float *z, int B, int H, int d, int dv, la_dtype dt,
                         float eps, void *stream);

/*
 * Non-causal forward that allocates nothing and takes no workspace.  The
 * pages have no counterpart to this entry point; it exists for callers that
 * cannot allocate device memory themselves, such as an operator or plugin
 * inside another framework that is handed only its input and output buffers,
 * or a latency-critical path that must not call cudaMalloc (which can
 * synchronise the whole device).  It computes exactly what
 * la_forward_noncausal computes, with the same arguments minus the workspace.
 *
 * Scratch: a fixed array of LA_NOALLOC_SCRATCH_BYTES compiled into the
 * library, resident on every GPU that loads the library until the process
 * exits.  Sizes whose scratch (la_noncausal_workspace_bytes) exceeds it are
 * rejected with LA_ERR_WORKSPACE before anything is launched.  The first call
 * on each device looks up the array's device address (a host-side runtime
 * call); make that first call before any stream capture begins.  All calls
 * share the array and leave their partial sums in it: calls that can overlap
 * on the GPU (different streams, different host threads) race and must be
 * ordered by the caller.  A bounded wait that runs out at run time is
 * recorded in the array's status word, which la_noalloc_status reads.
 */
#define LA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
LA_API la_status la_forward_noncausal_noalloc(const void *q, const void *k, const void *v,
                                              float *y, int B, int H, int N, int d, int dv,
                                              la_dtype dt, float eps, float *S_out, float *z_out,
                                              void *stream);

/*
 * Synchronise `stream` and report the run-time status that the last
 * la_forward_noncausal_noalloc call on the current device recorded in the
 * library's scratch array: LA_OK, or LA_ERR_TIMEOUT when one of its bounded
 * waits ran out (its outputs are then undefined).  The next such call clears
 * the record.  No counterpart on the pages; it exists because callers of the
 * no-allocation entry point hold no pointer to its scratch.  Allocates nothing.
 */
LA_API la_status la_noalloc_status(void *stream);

/*
 * Synchronise `stream` and report the run-time status recorded in a
 * workspace by the last call that used it: LA_OK, or LA_ERR_TIMEOUT when one
 * of its bounded waits ran out (its outputs are then undefined).  The next
 * call that uses the workspace clears the record.
 */
LA_API la_status la_workspace_status(const void *workspace, size_t workspace_bytes, void *stream);

/*
 * Test hook for the failure path (host side only, process-wide, not
 * thread-safe; no counterpart on the pages).  wait_limit_ns bounds every
 * wait of the tensor-core kernels (<= 0 restores the default of about one
 * second).  When drop_load_item >= 0, the tensor-core launch's work item
 * with that index (the CTA index: a (head, segment) item of
 * la_forward_causal, or a (head, query range) item of la_forward_noncausal)
 * announces its first tile copy on its mbarrier but never issues it, so every
 * wait on that tile runs out.  Nothing faults, traps or hangs: the waiter
 * records LA_ERR_TIMEOUT in the workspace header, the CTA unwinds (letting
 * the copies it did issue land and freeing its TMEM) and the call's outputs
 * are undefined; la_workspace_status then reports LA_ERR_TIMEOUT.  Pass
 * (-1, 0) to turn the hook off.
 */
LA_API void la_debug_set_fault(int drop_load_item, long long wait_limit_ns);

/*
 * Test hook (no counterpart on the pages): writes to out[i] (bf16) the
 * feature residual that the tensor-core kernels feed to the MMAs for the bf16
 * input x[i]: phi(x) - c rounded to bf16, phi(x) = elu(x) + 1 ("Mapas de
 * características"); c = 1 gives elu(x) itself.  x and out are DEVICE arrays
 * of n bfloat16 values (2-byte aligned, not overlapping); c must lie in
 * [0, 1] (the kernels use bf16 values of c), else LA_ERR_INVALID_ARG.
 * Enqueued on `stream`.
 */
LA_API la_status la_debug_feature_bf16(const void *x, void *out, long long n, float c,
                                       void *stream);

#ifdef __cplusplus
}
#endif
#endif /* LINATTN_H */
