/*
 * linattn — causal linear attention (Katharopoulos form, phi = elu + 1) for
 * NVIDIA B300 (sm_103a). C ABI: plain pointers and sizes only.
 *
 * The method (page "Attention_Kernel_Mask", allenlu2009.github.io, section
 * "Implementing Causality with Cumulative Sums"):
 *     z_t = z_{t-1} + phi(k_t)                 key sum, d
 *     M_t = M_{t-1} + phi(k_t) v_t^T           memory, d x dv
 *     out_t = phi(q_t)^T M_t / (phi(q_t)^T z_t + eps)
 * with one (M, z) per (batch, head), carried across calls as the compressive
 * memory of the page "Segment-Wise Attention" (github.com/beomi/infinitransformer,
 * issue 2). The three modes of the first page's table "Causal Attention
 * Training and Inferencing" are the three entry points: training forward (all
 * outputs), prompt/prefill (state plus last output) and generation (one step).
 *
 * Layouts (the [batch, heads, seq, head_dim] order of the KERPLE page's
 * Hugging Face attention code): q, k [B, H, T, d]; v, out [B, H, T, dv];
 * element (b, h, t, i) at b*sb + h*sh + t*st + i (contiguous: st = d or dv,
 * sh = T*st, sb = H*sh). State M [B, H, d, dv] float32 row-major, z [B, H, d]
 * float32, always contiguous.
 *
 * Ownership: the caller owns every buffer. All data pointers are DEVICE
 * pointers unless a parameter says otherwise. No call allocates device
 * memory. Scratch for the parallel schedules comes from a caller workspace
 * (the *_ex calls' `workspace`, or the buffer registered with
 * la_set_workspace for the plain calls); without one, the calls still run,
 * on schedules that need no scratch (one thread block per (batch, head)
 * carries that head's state through all T tokens).
 *
 * Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 * stream) and never synchronise. They return LA_OK or an error code for
 * problems found on the host before any launch; nothing is launched when a
 * call returns an error. Problems found on the device (a bounded wait that ran
 * out) are recorded in a per-device status word read by
 * la_get_last_device_status.
 *
 * Supported: dtype LA_F32 or LA_BF16 for q/k/v/out (same type for all four;
 * state is always float32); 1 <= d, dv <= 128 with d, dv multiples of 8;
 * T >= 1; chunk in {16, 32, 64, 128}. The bf16 tensor-core path takes
 * d, dv in {64, 128}, 16-byte aligned pointers and strides that are multiples of
 * 8 elements; other bf16 shapes run on the SIMT path. `chunk` sets the blocking
 * only (every chunk length gives the same outputs up to rounding): the
 * tensor-core path always works in 64-token chunks, the SIMT path (float32, and
 * bf16 shapes outside the tensor-core set) in chunks of the given length.
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* la_stream_t; /* identical to cudaStream_t */

typedef enum { LA_F32 = 0, LA_BF16 = 1 } la_dtype;

enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,   /* null/aliasing pointers, non-positive sizes, bad strides */
    LA_ERR_UNSUPPORTED = 2,   /* d, dv, chunk or dtype outside the supported set */
    LA_ERR_CUDA = 3,          /* a CUDA runtime/driver call or launch failed */
    LA_ERR_TIMEOUT = 4,       /* device status: a bounded wait inside a kernel ran out */
    LA_ERR_WORKSPACE = 5,     /* workspace pointer misaligned, or too small for la_causal_bwd */
    LA_ERR_SCRATCH_LIMIT = 6, /* la_prefill_state_noalloc: the problem needs more scratch than
                                 LA_NOALLOC_SCRATCH_BYTES */
    LA_ERR_BOUNDS = 7         /* device status, checked build only: an access outside a buffer's
                                 extent was found and skipped */
};

/* ---- training forward (mode 3 of the mode table: all outputs) -------------
 * Chunk-sequential form of the page's equation for "chunk sequential mode":
 * per chunk of `chunk` tokens, out = (phi(Q_c) M_{c-1} + ((phi(Q_c) phi(K_c)^T) o mask) V_c)
 * / (phi(Q_c) z_{c-1} + rowsum((phi(Q_c) phi(K_c)^T) o mask) + eps), mask = lower
 * triangle with diagonal; then M_c = M_{c-1} + phi(K_c)^T V_c, z_c = z_{c-1} + sum phi(K_c).
 *   q, k     [B,H,T,d]  dtype, read
 *   v        [B,H,T,dv] dtype, read
 *   out      [B,H,T,dv] dtype, written (all T outputs); must not alias q, k, v
 *   M_in,z_in  initial state [B,H,d,dv] / [B,H,d] float32, read; NULL = zero state
 *   M_out,z_out final state, written; NULL = not written; M_out may equal M_in
 *              (and z_out z_in): the update is then in place
 *   chunk    intra-chunk block length; eps >= 0 added to every denominator. */
int la_causal_fwd(const void* q, const void* k, const void* v, void* out,
                  const float* M_in, const float* z_in, float* M_out, float* z_out,
                  int B, int H, int64_t T, int d, int dv, int chunk, float eps,
                  la_dtype dtype, la_stream_t stream);

/* As la_causal_fwd, plus:
 *   strides    HOST pointer to 12 int64 element strides, or NULL for contiguous:
 *              {q_sb, q_sh, q_st, k_sb, k_sh, k_st, v_sb, v_sh, v_st, o_sb, o_sh, o_st}
 *              (innermost stride is 1). Lets a caller run one segment of a longer
 *              [B,H,T_total,d] tensor in place (the segment-wise use of the
 *              "Segment-Wise Attention" page) without copies.
 *   workspace  device scratch of workspace_bytes (256-byte aligned), or NULL/0.
 *              la_causal_fwd_workspace_size() gives the size that enables the
 *              sequence-split schedule; with less, the single-range schedule runs.
 *              On long sequences (at least 256 chunks of 64 tokens) split over two
 *              ranges per head, the first range hands its state to the second through
 *              the workspace inside the launch, which is then a cooperative launch (all
 *              blocks resident at once; it fits whenever that schedule is chosen). Calls
 *              that share one workspace must not run concurrently. */
int la_causal_fwd_ex(const void* q, const void* k, const void* v, void* out,
                     const float* M_in, const float* z_in, float* M_out, float* z_out,
                     int B, int H, int64_t T, int d, int dv, int chunk, float eps,
                     la_dtype dtype, const int64_t* strides,
                     void* workspace, size_t workspace_bytes, la_stream_t stream);

size_t la_causal_fwd_workspace_size(int B, int H, int64_t T, int d, int dv, int chunk,
                                    la_dtype dtype);

/* Segment-wise forward (the "Segment-Wise Attention" page: a sequence split into segments
 * with the compressive memory M, z carried from each segment to the next), in one call:
 * the outputs of all T tokens, which are those of la_causal_fwd over the whole sequence
 * (carrying the state across a segment boundary is the same recurrence step as across a
 * chunk boundary), and the state after every segment.
 *   q, k, v, out   contiguous [B,H,T,*] as for la_causal_fwd
 *   M_in, z_in     state before the first segment, [B,H,d,dv] / [B,H,d] float32; NULL = zero
 *   M_seg          [nseg][B,H,d,dv] float32, written: M after segment s (nseg = ceil(T / seg_len);
 *                  the last segment may be shorter, and its entry is the final state)
 *   z_seg          [nseg][B,H,d] float32, written: z after segment s
 *   seg_len        tokens per segment, a positive multiple of 64
 *   workspace      as for la_causal_fwd_ex (enables the sequence-split schedule)
 * bf16 with d, dv in {64, 128} (16-byte aligned q, k, v, out) runs as one launch of the
 * chunked kernel, the state staying on chip across segment boundaries and written at each;
 * other cases run one la_causal_fwd_ex per segment. Errors: LA_ERR_INVALID_ARG for null
 * M_seg or z_seg, a bad seg_len, or outputs that overlap each other or M_in / z_in; otherwise
 * as la_causal_fwd_ex. */
int la_causal_fwd_segments(const void* q, const void* k, const void* v, void* out,
                           const float* M_in, const float* z_in, float* M_seg, float* z_seg,
                           int B, int H, int64_t T, int d, int dv, int64_t seg_len, float eps,
                           la_dtype dtype, void* workspace, size_t workspace_bytes,
                           la_stream_t stream);

/* ---- other feature maps ------------------------------------------------------
 * The page "Attention_Kernel_Mask" lists positive random features (PRF) and orthogonal
 * random features (ORF) among the feature maps of its non-causal kernel discussion,
 * without printing them. They run through the same chunked kernels in two steps:
 *
 * la_feature_map_prf: out[r] = exp(W x_r - |x_r|^2 / 2) / sqrt(m) for every row r, the
 * positive random-feature map (ORF: the same map with rows of W orthogonal within blocks
 * of d, built by the caller). Tensor cores; bf16 only.
 *   x    [rows, d] bf16, contiguous rows (for q or k: rows = B*H*T), 16-byte aligned, read
 *   W    [m, d] bf16, 16-byte aligned, read
 *   out  [rows, m] bf16, written; must not alias x or W
 *   d, m in {64, 128}; otherwise LA_ERR_UNSUPPORTED.
 *
 * la_causal_fwd_mapped: la_causal_fwd_ex with q and k holding feature values already
 * (phi(q), phi(k) of any map, nonnegative for a positive denominator): the same
 * computation with the map applied by the caller instead of elu + 1; d is the feature
 * count. Same arguments, layouts and errors as la_causal_fwd_ex. */
int la_feature_map_prf(const void* x, const void* W, void* out, int64_t rows, int d, int m,
                       la_dtype dtype, la_stream_t stream);

int la_causal_fwd_mapped(const void* q, const void* k, const void* v, void* out,
                         const float* M_in, const float* z_in, float* M_out, float* z_out,
                         int B, int H, int64_t T, int d, int dv, int chunk, float eps,
                         la_dtype dtype, const int64_t* strides,
                         void* workspace, size_t workspace_bytes, la_stream_t stream);

/* ---- prefill (prompt mode: state plus last output) ---------------------------
 * Only the final state and the last token's output, as the mode table's note
 * on the prompt mode says (the state alone, with the output formed in the last
 * block); the key-
 * value sums are formed in parallel parts of `segment` tokens (the page's
 * remark that the sum can be done in parallel, e.g. as a tree) and added in
 * part order to M_in:  M_T = M_in + sum_p sum_{t in p} phi(k_t) v_t^T,
 * z_T = z_in + sum phi(k_t), out_last = phi(q_T)^T M_T / (phi(q_T)^T z_T + eps).
 *   out_last  [B,H,dv] dtype, written (may be NULL)
 *   M_out, z_out  written (may be NULL); M_out may equal M_in
 *   M_in, z_in, M_out, z_out  16-byte aligned when given (the parts are summed in
 *             16-byte vectors); otherwise LA_ERR_INVALID_ARG before any launch
 *   segment   tokens per part (0 = library choice). */
int la_prefill_state(const void* q, const void* k, const void* v, void* out_last,
                     const float* M_in, const float* z_in, float* M_out, float* z_out,
                     int B, int H, int64_t T, int d, int dv, int segment, float eps,
                     la_dtype dtype, la_stream_t stream);

int la_prefill_state_ex(const void* q, const void* k, const void* v, void* out_last,
                        const float* M_in, const float* z_in, float* M_out, float* z_out,
                        int B, int H, int64_t T, int d, int dv, int segment, float eps,
                        la_dtype dtype, const int64_t* strides,
                        void* workspace, size_t workspace_bytes, la_stream_t stream);

size_t la_prefill_workspace_size(int B, int H, int64_t T, int d, int dv, int segment,
                                 la_dtype dtype);

/* ---- prefill without any device allocation ---------------------------------
 * No counterpart on the method's pages: this entry point exists for callers that
 * cannot allocate device memory at all. Examples are a host framework that hands an
 * operator only its input and output buffers and owns every other byte of the GPU,
 * and latency-critical code that may not call cudaMalloc because it can synchronise
 * the device. Such callers cannot provide the workspace that la_prefill_state_ex
 * takes, and la_prefill_state without a registered workspace falls back to the slow
 * one-part schedule.
 *
 * Same arguments, results and layouts as la_prefill_state. The per-part sums go to a
 * scratch array of LA_NOALLOC_SCRATCH_BYTES that lives inside the library as a
 * statically sized device variable: every GPU that loads the library holds it until
 * the process exits. The call allocates nothing and runs the same kernels as
 * la_prefill_state_ex with a workspace of that size.
 *   - Returns LA_ERR_SCRATCH_LIMIT, without launching, when the scratch this call needs
 *     is more than LA_NOALLOC_SCRATCH_BYTES. It needs 4*(d*dv + d) bytes per part and
 *     head when T is split into more than one part (T > segment), plus 4*(d*dv + d) bytes
 *     per head when out_last is asked for without both M_out and z_out, and nothing
 *     otherwise. la_prefill_workspace_size counts both terms, so it is an upper bound.
 *     Raise `segment` to use fewer parts.
 *   - The first call on a device looks up the array's device address (with that device
 *     current), and so does the first call after a new context was created on the device
 *     (for example after cudaDeviceReset); make that first call before any stream capture.
 *   - All calls on a device share the one array and it keeps the last call's contents
 *     (every byte a call reads it has written first). Calls whose executions overlap on
 *     the GPU (different streams, not ordered) race on it: order them. */
#define LA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

int la_prefill_state_noalloc(const void* q, const void* k, const void* v, void* out_last,
                             const float* M_in, const float* z_in, float* M_out, float* z_out,
                             int B, int H, int64_t T, int d, int dv, int segment, float eps,
                             la_dtype dtype, la_stream_t stream);

/* ---- generation (pure sequential mode: one recurrent step) -----------------
 * For N independent streams x H heads, one token each:
 *   M <- M + phi(k) v^T;  z <- z + phi(k);  out = phi(q)^T M / (phi(q)^T z + eps)
 *   q, k [N,H,d], v [N,H,dv] dtype contiguous, read
 *   out  [N,H,dv] dtype, written
 *   M [N,H,d,dv], z [N,H,d] float32, read and written in place. */
int la_decode_step(const void* q, const void* k, const void* v, void* out,
                   float* M, float* z, int N, int H, int d, int dv, float eps,
                   la_dtype dtype, la_stream_t stream);

/* ---- training backward -----------------------------------------------------------
 * Gradients of the training forward (the mode table's training-backward row; the page
 * prints no formula, so these are the chain rule on the chunk form above). For a scalar
 * loss L with given dL/dout (dout), dL/dM_out and dL/dz_out, with D_t the denominator
 * and g_t = dout_t / D_t, e_t = -(g_t . out_t):
 *   dq_t = (M_t g_t + e_t z_t) o phi'(q_t)
 *   dk_i = (R_i v_i + r_i) o phi'(k_i),   dv_i = R_i^T phi(k_i)
 *   R_i = dM_out + sum_{t >= i} phi(q_t) g_t^T,   r_i = dz_out + sum_{t >= i} e_t phi(q_t)
 *   dM_in = R_0,   dz_in = r_0
 * (M_t, z_t include token t; phi'(x) = 1 for x > 0, exp(x) otherwise; "o" is the
 * elementwise product). The forward quantities are recomputed from q, k, v, M_in, z_in
 * in float32; nothing from the forward call is needed.
 *   q, k [B,H,T,d], v, dout [B,H,T,dv]  dtype, contiguous, 16-byte aligned, read
 *   M_in, z_in        float32, read (NULL = zero initial state)
 *   dM_out, dz_out    float32 [B,H,d,dv] / [B,H,d], read (NULL = zero)
 *   dq, dk [B,H,T,d], dv [B,H,T,dv]  dtype, contiguous, written; must not alias an input
 *                     or each other
 *   dM_in, dz_in      float32, written (NULL = not wanted); may equal dM_out / dz_out
 * Scratch: la_causal_bwd_workspace_size(B, H, T, d, dv) bytes (two float32 state records
 * per 64-token chunk and head, plus T*(dv+1) floats per head), from the registered
 * workspace (la_causal_bwd) or `workspace` (la_causal_bwd_ex, 256-byte aligned); with
 * less, the call returns LA_ERR_WORKSPACE and launches nothing. Six kernel launches on
 * `stream`. Supported: the forward's d, dv and dtypes; B*H <= 65535. */
int la_causal_bwd(const void* q, const void* k, const void* v, const void* dout,
                  const float* M_in, const float* z_in, const float* dM_out, const float* dz_out,
                  void* dq, void* dk, void* dv, float* dM_in, float* dz_in,
                  int B, int H, int64_t T, int d, int dv_dim, float eps, la_dtype dtype,
                  la_stream_t stream);

int la_causal_bwd_ex(const void* q, const void* k, const void* v, const void* dout,
                     const float* M_in, const float* z_in, const float* dM_out, const float* dz_out,
                     void* dq, void* dk, void* dv, float* dM_in, float* dz_in,
                     int B, int H, int64_t T, int d, int dv_dim, float eps, la_dtype dtype,
                     void* workspace, size_t workspace_bytes, la_stream_t stream);

size_t la_causal_bwd_workspace_size(int B, int H, int64_t T, int d, int dv);

/* ---- runtime -------------------------------------------------------------------
 * la_set_workspace: register (ptr, bytes) as the scratch of the plain calls on
 * the CURRENT device (the caller keeps ownership; NULL/0 unregisters). The
 * buffer must stay valid until the last call that may use it has completed,
 * and calls that share it must be ordered (same stream or synchronised). */
int la_set_workspace(void* ptr, size_t bytes);

/* Reads and clears this device's status word; synchronises `stream` first.
 * Returns LA_OK, or the device-side error recorded since the last read (LA_ERR_TIMEOUT
 * before LA_ERR_BOUNDS when both were). */
int la_get_last_device_status(la_stream_t stream);

const char* la_get_error_string(int code);

/* Failure-path self-test: launches one block that waits on a barrier nothing ever
 * completes, with a limit of `limit_cycles` SM clock cycles (1 .. 2^32); the wait runs
 * out, the kernel records LA_ERR_TIMEOUT in this device's status word and returns, so
 * the next la_get_last_device_status reports LA_ERR_TIMEOUT and the context stays usable.
 * It checks the same bounded-wait and status path that every kernel's mbarrier waits use.
 * Returns LA_ERR_INVALID_ARG for a limit outside that range. */
int la_selftest_wait_timeout(unsigned long long limit_cycles, la_stream_t stream);

/* Number of kernels the most recent call on this host thread launched. */
int la_last_launch_count(void);

/* 1 in the checked library (liblinattn_checked.so, built with LA_CHECKS=1), 0 otherwise. The
 * checked library tests every global-memory access of its SIMT, reduce, read-out and decode
 * kernels against the extent of the caller's buffer (from the shapes and strides given);
 * an access outside it is skipped and recorded, and la_get_last_device_status then returns
 * LA_ERR_BOUNDS. It is a debugging build: slower, same results otherwise. */
int la_checked_build(void);

#ifdef __cplusplus
}
#endif

#endif /* LINATTN_H */
