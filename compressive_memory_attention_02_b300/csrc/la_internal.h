// Internal parameter blocks and launchers shared by the kernel files and the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/linattn.h"
#include "la_ptx.cuh"

// LA_CHECKS=1 builds the checked library: every global-memory access of the SIMT, reduce,
// read-out and decode kernels is tested against the extent of the caller's buffer first;
// an access outside it is skipped and STATUS_BOUNDS is recorded in the device status word
// (read back by la_get_last_device_status as LA_ERR_BOUNDS). Nothing traps. The tensor-core
// kernels' tiles are bounded by their tensor maps either way.
#ifndef LA_CHECKS
#define LA_CHECKS 0
#endif

namespace la {

// Element counts of the buffers a SIMT kernel may touch, for the checked build: q, k, v,
// out (strided spans), the initial and final state, and the workspace records.
struct Extents {
    int64_t q, k, v, o;
    int64_t M_in, z_in, M_out, z_out;
    int64_t ws;
};

// Element strides (innermost stride is 1) of q, k, v and out in [B, H, T, .].
struct Strides {
    int64_t q_sb, q_sh, q_st;
    int64_t k_sb, k_sh, k_st;
    int64_t v_sb, v_sh, v_st;
    int64_t o_sb, o_sh, o_st;
};

struct FwdParams {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    const float* M_in;
    const float* z_in;
    float* M_out;
    float* z_out;
    int B, H;
    int64_t T;
    int d, dv, chunk;
    float eps;
    Strides st;
    Extents ext;
    int* status;
    int phi_ident;         // q, k hold feature values already (no elu + 1)
};

// Per-part state sums. Record (bh, p) is at dst_M + (bh*nparts + p)*rec_M (d x dv,
// row-major) and dst_z + (bh*nparts + p)*rec_z (d).
struct PartsParams {
    const void* q;
    const void* k;
    const void* v;
    void* out_last;        // SIMT kernel only, nparts == 1: read-out of the last token
    const float* base_M;   // added to every record (used with nparts == 1), may be null
    const float* base_z;
    float* dst_M;
    float* dst_z;
    int64_t rec_M, rec_z;
    int B, H;
    int64_t T;
    int d, dv;
    int64_t part_len;
    int nparts;
    float eps;
    Strides st;
    Extents ext;           // M_out / z_out: the extents of dst_M / dst_z, records or state
    int* status;
    int phi_ident;         // k (and q) hold feature values already (no elu + 1)
};

struct ReduceParams {
    const float* base_M;   // may be null (zero state)
    const float* base_z;
    const float* parts_M;
    const float* parts_z;
    int64_t rec_M, rec_z;
    float* dst_M;
    float* dst_z;
    int BH, d, dv, nparts;
    Extents ext;           // ws: the part records
    int* status;
};

struct PrefillOutParams {
    const void* q;
    void* out;
    const float* M;
    const float* z;
    int B, H;
    int64_t T;
    int d, dv;
    float eps;
    Strides st;
    Extents ext;           // M_out, z_out: the final state read here
    int* status;
};

struct DecodeParams {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    float* M;
    float* z;
    int N, H, d, dv;
    float eps;
    Extents ext;           // q, k, v, o: the token tensors; M_out, z_out: the state
    int* status;
};

// Tensor-core forward: one block per (range, b*H + h). Range r processes the main
// chunks [main_begin(r), main_end(r)); its start state is M_in (or zero) plus, in the
// "parts" schedule, the aggregates of ranges 0..r-1 from parts_tc (records in ws),
// or, in the "fused two-range" schedule, the aggregate of chunks [0, split) that
// range 1 forms itself before its main chunks.
struct FwdTcParams {
    const float* M_in;
    const float* z_in;
    float* M_out;
    float* z_out;
    const float* ws;       // parts schedule: records of ranges 0..nranges-2
    int64_t rec;           // floats per record (d*dv + d); M at +0, z at +d*dv
    int nranges;
    int chunks_per_range;  // parts schedule
    int split;             // fused schedule: first chunk of range 1 (0 = parts schedule)
    int H;
    int64_t T;
    float eps;
    int* status;
    int phi_ident;         // q, k hold feature values already (no elu + 1)
    float* pub;            // fused schedule with a hand-off (or null): range 0's state after chunk
                           // `meet`, [B*H][rec] (M at +0, z at +d*dv), read by range 1
    int* pub_flag;         // [B*H] hand-off words: armed by range 1, published by range 0
    int meet;              // range 1 sums chunks meet+1 .. split-1 and adds range 0's state after meet
    float* M_seg;          // state after every segment of seg_chunks chunks: [nseg][B*H][d][dv] (or null)
    float* z_seg;          // [nseg][B*H][d] (or null)
    int seg_chunks;        // 64-token chunks per segment (> 0 when M_seg or z_seg is set)
};

// device status word bits
enum : int { STATUS_TIMEOUT = 1, STATUS_BOUNDS = 2 };

// Checked build: true iff elements [i, i + n) lie inside [0, len); otherwise STATUS_BOUNDS
// is recorded and the caller skips the access. The normal build compiles this to true.
__device__ __forceinline__ bool inb(int64_t i, int64_t n, int64_t len, int* status) {
#if LA_CHECKS
    if (i >= 0 && i + n <= len) return true;
    if (status) atomicOr(status, STATUS_BOUNDS);
    return false;
#else
    (void)i, (void)n, (void)len, (void)status;
    return true;
#endif
}

// SIMT launchers (la_simt.cu)
size_t fwd_simt_smem(int d, int dv, int C);
size_t parts_simt_smem(int d, int dv);
cudaError_t launch_fwd_simt(const FwdParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_parts_simt(const PartsParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_reduce_parts(const ReduceParams& p, cudaStream_t s);
cudaError_t launch_prefill_out(const PrefillOutParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams& p, bool bf16, cudaStream_t s);

// Tensor-core launchers (la_tc.cu). Maps are 4-D bf16 tensor maps {inner, T, H, B}
// with 64 x 64 boxes and 128-byte swizzle.
cudaError_t launch_parts_tc(const PartsParams& p, const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t s);
cudaError_t launch_fwd_tc(const FwdTcParams& p, int d, int dv, int B, const CUtensorMap& mq, const CUtensorMap& mk,
                          const CUtensorMap& mv, const CUtensorMap& mo, const CUtensorMap& mk2, const CUtensorMap& mv2,
                          cudaStream_t s);

// Positive random-feature map (la_fmap.cu): maps {d, rows} over x [rows, d] and {d, m} over
// W [m, d], both bf16; out [rows, m] bf16.
cudaError_t launch_fmap_prf(const CUtensorMap& mx, const CUtensorMap& mw, void* out, int64_t rows, int d, int m,
                            int* status, cudaStream_t s);

// Device address of the current device's status word (la_api.cu).
int device_status_word(int** status);

// Unique id (cuCtxGetId) of the context current on this thread, after making the
// current device's primary context current; LA_ERR_CUDA if it cannot be had.
int current_context_id(unsigned long long* id);

// Scratch bytes the prefill uses for this call when the scratch is large enough for its
// fastest schedule: the per-part state sums when T is split into more than one part, plus
// a final state when the last output is asked for without both M_out and z_out.
size_t prefill_scratch_bytes(int B, int H, int64_t T, int d, int dv, int segment, la_dtype dtype,
                             const void* out_last, const float* M_out, const float* z_out);

// Prefill behind la_prefill_state / la_prefill_state_ex (la_api.cu): with use_registered the
// buffer given to la_set_workspace is the scratch, otherwise (ws, ws_bytes).
int prefill_impl(const void* q, const void* k, const void* v, void* out_last, const float* M_in, const float* z_in,
                 float* M_out, float* z_out, int B, int H, int64_t T, int d, int dv, int segment, float eps,
                 la_dtype dtype, const int64_t* strides, void* ws, size_t ws_bytes, bool use_registered,
                 cudaStream_t stream);

}  // namespace la
