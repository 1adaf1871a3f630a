// Training backward (la_bwd.cu): parameter block and launchers.
#pragma once
#include "la_internal.h"

namespace la {

constexpr int BWD_CH = 64;  // tokens per block of the backward

// Workspace of the backward, in floats (each region starts on a 256-byte boundary):
//   states [B*H][nch][rec]  chunk sums, then (after the prefix scan) the state before
//                           chunk c (M at +0, z at +d*dv), float32
//   rev    [B*H][nch][rec]  chunk sums phi(Q_c)^T G_c and phi(Q_c)^T e_c; after the
//                           reverse scan, the state gradient from every token after chunk c
//   G      [B*H][T][dv]     g_t = dout_t / D_t
//   E      [B*H][T]         e_t = -(g_t . out_t)
struct BwdParams {
    const void* q;
    const void* k;
    const void* v;
    const void* dout;
    void* dq;
    void* dk;
    void* dv;
    float* states;
    float* rev;
    float* G;
    float* E;
    int B, H;
    int64_t T;
    int d, dv_dim, nch;
    int64_t rec;
    float eps;
};

struct ScanParams {
    float* rec;            // [B*H][nch][len]
    const float* base_M;   // [B*H][d*dv], may be null (zero)
    const float* base_z;   // [B*H][d], may be null (zero)
    float* total_M;        // written when non-null: base + sum of all records
    float* total_z;
    int BH, nch, d, dv;
    int64_t len;           // d*dv + d
    bool reverse;          // false: record c <- base + sum_{c' < c}; true: base + sum_{c' > c}
};

// Tensor-core sweeps (la_bwd_tc.cu), bf16 storage, d and dv in {64, 128}: one block per
// (range of cpr 64-token chunks, b*H + h); nr ranges per head; rev gets one record per
// range from the dq sweep (its sums phi(Q)^T G and phi(Q)^T e). Two ways to carry the
// state between ranges:
//   folded (scanned == 0, nr <= BWD_FOLD_RANGES): states holds the key-value sums of ranges
//     0 .. nr-2 ([B*H][nr-1] records from parts_tc); a block adds M_in, z_in (or dM_out,
//     dz_out) and the records before (after) its range itself, and range 0 of the dk/dv
//     sweep writes dM_in, dz_in. Any of these six may be null (zero / not written).
//   scanned (scanned == 1): states and rev are [B*H][nr] records already turned into the
//     state before / the state gradient after each range by the ordered scans of
//     la_bwd.cu, which also take the caller's arrays; the six pointers are unused.
// Dn, E: D_t and e_t per token [B*H][T], written by the dq sweep and read by the dk/dv sweep.
constexpr int BWD_FOLD_RANGES = 8;
struct BwdTcParams {
    void* dq;
    void* dk;
    void* dv;
    const float* states;
    float* rev;
    const float* M_in;
    const float* z_in;
    const float* dM_out;
    const float* dz_out;
    float* dM_in;
    float* dz_in;
    float* Dn;
    float* E;
    int B, H;
    int64_t T;
    int d, dv_dim, nch;
    int nr, cpr, scanned;
    int64_t rec;
    float eps;
    int* status;
};

cudaError_t launch_bwd_dq_tc(const BwdTcParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                             const CUtensorMap& mv, const CUtensorMap& mdo, cudaStream_t s);
cudaError_t launch_bwd_dkdv_tc(const BwdTcParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                               const CUtensorMap& mv, const CUtensorMap& mdo, cudaStream_t s);
// blocks of both sweeps that fit on one SM at once (shared memory, registers, TMEM)
int bwd_sweep_occupancy(int d, int dv);

size_t bwd_workspace_floats(int64_t BH, int64_t T, int d, int dv, size_t* off_rev, size_t* off_G, size_t* off_E);
cudaError_t launch_scan_states(const ScanParams& p, cudaStream_t s);
cudaError_t launch_bwd_sums(const BwdParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_dq(const BwdParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_dk(const BwdParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_bwd_dv(const BwdParams& p, bool bf16, cudaStream_t s);

}  // namespace la
