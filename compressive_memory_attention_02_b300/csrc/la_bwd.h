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
// (range of cpr 64-token chunks, b*H + h); nr ranges per head. states: one record per range
// (the state before it, after the prefix scan); rev: one record per range (its sums
// phi(Q)^T G and phi(Q)^T e from the dq sweep; after the reverse scan, the state gradient
// from every token after the range). Dn, E: D_t and e_t per token [B*H][T], written by the
// dq sweep and read by the dk/dv sweep.
struct BwdTcParams {
    void* dq;
    void* dk;
    void* dv;
    const float* states;
    float* rev;
    float* Dn;
    float* E;
    int B, H;
    int64_t T;
    int d, dv_dim, nch;
    int nr, cpr;
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
