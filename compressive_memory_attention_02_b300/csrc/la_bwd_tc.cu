// Tensor-core (tcgen05 + TMEM + TMA) sweeps of the training backward, bf16 storage, f32
// accumulation. The page "Attention_Kernel_Mask" names the training-backward mode (table
// "Causal Attention Training and Inferencing") but prints no formula; these kernels apply
// the chain rule to the chunk form of that page's "chunk sequential mode" (mode 3), as the
// float32 kernels of la_bwd.cu do. For chunk c with the state (M, z) of every token before
// it and S = phi(Q_c) phi(K_c)^T kept for keys at or before the query (P):
//   D_t = phi(q_t).z + sum_j P_tj + eps,   out_t = (phi(q_t)^T M + sum_j P_tj v_j) / D_t
//   g_t = dout_t / D_t,   e_t = -(g_t . out_t),   dA_tj = g_t . v_j + e_t   (j <= t)
//   dphi(q_t) = M g_t + e_t z + sum_j dA_tj phi(k_j)
//   dphi(k_j) = sum_{t >= j} dA_tj phi(q_t) + R v_j + r,   dv_j = sum_{t >= j} P_tj g_t + R^T phi(k_j)
// with (R, r) = (sum phi(q_t) g_t^T, sum e_t phi(q_t)) over every token after the chunk, and
// dx = dphi(x) phi'(x), phi'(x) = min(phi(x), 1). out_t itself is never formed:
//   g_t . out_t = (phi(q_t) . (M g_t) + sum_j P_tj (g_t . v_j)) / D_t,
// and M g_t and g_t . v_j are the products dq needs anyway.
//
//   bwd_dq_sweep    one block per (range of chunks, b*H + h), chunks in order, the state
//                   (M in TMEM as f32, a bf16 copy in shared memory; z in shared memory)
//                   carried from chunk to chunk: dq, D_t and e_t per token, and the range's
//                   share of the state gradient (sum phi(Q)^T G, sum phi(Q)^T e)
//   bwd_dkdv_sweep  one block per (range, b*H + h), chunks in reverse, (R, r) carried the
//                   same way: G re-formed from dout and D_t, dk and dv
// The state before a range is the initial state plus the key-value sums of the ranges
// before it (parts_tc writes one record per range), and (R, r) after it the gradient of
// the final state plus the state-gradient sums of the ranges after it (one record per
// range from the first sweep). With a few ranges per head each block adds them up in
// order in its prologue and range 0 of the second sweep ends with the gradient of the
// initial state; with more, the ordered scans of la_bwd.cu do it between the launches.
//
// G and dA are formed in f32 and enter the dq sweep's products as two bf16 operands, the
// high part and the rounded remainder (x = hi + lo to ~16 bits), so that the cancellations
// in dq (M g + e z against the intra-chunk sum, and g . v_j + e inside dA) act on
// f32-accurate values. In the dk/dv sweep G stays split where it forms dA^T and sums into the
// state gradient R; dv's P^T G and dk's dA^T phi(Q) take the high parts alone. phi, V, dout,
// the carried states and P enter as bf16.
//
// 256 threads; warp w may touch only TMEM lane quarter w % 4. Per-token passes use warps 0
// and 1 (lanes 0-63 = the chunk's tokens), state copies warps 4-7. Thread 0 issues the TMA
// loads, the MMAs and their commits; every wait is a bounded mbarrier wait. Q and K are
// double-buffered (the next chunk's load is issued when a chunk starts); V and dout are
// reloaded as soon as their last reader is done.
//
// Operand layouts (128-byte swizzle, 1024-byte aligned): token tiles [64 tokens][64
// features] per atom as TMA loads them; a state tile (M or R, bf16) as [d rows][64 dv]
// blocks, stored right after a 64-row token atom (V, or the high part of G) so that
// [V; M] and [G; R] are each one K-major B operand of 64 + d rows; G, P, dA and their
// transposes [64][64] K-major, high and low parts in adjacent atoms. Every A-operand tile
// of 64 rows is followed by at least one atom of shared memory (an M = 128 MMA reads 64
// rows past it; those rows of the result are never used).
#include "la_bwd.h"
#include "la_tc_common.cuh"

namespace la {
namespace {

constexpr int BT = 256;  // threads per block

// Two f32 values as bf16 high parts (hi) and bf16 remainders (lo): x = hi + lo to ~16 bits.
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16(a, b);
    lo = pack_bf16(a - bf16lo(hi), b - bf16hi(hi));
}

// Row `row`, columns c0..c0+15 of a swizzled bf16 tile, as two 16-byte stores.
__device__ __forceinline__ void tile_put16(uint8_t* tile, int row, int c0, int bstride, const uint32_t* w) {
    uint8_t* r = tile + (c0 >> 6) * bstride + row * 128;
    const int ch = (c0 & 63) >> 3;
    *reinterpret_cast<uint4*>(r + ((ch ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(r + (((ch + 1) ^ (row & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
}

// Row `row`, columns c0..c0+7 of a swizzled bf16 tile as floats.
__device__ __forceinline__ void tile_get8(const uint8_t* tile, int row, int c0, int bstride, float* x) {
    const uint4 u = *reinterpret_cast<const uint4*>(tile + (c0 >> 6) * bstride + row * 128 +
                                                    ((((c0 & 63) >> 3) ^ (row & 7)) << 4));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) x[2 * e] = bf16lo(w[e]), x[2 * e + 1] = bf16hi(w[e]);
}

// Bounded wait by every thread of the block; false (and the status recorded) if it ran out.
__device__ __forceinline__ bool block_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status) {
    const bool ok = mbar_wait(bar, parity, abort_flag);
    if (!ok) record_timeout(status, abort_flag);
    return __syncthreads_and(ok) != 0;
}

// Two bounded waits by every thread, then one block-wide barrier.
__device__ __forceinline__ bool block_wait2(uint64_t* b1, uint32_t p1, uint64_t* b2, uint32_t p2,
                                            volatile int* abort_flag, int* status) {
    const bool ok = mbar_wait(b1, p1, abort_flag) && mbar_wait(b2, p2, abort_flag);
    if (!ok) record_timeout(status, abort_flag);
    return __syncthreads_and(ok) != 0;
}

__device__ __forceinline__ void sync_tc() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// 16 f32 columns of TMEM (this thread's lane) starting at column col
__device__ __forceinline__ void ld16f(uint32_t taddr, float* x) {
    uint32_t r[16];
    tmem_ld16(taddr, r);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) x[e] = __uint_as_float(r[e]);
}

// 32 f32 columns of TMEM (this thread's lane) starting at column col
__device__ __forceinline__ void ld32f(uint32_t taddr, float* x) {
    uint32_t r[32];
    tmem_ld32(taddr, r);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(r[e]);
}

// Warp roles: token warps 0, 1, 4, 5 reach TMEM lanes 0-63 (the chunk's tokens): row
// 32 (w % 4) + lane, column half w / 4. Aux warps 2, 3, 6, 7 (lanes 64-127, unused by the
// token accumulators) prepare the next chunk's operands; aux index 0..127.
__device__ __forceinline__ bool is_token_warp(int warp) { return (warp & 2) == 0; }
__device__ __forceinline__ int aux_index(int warp, int lane) { return (warp >> 2) * 64 + (warp & 1) * 32 + lane; }

// A carried state (D x DV, f32, lanes = rows) between memory, TMEM and its bf16 tile.
//
// sum_to_state: base (the caller's [D][DV] state, any alignment, may be null) plus the nrec
// records recs + k * rstride (workspace, 16-byte aligned) into TMEM and the tile. Warps w
// and w + 4 share lane quarter w % 4 and take one half of the columns each; the records
// are read two at a time so that their loads are in flight together.
template <int D, int DV>
__device__ __forceinline__ void sum_to_state(const float* base, const float* recs, int64_t rstride, int nrec,
                                             uint32_t tacc, uint8_t* tile, int bstride, int warp, int lane) {
    const int q = warp & 3, half = warp >> 2;
    if (32 * q >= D) return;
    const int i = 32 * q + lane;
    const uint32_t ta = tacc + ((uint32_t)(32 * q) << 16);
#pragma unroll 1
    for (int j0 = half * (DV / 2); j0 < (half + 1) * (DV / 2); j0 += 16) {
        float x[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = base ? base[(int64_t)i * DV + j0 + e] : 0.f;
        const float* rec = recs + (int64_t)i * DV + j0;
        int k = 0;
#pragma unroll 1
        for (; k + 2 <= nrec; k += 2) {
            float4 a[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                a[e] = __ldg(reinterpret_cast<const float4*>(rec + k * rstride) + e);
                a[4 + e] = __ldg(reinterpret_cast<const float4*>(rec + (k + 1) * rstride) + e);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[4 * e] += a[e].x + a[4 + e].x, x[4 * e + 1] += a[e].y + a[4 + e].y;
                x[4 * e + 2] += a[e].z + a[4 + e].z, x[4 * e + 3] += a[e].w + a[4 + e].w;
            }
        }
        if (k < nrec) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 a = __ldg(reinterpret_cast<const float4*>(rec + k * rstride) + e);
                x[4 * e] += a.x, x[4 * e + 1] += a.y, x[4 * e + 2] += a.z, x[4 * e + 3] += a.w;
            }
        }
        uint32_t r[16], w[8];
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(x[e]);
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = pack_bf16(x[2 * e], x[2 * e + 1]);
        tmem_st16(ta + j0, r);
        tile_put16(tile, i, j0, bstride, w);
    }
    tmem_wait_st();
}

// The same sum for the vector part (z or r) of feature i: base[i] + recs[k * rstride + i].
__device__ __forceinline__ float sum_vec(const float* base, const float* recs, int64_t rstride, int nrec, int i) {
    float a = base ? base[i] : 0.f;
    for (int k = 0; k < nrec; ++k) a += recs[k * rstride + i];
    return a;
}

// TMEM state -> its bf16 tile, split over every warp whose lane quarter holds state rows:
// quarter w % 4, column half w / 4.
template <int D, int DV>
__device__ __forceinline__ void state_to_tile_split(uint32_t tacc, uint8_t* tile, int bstride, int warp, int lane) {
    const int q = warp & 3, hf = warp >> 2;
    if (32 * q >= D) return;
    const int i = 32 * q + lane;
    const uint32_t ta = tacc + ((uint32_t)(32 * q) << 16);
#pragma unroll 1
    for (int j0 = hf * (DV / 2); j0 < (hf + 1) * (DV / 2); j0 += 32) {
        float x[32];
        ld32f(ta + j0, x);
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = pack_bf16(x[2 * e], x[2 * e + 1]);
        tile_put16(tile, i, j0, bstride, w);
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = pack_bf16(x[16 + 2 * e], x[16 + 2 * e + 1]);
        tile_put16(tile, i, j0 + 16, bstride, w);
    }
}

// TMEM state -> the caller's [D][DV] array (any alignment); warps w and w + 4 share lane
// quarter w % 4 and take one half of the columns each.
template <int D, int DV>
__device__ __forceinline__ void state_to_array(uint32_t tacc, float* dst, int warp, int lane) {
    const int q = warp & 3, half = warp >> 2;
    if (32 * q >= D) return;
    const int i = 32 * q + lane;
    const uint32_t ta = tacc + ((uint32_t)(32 * q) << 16);
#pragma unroll 1
    for (int j0 = half * (DV / 2); j0 < (half + 1) * (DV / 2); j0 += 16) {
        float x[16];
        ld16f(ta + j0, x);
#pragma unroll
        for (int e = 0; e < 16; ++e) dst[(int64_t)i * DV + j0 + e] = x[e];
    }
}

template <int D, int DV>
__device__ __forceinline__ void state_to_record(uint32_t tacc, float* rec, int warp, int lane) {
    const int q = warp - 4;
    if (q < 0 || 32 * q >= D) return;
    const int i = 32 * q + lane;
    const uint32_t ta = tacc + ((uint32_t)(32 * q) << 16);
#pragma unroll 1
    for (int j0 = 0; j0 < DV; j0 += 16) {
        float x[16];
        ld16f(ta + j0, x);
#pragma unroll
        for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(rec + (int64_t)i * DV + j0 + e) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
    }
}

// Aux warps (128 threads): out[i] += sum_t w_t tile[t][i] over the 64 rows of a swizzled
// [64][D] bf16 tile. Thread act takes 16-byte column chunk act % (D/8) of every
// (128 / (D/8))-th row; warp shuffles and shared-memory atomics combine the rows.
template <int D>
__device__ __forceinline__ void aux_weighted_colsum(const uint8_t* tile, const float* w, float* out, int act) {
    constexpr int CPR = D / 8, RG = 128 / CPR;
    const int c = act % CPR, g = act / CPR;
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int t = g; t < CH; t += RG) {
        float x[8];
        tile_get8(tile, t, 8 * c, ATOM, x);
        const float wt = w[t];
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] += x[e] * wt;
    }
#pragma unroll
    for (int o = CPR; o < 32; o <<= 1)
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] += __shfl_xor_sync(0xffffffffu, a[e], o);
    if ((act & 31) < CPR)
#pragma unroll
        for (int e = 0; e < 8; ++e) atomicAdd(&out[8 * c + e], a[e]);
}

// Outstanding TMA / MMA phases of one barrier: issued by thread 0, waited by the block.
struct Pending {
    uint32_t issued, waited;
};

// After a wait ran out: let every copy and MMA still in flight land (bounded) before the
// block releases its shared memory and TMEM.
__device__ __forceinline__ void drain(uint64_t* bars, Pending* pend, int n) {
    for (int b = 0; b < n; ++b)
        for (uint32_t ph = pend[b].waited; ph < pend[b].issued; ++ph) mbar_wait_drain(&bars[b], ph & 1);
}

}  // namespace

// Ranges: block (r, bh) takes chunks [r * cpr, min((r + 1) * cpr, nch)).
__device__ __forceinline__ void range_of(const BwdTcParams& p, int r, int& c0, int& n) {
    c0 = r * p.cpr;
    n = (int)min64(p.cpr, (int64_t)p.nch - c0);
}

// ================================================================================ dq sweep
template <int D, int DV>
struct DqLayout {
    static constexpr int VMB = ATOM + D * 128;            // one 64-dv block of [V; M]
    static constexpr int QT = 0;                          // phi(Q), 2 stages of D/64 atoms
    static constexpr int KT = QT + 2 * (D / 64) * ATOM;   // phi(K), 2 stages
    static constexpr int VM = KT + 2 * (D / 64) * ATOM;   // [V; M], DV/64 blocks
    static constexpr int OT = VM + DV / 64 * VMB;         // dout, DV/64 atoms
    static constexpr int GT = OT + DV / 64 * ATOM;        // G high (DV/64 atoms), then low
    static constexpr int AT = GT + 2 * (DV / 64) * ATOM;  // dA (masked, + e) high, then low
    static constexpr int PF = AT + 2 * ATOM;              // P as f32 [64][64], 16-byte chunks swizzled
    static constexpr int DEN = PF + 64 * 64 * 4;          // 64 floats: D_t
    static constexpr int ZQ = DEN + 256;                  // 64 floats: phi(q_t) . z
    static constexpr int EV = ZQ + 256;                   // 64 floats: e_t
    static constexpr int XS = EV + 256;                   // 2 x 64 floats: per-half partial row sums
    static constexpr int ZF = XS + 512;                   // 2 x D floats: z before the chunk, by chunk parity
    static constexpr int ZP = ZF + 2 * D * 4;             // 4 x D floats: per-warp column sums of phi(K)
    static constexpr int RS = ZP + 4 * D * 4;             // D floats: the range's sum of e_t phi(q_t)
    static constexpr int BAR = RS + D * 4;                // ld_qk[2], ld_v, ld_o, mma_done
    static constexpr int MISC = BAR + 5 * 8;
    static constexpr int ALLOC = MISC + 16 + 1024;
    // TMEM columns
    static constexpr uint32_t TA = 0;                     // S, then dA (64) | dphi(Q) (D): one MMA target
    static constexpr uint32_t TQ = 64;
    static constexpr uint32_t TR = 64 + D;                // sum over the range of phi(Q)^T G (DV), lanes = features
    static constexpr uint32_t TM = TR + DV;               // the state M (DV), lanes = features
    static constexpr uint32_t NCOL = TM + DV <= 256 ? 256 : 512;
};

// Chunk steps of the dq sweep (thread 0 issues loads and MMAs; token warps 0, 1, 4, 5
// run the per-token passes on column halves; aux warps 2, 3, 6, 7 prepare chunk idx + 1):
//   start   wait Q, K (phi already applied), V
//   g1      S = phi(Q) phi(K)^T, M += phi(K)^T V           | aux: z after the chunk
//   P pass  P (f32), D_t, G = dout / D (hi, lo)             | aux: phi(Q) of the next chunk
//   g2      [dA | dphi(Q)] = G [V; M]^T, R_range += phi(Q)^T G
//   e pass  e_t, dA + e masked (hi, lo)                     | aux: phi(K) of the next chunk
//   g3      dphi(Q) += dA phi(K)        | token: M to its bf16 tile; aux: r_range, phi(q).z next
//   end     dq = (dphi(Q) + e z) phi'(q), D_t, e_t to the workspace
template <int D, int DV>
__global__ void __launch_bounds__(BT, D == 64 && DV == 64 ? 2 : 1)
    bwd_dq_sweep_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                        const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                        BwdTcParams p) {
    using L = DqLayout<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    enum { B_QK0 = 0, B_QK1 = 1, B_V = 2, B_O = 3, B_MMA = 4, NB = 5 };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
    float* den = reinterpret_cast<float*>(sm + L::DEN);
    float* zq = reinterpret_cast<float*>(sm + L::ZQ);
    float* ev = reinterpret_cast<float*>(sm + L::EV);
    float* xs = reinterpret_cast<float*>(sm + L::XS);
    float* zf = reinterpret_cast<float*>(sm + L::ZF);
    float* zpart = reinterpret_cast<float*>(sm + L::ZP);
    float* rsum = reinterpret_cast<float*>(sm + L::RS);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool tok = is_token_warp(warp);
    const int trow = 32 * (warp & 3) + lane, thalf = warp >> 2;  // token warps: row, column half
    const int act = aux_index(warp, lane);                         // aux warps
    const int r = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H;
    int c0, n;
    range_of(p, r, c0, n);
    const int64_t rec_i = (int64_t)bh * p.nr + r;
    Pending pend[NB] = {};

    if (tid == 0) {
        for (int i = 0; i < NB; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
        tma_prefetch_desc(&mdo);
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, L::NCOL);
        tmem_relinquish();
    }
    sync_tc();
    const uint32_t tmem = *tmem_holder;

    const uint64_t pol = l2_evict_first_policy();
    auto load_qk = [&](int idx) {  // thread 0
        const int s = idx & 1;
        const int t0 = (c0 + idx) * CH;
        mbar_expect_tx(&bars[B_QK0 + s], 2 * D * CH * 2);
        for (int a = 0; a < D / 64; ++a) {
            tma_load_4d_hint(sm + L::QT + (s * (D / 64) + a) * ATOM, &mq, &bars[B_QK0 + s], a * 64, t0, h, b, pol);
            tma_load_4d_hint(sm + L::KT + (s * (D / 64) + a) * ATOM, &mk, &bars[B_QK0 + s], a * 64, t0, h, b, pol);
        }
        ++pend[B_QK0 + s].issued;
    };
    auto load_v = [&](int idx) {
        const int t0 = (c0 + idx) * CH;
        mbar_expect_tx(&bars[B_V], DV * CH * 2);
        for (int a = 0; a < DV / 64; ++a)
            tma_load_4d_hint(sm + L::VM + a * L::VMB, &mv, &bars[B_V], a * 64, t0, h, b, pol);
        ++pend[B_V].issued;
    };
    auto load_o = [&](int idx) {
        const int t0 = (c0 + idx) * CH;
        mbar_expect_tx(&bars[B_O], DV * CH * 2);
        for (int a = 0; a < DV / 64; ++a)
            tma_load_4d_hint(sm + L::OT + a * ATOM, &mdo, &bars[B_O], a * 64, t0, h, b, pol);
        ++pend[B_O].issued;
    };
    auto valid_of = [&](int idx) { return (int)min64(CH, p.T - (int64_t)(c0 + idx) * CH); };
    auto qtile = [&](int idx) { return sm + L::QT + (idx & 1) * (D / 64) * ATOM; };
    auto ktile = [&](int idx) { return sm + L::KT + (idx & 1) * (D / 64) * ATOM; };
    // aux warps: wait for chunk idx's Q and K (bounded), then phi on Q in place
    auto aux_phi_q = [&](int idx) {
        if (!mbar_wait(&bars[B_QK0 + (idx & 1)], (idx >> 1) & 1, abort_flag)) {
            record_timeout(p.status, abort_flag);
            return;
        }
        phi_tile<D, 128>(qtile(idx), ATOM, valid_of(idx), act, nullptr);
        fence_proxy_async_smem();
    };
    // aux warps: phi on chunk idx's K in place, its column sums to zpart
    auto aux_phi_k = [&](int idx) {
        float cs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        phi_tile<D, 128>(ktile(idx), ATOM, valid_of(idx), act, cs);
        colsum_to_smem<D>(cs, zpart, act);
        fence_proxy_async_smem();
    };
    // aux warps 6-7: phi(q_t) . z for chunk idx (z before it in zb)
    auto aux_zq = [&](int idx, const float* zb) {
        if (act < 64) return;
        const int t = act - 64;
        const uint8_t* qt = qtile(idx);
        float a = 0.f;
#pragma unroll 4
        for (int i0 = 0; i0 < D; i0 += 8) {
            float x[8];
            tile_get8(qt, t, i0, ATOM, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) a += x[e] * zb[i0 + e];
        }
        zq[t] = a;
    };

    if (tid == 0 && n > 0) {
        load_qk(0);
        load_v(0);
        load_o(0);
    }
    // the state before the range (the initial state plus the key-value sums of the ranges
    // before it; one record when scanned): M into TMEM and its bf16 tile, z; the range's
    // sums start at 0
    const float* recs = p.scanned ? p.states + rec_i * p.rec : p.states + (int64_t)bh * (p.nr - 1) * p.rec;
    const int nbefore = p.scanned ? 1 : r;
    const float* Mb = p.M_in ? p.M_in + (int64_t)bh * D * DV : nullptr;
    sum_to_state<D, DV>(Mb, recs, p.rec, nbefore, tmem + L::TM, sm + L::VM + ATOM, L::VMB, warp, lane);
    if (tid < D) {
        zf[tid] = sum_vec(p.z_in ? p.z_in + (int64_t)bh * D : nullptr, recs + D * DV, p.rec, nbefore, tid);
        rsum[tid] = 0.f;
    }
    if (!tok && n > 0) {  // the first chunk's operands, alongside the sums above
        aux_phi_q(0);
        aux_phi_k(0);
    }
    fence_proxy_async_smem();
    sync_tc();
    if (!tok && n > 0) aux_zq(0, zf);

    auto off = [](uint32_t bytes) { return (uint64_t)(bytes >> 4); };
    const uint64_t dVMk = sdesc_sw128(smem_u32(sm + L::VM), 16, 1024);      // [V; M], K-major (K = dv)
    const uint64_t dVm = sdesc_sw128(smem_u32(sm + L::VM), L::VMB, 1024);   // V, MN-major (K = tokens)
    const uint64_t dGk = sdesc_sw128(smem_u32(sm + L::GT), 16, 1024);       // G, K-major (K = dv)
    const uint64_t dGm = sdesc_sw128(smem_u32(sm + L::GT), ATOM, 1024);     // G, MN-major (K = tokens)
    const uint64_t dAk = sdesc_sw128(smem_u32(sm + L::AT), 16, 1024);
    constexpr uint32_t GLO = (DV / 64) * ATOM;  // offset of the low parts of G
    uint32_t mph = 0;                           // MMA-completion phases waited
    bool ok = true;

    for (int idx = 0; idx < n && ok; ++idx) {
        const int s = idx & 1;
        const int64_t t0 = (int64_t)(c0 + idx) * CH;
        const int valid = valid_of(idx);
        const bool more = idx + 1 < n;
        uint8_t* qt = qtile(idx);
        uint8_t* kt = ktile(idx);
        const float* zc = zf + s * D;
        float* zn = zf + (s ^ 1) * D;
        // (this barrier also ends the previous chunk: its end phase has read the stage that the
        // next prefetch overwrites, and z before this chunk)
        ok = block_wait2(&bars[B_QK0 + s], (idx >> 1) & 1, &bars[B_V], idx & 1, abort_flag, p.status);
        if (!ok) break;
        ++pend[B_QK0 + s].waited, ++pend[B_V].waited;
        if (tid == 0 && more) load_qk(idx + 1);
        tc_fence_after();
        const uint64_t dQk = sdesc_sw128(smem_u32(qt), 16, 1024);     // phi(Q), K-major (K = d)
        const uint64_t dQm = sdesc_sw128(smem_u32(qt), ATOM, 1024);   // phi(Q), MN-major (M = d, K = tokens)
        const uint64_t dKk = sdesc_sw128(smem_u32(kt), 16, 1024);
        const uint64_t dKm = sdesc_sw128(smem_u32(kt), ATOM, 1024);
        // ---- g1: S = phi(Q) phi(K)^T; M += phi(K)^T V (the state after the chunk, in TMEM)
        if (tid == 0) {
            constexpr uint32_t id_s = idesc_bf16(128, CH, 0, 0);
            constexpr uint32_t id_m = idesc_bf16(128, DV, 1, 1);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t o = (ks >> 2) * ATOM + (ks & 3) * 32;
                mma_bf16_ss(tmem + L::TA, dQk + off(o), dKk + off(o), id_s, ks != 0);
            }
#pragma unroll
            for (int ks = 0; ks < CH / 16; ++ks)
                mma_bf16_ss(tmem + L::TM, dKm + off(ks * 2048), dVm + off(ks * 2048), id_m, 1);
            mma_commit(&bars[B_MMA]);
            ++pend[B_MMA].issued;
        }
        if (!tok && act < D) {  // z after the chunk
            float a = zc[act];
#pragma unroll
            for (int w = 0; w < 4; ++w) a += zpart[w * D + act];
            zn[act] = a;
        }
        ok = block_wait2(&bars[B_MMA], mph & 1, &bars[B_O], idx & 1, abort_flag, p.status);
        if (!ok) break;
        ++mph, ++pend[B_MMA].waited, ++pend[B_O].waited;
        tc_fence_after();
        // ---- P pass: P (f32), D_t, G = dout / D (high and low parts)
        if (tok) {
            const int t = trow, hf = thalf;
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            uint8_t* prow = sm + L::PF + t * 256;
            float x[32];
            ld32f(tmem + L::TA + lb + 32 * hf, x);
            float rs = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                x[e] = (32 * hf + e <= t) ? x[e] : 0.f;
                rs += x[e];
            }
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const int ch = (32 * hf + e) >> 2;
                *reinterpret_cast<float4*>(prow + ((ch ^ (t & 15)) << 4)) = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
            }
            xs[hf * 64 + t] = rs;
            named_bar_sync(1, 128);
            const float dt = zq[t] + xs[t] + xs[64 + t] + p.eps;
            if (hf == 0) den[t] = dt;
            const float rd = t < valid ? 1.f / dt : 0.f;  // rows past the end: g = 0
#pragma unroll 1
            for (int j0 = hf * (DV / 2); j0 < (hf + 1) * (DV / 2); j0 += 16) {
                float o[16];
                tile_get8(sm + L::OT, t, j0, ATOM, o);
                tile_get8(sm + L::OT, t, j0 + 8, ATOM, o + 8);
                uint32_t gh[8], gl[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) split2(o[2 * e] * rd, o[2 * e + 1] * rd, gh[e], gl[e]);
                tile_put16(sm + L::GT, t, j0, ATOM, gh);
                tile_put16(sm + L::GT + GLO, t, j0, ATOM, gl);
            }
            fence_proxy_async_smem();
        } else if (more) {
            aux_phi_q(idx + 1);
        }
        sync_tc();
        // ---- g2: [dA | dphi(Q)] = G [V; M]^T; the range's phi(Q)^T G
        if (tid == 0) {
            if (more) load_o(idx + 1);
            constexpr uint32_t id_am = idesc_bf16(128, CH + D, 0, 0);
            constexpr uint32_t id_r = idesc_bf16(128, DV, 1, 1);
#pragma unroll
            for (int ks = 0; ks < DV / 16; ++ks) {
                const uint32_t go = (ks >> 2) * ATOM + (ks & 3) * 32;
                const uint64_t bo = off((ks >> 2) * L::VMB + (ks & 3) * 32);
                mma_bf16_ss(tmem + L::TA, dGk + off(go), dVMk + bo, id_am, ks != 0);
                mma_bf16_ss(tmem + L::TA, dGk + off(GLO + go), dVMk + bo, id_am, 1);
            }
#pragma unroll
            for (int ks = 0; ks < CH / 16; ++ks) {
                mma_bf16_ss(tmem + L::TR, dQm + off(ks * 2048), dGm + off(ks * 2048), id_r, idx != 0 || ks != 0);
                mma_bf16_ss(tmem + L::TR, dQm + off(ks * 2048), dGm + off(GLO + ks * 2048), id_r, 1);
            }
            mma_commit(&bars[B_MMA]);
            ++pend[B_MMA].issued;
        }
        ok = block_wait(&bars[B_MMA], mph & 1, abort_flag, p.status);
        if (!ok) break;
        ++mph, ++pend[B_MMA].waited;
        tc_fence_after();
        if (tid == 0 && more) load_v(idx + 1);  // V's last readers (g1, g2) are done
        // ---- e pass: e_t = -(phi(q_t) . M g_t + sum_j P_tj dA_tj) / D_t; dA + e masked (hi, lo)
        if (tok) {
            const int t = trow, hf = thalf;
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            float a = 0.f;
#pragma unroll 1
            for (int i0 = hf * (D / 2); i0 < (hf + 1) * (D / 2); i0 += 32) {
                float x[32];
                ld32f(tmem + L::TQ + lb + i0, x);
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    float f[8];
                    tile_get8(qt, t, i0 + c, ATOM, f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) a += f[e] * x[c + e];
                }
            }
            float da[32];
            ld32f(tmem + L::TA + lb + 32 * hf, da);
            const uint8_t* prow = sm + L::PF + t * 256;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const int ch = (32 * hf + e) >> 2;
                const float4 pv = *reinterpret_cast<const float4*>(prow + ((ch ^ (t & 15)) << 4));
                a += pv.x * da[e] + pv.y * da[e + 1] + pv.z * da[e + 2] + pv.w * da[e + 3];
            }
            xs[hf * 64 + t] = a;
            named_bar_sync(1, 128);
            const float e = t < valid ? -(xs[t] + xs[64 + t]) / den[t] : 0.f;
            if (hf == 0) ev[t] = e;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                uint32_t ah[8], al[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int c = 32 * hf + 16 * g + 2 * q;
                    const float a0 = c <= t ? da[16 * g + 2 * q] + e : 0.f;
                    const float a1 = c + 1 <= t ? da[16 * g + 2 * q + 1] + e : 0.f;
                    split2(a0, a1, ah[q], al[q]);
                }
                tile_put16(sm + L::AT, t, 32 * hf + 16 * g, ATOM, ah);
                tile_put16(sm + L::AT + ATOM, t, 32 * hf + 16 * g, ATOM, al);
            }
            fence_proxy_async_smem();
        } else if (more) {
            aux_phi_k(idx + 1);
        }
        sync_tc();
        // ---- g3: dphi(Q) += dA phi(K)
        if (tid == 0) {
            constexpr uint32_t id_q = idesc_bf16(128, D, 0, 1);
#pragma unroll
            for (int ks = 0; ks < CH / 16; ++ks) {
                mma_bf16_ss(tmem + L::TQ, dAk + off(ks * 32), dKm + off(ks * 2048), id_q, 1);
                mma_bf16_ss(tmem + L::TQ, dAk + off(ATOM + ks * 32), dKm + off(ks * 2048), id_q, 1);
            }
            mma_commit(&bars[B_MMA]);
            ++pend[B_MMA].issued;
        }
        // meanwhile: the state after the chunk to its bf16 tile (g3 does not read it); the
        // range's sum of e_t phi(q_t) and phi(q).z of the next chunk (aux warps)
        state_to_tile_split<D, DV>(tmem + L::TM, sm + L::VM + ATOM, L::VMB, warp, lane);
        if (!tok) {
            aux_weighted_colsum<D>(qt, ev, rsum, act);
            if (more) aux_zq(idx + 1, zn);
        }
        fence_proxy_async_smem();
        ok = block_wait(&bars[B_MMA], mph & 1, abort_flag, p.status);
        if (!ok) break;
        ++mph, ++pend[B_MMA].waited;
        tc_fence_after();
        // ---- end: dq = (dphi(Q) + e z) phi'(q), column half per warp; D_t and e_t to the
        // workspace. The TMEM loads are warp-wide; only rows inside the sequence are stored.
        if (tok) {
            const int t = trow;
            const bool store = t < valid;
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            const float e = ev[t];
            __nv_bfloat16* dq = reinterpret_cast<__nv_bfloat16*>(p.dq) + ((int64_t)bh * p.T + t0 + t) * D;
#pragma unroll 1
            for (int i0 = thalf * (D / 2); i0 < (thalf + 1) * (D / 2); i0 += 32) {
                float x[32];
                ld32f(tmem + L::TQ + lb + i0, x);
#pragma unroll
                for (int g = 0; g < 32; g += 8) {
                    float f[8];
                    tile_get8(qt, t, i0 + g, ATOM, f);
                    uint32_t w[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        w[q] = pack_bf16((x[g + 2 * q] + e * zc[i0 + g + 2 * q]) * fminf(f[2 * q], 1.f),
                                         (x[g + 2 * q + 1] + e * zc[i0 + g + 2 * q + 1]) * fminf(f[2 * q + 1], 1.f));
                    if (store) *reinterpret_cast<uint4*>(dq + i0 + g) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            if (thalf == 0 && store) {
                p.Dn[(int64_t)bh * p.T + t0 + t] = den[t];
                p.E[(int64_t)bh * p.T + t0 + t] = e;
            }
        }
        tc_fence_before();  // (the next chunk's first wait is the barrier)
    }
    if (ok && n > 0) {
        // the range's share of the state gradient: sum phi(Q)^T G (TMEM) and sum phi(Q)^T e
        float* rrec = p.rev + rec_i * p.rec;
        state_to_record<D, DV>(tmem + L::TR, rrec, warp, lane);
        if (tid < D) rrec[D * DV + tid] = rsum[tid];
    } else if (!ok && tid == 0) {
        drain(bars, pend, NB);
    }
    sync_tc();
    if (warp == 0) tmem_dealloc(tmem, L::NCOL);
}

// ================================================================================ dk, dv sweep
template <int D, int DV>
struct DkvLayout {
    static constexpr int GRB = ATOM + D * 128;            // one 64-dv block of [G high; R]
    // A operands (phi, P^T, dA^T, V) come before tiles that are only B operands or plain
    // data, so the rows an M = 128 MMA reads past each of them stay inside the allocation
    static constexpr int QT = 0;                          // phi(Q), 2 stages
    static constexpr int KT = QT + 2 * (D / 64) * ATOM;   // phi(K), 2 stages
    static constexpr int PT = KT + 2 * (D / 64) * ATOM;   // P^T [64 keys][64 queries] bf16 (+ one atom read past)
    static constexpr int AT = PT + 2 * ATOM;              // dA^T (masked, + e) high, then low
    static constexpr int VT = AT + 2 * ATOM;              // V, DV/64 atoms
    static constexpr int OT = VT + DV / 64 * ATOM;        // dout, DV/64 atoms
    static constexpr int GR = OT + DV / 64 * ATOM;        // [G high; R], DV/64 blocks
    static constexpr int GL = GR + DV / 64 * GRB;         // G low, DV/64 atoms
    static constexpr int DN = GL + DV / 64 * ATOM;        // 2 x 64 floats: D_t by chunk parity
    static constexpr int EV = DN + 512;                   // 2 x 64 floats: e_t
    static constexpr int RV = EV + 512;                   // 2 x D floats: r after the chunk, by chunk parity
    static constexpr int BAR = RV + 2 * D * 4;            // ld_qk[2], ld_v, ld_o, mma_done
    static constexpr int MISC = BAR + 5 * 8;
    static constexpr int ALLOC = MISC + 16 + 1024;
    static constexpr uint32_t TS = 0;                     // S^T (64), then dv (DV)
    static constexpr uint32_t TA = DV > 64 ? DV : 64;     // dA^T (64) | dphi(K) (D): one MMA target
    static constexpr uint32_t TK = TA + 64;
    static constexpr uint32_t TRR = TK + D;               // R (DV), lanes = features
    static constexpr uint32_t NCOL = TRR + DV <= 256 ? 256 : 512;
};

// Chunk steps of the dk/dv sweep (chunks in reverse; roles as in the dq sweep):
//   start   wait Q, K (phi already applied), dout; G = dout / D (hi, lo), column halves
//   g1      S^T = phi(K) phi(Q)^T, [dA^T | V R^T] = V [G; R]^T, R += phi(Q)^T G
//   mask    P^T, dA^T + e masked to queries at or after the key (bf16)  | aux: phi(Q) next
//   g2      dv = P^T G + phi(K) R, dphi(K) += dA^T phi(Q)      | aux: phi(K) next, r
//   end     dk = (dphi(K) + r) phi'(k), dv; R to its bf16 tile
template <int D, int DV>
__global__ void __launch_bounds__(BT, D == 64 && DV == 64 ? 2 : 1)
    bwd_dkdv_sweep_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                          const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                          BwdTcParams p) {
    using L = DkvLayout<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    enum { B_QK0 = 0, B_QK1 = 1, B_V = 2, B_O = 3, B_MMA = 4, NB = 5 };
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
    float* dn = reinterpret_cast<float*>(sm + L::DN);
    float* evs = reinterpret_cast<float*>(sm + L::EV);
    float* rv = reinterpret_cast<float*>(sm + L::RV);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool tok = is_token_warp(warp);
    const int trow = 32 * (warp & 3) + lane, thalf = warp >> 2;
    const int act = aux_index(warp, lane);
    const int r = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H;
    int c0, n;
    range_of(p, r, c0, n);
    const int64_t rec_i = (int64_t)bh * p.nr + r;
    Pending pend[NB] = {};
    auto chunk_of = [&](int idx) { return c0 + n - 1 - idx; };  // the range in reverse

    if (tid == 0) {
        for (int i = 0; i < NB; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
        tma_prefetch_desc(&mdo);
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, L::NCOL);
        tmem_relinquish();
    }
    sync_tc();
    const uint32_t tmem = *tmem_holder;

    const uint64_t pol = l2_evict_first_policy();
    auto load_qk = [&](int idx) {
        const int s = idx & 1;
        const int t0 = chunk_of(idx) * CH;
        mbar_expect_tx(&bars[B_QK0 + s], 2 * D * CH * 2);
        for (int a = 0; a < D / 64; ++a) {
            tma_load_4d_hint(sm + L::QT + (s * (D / 64) + a) * ATOM, &mq, &bars[B_QK0 + s], a * 64, t0, h, b, pol);
            tma_load_4d_hint(sm + L::KT + (s * (D / 64) + a) * ATOM, &mk, &bars[B_QK0 + s], a * 64, t0, h, b, pol);
        }
        ++pend[B_QK0 + s].issued;
    };
    auto load_v = [&](int idx) {
        const int t0 = chunk_of(idx) * CH;
        mbar_expect_tx(&bars[B_V], DV * CH * 2);
        for (int a = 0; a < DV / 64; ++a)
            tma_load_4d_hint(sm + L::VT + a * ATOM, &mv, &bars[B_V], a * 64, t0, h, b, pol);
        ++pend[B_V].issued;
    };
    auto load_o = [&](int idx) {
        const int t0 = chunk_of(idx) * CH;
        mbar_expect_tx(&bars[B_O], DV * CH * 2);
        for (int a = 0; a < DV / 64; ++a)
            tma_load_4d_hint(sm + L::OT + a * ATOM, &mdo, &bars[B_O], a * 64, t0, h, b, pol);
        ++pend[B_O].issued;
    };
    auto valid_of = [&](int idx) { return (int)min64(CH, p.T - (int64_t)chunk_of(idx) * CH); };
    auto qtile = [&](int idx) { return sm + L::QT + (idx & 1) * (D / 64) * ATOM; };
    auto ktile = [&](int idx) { return sm + L::KT + (idx & 1) * (D / 64) * ATOM; };
    // D_t and e_t of a chunk (rows past the end: D = 1, e = 0), by aux warps 6-7
    auto load_de = [&](int idx, float& dd, float& ee) {
        const int t = act - 64;
        const int64_t t0 = (int64_t)chunk_of(idx) * CH;
        const bool in = t0 + t < p.T;
        const int64_t gi = (int64_t)bh * p.T + t0 + t;
        dd = in ? p.Dn[gi] : 1.f;
        ee = in ? p.E[gi] : 0.f;
    };
    auto aux_phi_q = [&](int idx) {
        if (!mbar_wait(&bars[B_QK0 + (idx & 1)], (idx >> 1) & 1, abort_flag)) {
            record_timeout(p.status, abort_flag);
            return;
        }
        phi_tile<D, 128>(qtile(idx), ATOM, valid_of(idx), act, nullptr);
        fence_proxy_async_smem();
    };
    auto aux_phi_k = [&](int idx) {
        phi_tile<D, 128>(ktile(idx), ATOM, valid_of(idx), act, nullptr);
        fence_proxy_async_smem();
    };

    if (tid == 0 && n > 0) {
        load_qk(0);
        load_v(0);
        load_o(0);
    }
    // (R, r) after the range (the gradient of the final state plus the sums of the ranges
    // after it; one record when scanned): R into TMEM and its bf16 tile
    const float* rrecs = p.rev + (p.scanned ? rec_i : rec_i + 1) * p.rec;
    const int nafter = p.scanned ? 1 : p.nr - 1 - r;
    const float* Rb = p.dM_out ? p.dM_out + (int64_t)bh * D * DV : nullptr;
    sum_to_state<D, DV>(Rb, rrecs, p.rec, nafter, tmem + L::TRR, sm + L::GR + ATOM, L::GRB, warp, lane);
    if (tid < D) rv[tid] = sum_vec(p.dz_out ? p.dz_out + (int64_t)bh * D : nullptr, rrecs + D * DV, p.rec, nafter, tid);
    if (!tok && act >= 64 && n > 0) {
        float dd, ee;
        load_de(0, dd, ee);
        dn[act - 64] = dd;
        evs[act - 64] = ee;
    }
    if (!tok && n > 0) {  // the first chunk's operands, alongside the sums above
        aux_phi_q(0);
        aux_phi_k(0);
    }
    fence_proxy_async_smem();
    sync_tc();

    auto off = [](uint32_t bytes) { return (uint64_t)(bytes >> 4); };
    const uint64_t dVk = sdesc_sw128(smem_u32(sm + L::VT), 16, 1024);       // V, K-major (K = dv)
    const uint64_t dGRk = sdesc_sw128(smem_u32(sm + L::GR), 16, 1024);      // [G high; R], K-major (K = dv)
    const uint64_t dGHm = sdesc_sw128(smem_u32(sm + L::GR), L::GRB, 1024);  // G high, MN-major (K = queries)
    const uint64_t dGLk = sdesc_sw128(smem_u32(sm + L::GL), 16, 1024);      // G low, K-major
    const uint64_t dGLm = sdesc_sw128(smem_u32(sm + L::GL), ATOM, 1024);    // G low, MN-major
    const uint64_t dRm = sdesc_sw128(smem_u32(sm + L::GR + ATOM), L::GRB, 1024);  // R, MN-major (K = d, N = dv)
    const uint64_t dPk = sdesc_sw128(smem_u32(sm + L::PT), 16, 1024);
    const uint64_t dAk = sdesc_sw128(smem_u32(sm + L::AT), 16, 1024);
    uint32_t mph = 0;
    bool ok = true;

    for (int idx = 0; idx < n && ok; ++idx) {
        const int s = idx & 1;
        const int64_t t0 = (int64_t)chunk_of(idx) * CH;
        const int valid = valid_of(idx);
        const bool more = idx + 1 < n;
        uint8_t* qt = qtile(idx);
        uint8_t* kt = ktile(idx);
        const float* dc = dn + s * 64;
        const float* ec = evs + s * 64;
        const float* rc = rv + s * D;
        float* rn = rv + (s ^ 1) * D;
        float nd = 1.f, ne = 0.f;  // the next chunk's D_t and e_t (aux warps 6-7), stored at the end
        if (!tok && act >= 64 && more) load_de(idx + 1, nd, ne);
        // (this barrier also ends the previous chunk: its stage is read and R's tile written)
        ok = block_wait2(&bars[B_QK0 + s], (idx >> 1) & 1, &bars[B_O], idx & 1, abort_flag, p.status);
        if (!ok) break;
        ++pend[B_QK0 + s].waited, ++pend[B_O].waited;
        if (tid == 0 && more) load_qk(idx + 1);
        // ---- G = dout / D: high parts into [G; R], low parts; every warp (no TMEM access):
        // thread tid takes query row tid % 64 and a quarter of the DV columns
        if (!tok && act < D) rn[act] = rc[act];  // r before this chunk, completed during g2
        {
            const int t = tid & 63, cq = tid >> 6;
            const float rd = t < valid ? 1.f / dc[t] : 0.f;
#pragma unroll 1
            for (int j0 = cq * (DV / 4); j0 < (cq + 1) * (DV / 4); j0 += 16) {
                float o[16];
                tile_get8(sm + L::OT, t, j0, ATOM, o);
                tile_get8(sm + L::OT, t, j0 + 8, ATOM, o + 8);
                uint32_t gh[8], gl[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) split2(o[2 * e] * rd, o[2 * e + 1] * rd, gh[e], gl[e]);
                tile_put16(sm + L::GR, t, j0, L::GRB, gh);
                tile_put16(sm + L::GL, t, j0, ATOM, gl);
            }
            fence_proxy_async_smem();
        }
        tc_fence_before();  // (the barrier of the V wait orders the G tiles before g1)
        ok = block_wait(&bars[B_V], idx & 1, abort_flag, p.status);
        if (!ok) break;
        ++pend[B_V].waited;
        tc_fence_after();
        const uint64_t dQk = sdesc_sw128(smem_u32(qt), 16, 1024);
        const uint64_t dQm = sdesc_sw128(smem_u32(qt), ATOM, 1024);
        const uint64_t dKk = sdesc_sw128(smem_u32(kt), 16, 1024);
        // ---- g1: S^T = phi(K) phi(Q)^T; [dA^T | V R^T] = V [G; R]^T; R += phi(Q)^T G
        if (tid == 0) {
            if (more) load_o(idx + 1);
            constexpr uint32_t id_t = idesc_bf16(128, CH, 0, 0);
            constexpr uint32_t id_ar = idesc_bf16(128, CH + D, 0, 0);
            constexpr uint32_t id_r = idesc_bf16(128, DV, 1, 1);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint32_t o = (ks >> 2) * ATOM + (ks & 3) * 32;
                mma_bf16_ss(tmem + L::TS, dKk + off(o), dQk + off(o), id_t, ks != 0);
            }
#pragma unroll
            for (int ks = 0; ks < DV / 16; ++ks) {
                const uint32_t o = (ks >> 2) * ATOM + (ks & 3) * 32;
                mma_bf16_ss(tmem + L::TA, dVk + off(o), dGRk + off((ks >> 2) * L::GRB + (ks & 3) * 32), id_ar, ks != 0);
                mma_bf16_ss(tmem + L::TA, dVk + off(o), dGLk + off(o), id_t, 1);
            }
#pragma unroll
            for (int ks = 0; ks < CH / 16; ++ks) {
                mma_bf16_ss(tmem + L::TRR, dQm + off(ks * 2048), dGHm + off(ks * 2048), id_r, 1);
                mma_bf16_ss(tmem + L::TRR, dQm + off(ks * 2048), dGLm + off(ks * 2048), id_r, 1);
            }
            mma_commit(&bars[B_MMA]);
            ++pend[B_MMA].issued;
        }
        ok = block_wait(&bars[B_MMA], mph & 1, abort_flag, p.status);
        if (!ok) break;
        ++mph, ++pend[B_MMA].waited;
        tc_fence_after();
        if (tid == 0 && more) load_v(idx + 1);  // V's only reader (g1) is done
        // ---- mask: P^T and dA^T + e (bf16: each enters one product of the high parts), masked to
        // queries at or after the key; key rows, query-column halves
        if (tok) {
            const int j = trow, hf = thalf;
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            float sv[32], a[32];
            ld32f(tmem + L::TS + lb + 32 * hf, sv);
            ld32f(tmem + L::TA + lb + 32 * hf, a);
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                uint32_t ph[8], ah[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int c = 16 * g + 2 * q, tq = 32 * hf + c;
                    const bool m0 = tq >= j, m1 = tq + 1 >= j;
                    ph[q] = pack_bf16(m0 ? sv[c] : 0.f, m1 ? sv[c + 1] : 0.f);
                    ah[q] = pack_bf16(m0 ? a[c] + ec[tq] : 0.f, m1 ? a[c + 1] + ec[tq + 1] : 0.f);
                }
                const int col = 32 * hf + 16 * g;
                tile_put16(sm + L::PT, j, col, ATOM, ph);
                tile_put16(sm + L::AT, j, col, ATOM, ah);
            }
            fence_proxy_async_smem();
        } else if (more) {
            aux_phi_q(idx + 1);
        }
        sync_tc();
        // ---- g2: dv = P^T G + phi(K) R, dphi(K) += dA^T phi(Q)
        if (tid == 0) {
            constexpr uint32_t id_vg = idesc_bf16(128, DV, 0, 1);
            constexpr uint32_t id_kq = idesc_bf16(128, D, 0, 1);
#pragma unroll
            for (int ks = 0; ks < CH / 16; ++ks) {
                // dv's P^T G and dk's dA^T phi(Q) on the high parts alone; the state gradient R,
                // which sums over the whole range, keeps G's low part
                mma_bf16_ss(tmem + L::TS, dPk + off(ks * 32), dGHm + off(ks * 2048), id_vg, ks != 0);
                mma_bf16_ss(tmem + L::TK, dAk + off(ks * 32), dQm + off(ks * 2048), id_kq, 1);
            }
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_bf16_ss(tmem + L::TS, dKk + off((ks >> 2) * ATOM + (ks & 3) * 32), dRm + off(ks * 2048), id_vg, 1);
            mma_commit(&bars[B_MMA]);
            ++pend[B_MMA].issued;
        }
        // meanwhile (aux): phi(K) of the next chunk; r before this chunk's tokens are added =
        // r after them + sum e_t phi(q_t)
        if (!tok) {
            if (more) aux_phi_k(idx + 1);
            aux_weighted_colsum<D>(qt, ec, rn, act);
        }
        ok = block_wait(&bars[B_MMA], mph & 1, abort_flag, p.status);
        if (!ok) break;
        ++mph, ++pend[B_MMA].waited;
        tc_fence_after();
        // ---- end: dk = (dphi(K) + r) phi'(k) (warps 0-1), dv (warps 4-5); then R after this
        // chunk's tokens to its bf16 tile. The TMEM loads are warp-wide; only key rows inside
        // the sequence are stored.
        if (tok) {
            const int j = trow;
            const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
            const bool store = j < valid;
            if (thalf == 0) {
                __nv_bfloat16* dk = reinterpret_cast<__nv_bfloat16*>(p.dk) + ((int64_t)bh * p.T + t0 + j) * D;
#pragma unroll 1
                for (int i0 = 0; i0 < D; i0 += 32) {
                    float x[32];
                    ld32f(tmem + L::TK + lb + i0, x);
#pragma unroll
                    for (int g = 0; g < 32; g += 8) {
                        float f[8];
                        tile_get8(kt, j, i0 + g, ATOM, f);
                        uint32_t w[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            w[q] = pack_bf16((x[g + 2 * q] + rc[i0 + g + 2 * q]) * fminf(f[2 * q], 1.f),
                                             (x[g + 2 * q + 1] + rc[i0 + g + 2 * q + 1]) * fminf(f[2 * q + 1], 1.f));
                        if (store) *reinterpret_cast<uint4*>(dk + i0 + g) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            } else {
                __nv_bfloat16* dvp = reinterpret_cast<__nv_bfloat16*>(p.dv) + ((int64_t)bh * p.T + t0 + j) * DV;
#pragma unroll 1
                for (int j0 = 0; j0 < DV; j0 += 32) {
                    float x[32];
                    ld32f(tmem + L::TS + lb + j0, x);
#pragma unroll
                    for (int g = 0; g < 32; g += 8) {
                        uint32_t w[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) w[q] = pack_bf16(x[g + 2 * q], x[g + 2 * q + 1]);
                        if (store) *reinterpret_cast<uint4*>(dvp + j0 + g) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        } else if (act >= 64) {
            dn[(s ^ 1) * 64 + act - 64] = nd;
            evs[(s ^ 1) * 64 + act - 64] = ne;
        }
        state_to_tile_split<D, DV>(tmem + L::TRR, sm + L::GR + ATOM, L::GRB, warp, lane);
        fence_proxy_async_smem();
        tc_fence_before();  // (the next chunk's first wait is the barrier)
    }
    if (ok && r == 0 && n > 0 && !p.scanned) {
        // range 0 has added every chunk's share: (R, r) is now the gradient of the initial state
        if (p.dM_in) state_to_array<D, DV>(tmem + L::TRR, p.dM_in + (int64_t)bh * D * DV, warp, lane);
        if (p.dz_in && tid < D) p.dz_in[(int64_t)bh * D + tid] = rv[(n & 1) * D + tid];
    } else if (!ok && tid == 0) {
        drain(bars, pend, NB);
    }
    sync_tc();
    if (warp == 0) tmem_dealloc(tmem, L::NCOL);
}

// ================================================================================ launchers
// Blocks of a kernel that fit on one SM by shared memory, registers and TMEM columns
// (computed from the device limits: the runtime's occupancy query does not know TMEM).
template <typename L>
static int ctas_per_sm(const void* fn) {
    cudaFuncAttributes fa;
    int dev = 0, smem_sm = 0, regs_sm = 0, reserved = 0;
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
        return 1;
    const int by_smem = smem_sm / (L::ALLOC + (int)fa.sharedSizeBytes + reserved);
    const int regs_warp = (fa.numRegs * 32 + 255) / 256 * 256;  // allocated per warp in units of 256
    const int by_regs = regs_sm / (regs_warp * (BT / 32));
    const int by_tmem = 512 / (int)L::NCOL;
    int occ = by_smem < by_regs ? by_smem : by_regs;
    occ = occ < by_tmem ? occ : by_tmem;
    return occ > 0 ? occ : 1;
}

template <int D, int DV>
static int sweep_occupancy_t() {
    auto f1 = bwd_dq_sweep_kernel<D, DV>;
    auto f2 = bwd_dkdv_sweep_kernel<D, DV>;
    if (set_smem_attrs(reinterpret_cast<const void*>(f1), DqLayout<D, DV>::ALLOC) != cudaSuccess ||
        set_smem_attrs(reinterpret_cast<const void*>(f2), DkvLayout<D, DV>::ALLOC) != cudaSuccess)
        return 1;
    const int a = ctas_per_sm<DqLayout<D, DV>>(reinterpret_cast<const void*>(f1));
    const int b = ctas_per_sm<DkvLayout<D, DV>>(reinterpret_cast<const void*>(f2));
    return a < b ? a : b;
}

int bwd_sweep_occupancy(int d, int dv) {
    static int cache[2][2] = {};  // by (d == 128, dv == 128); 0 = not yet asked
    if ((d != 64 && d != 128) || (dv != 64 && dv != 128)) return 1;
    int& c = cache[d == 128][dv == 128];
    if (c == 0) {
        if (d == 128 && dv == 128) c = sweep_occupancy_t<128, 128>();
        if (d == 128 && dv == 64) c = sweep_occupancy_t<128, 64>();
        if (d == 64 && dv == 128) c = sweep_occupancy_t<64, 128>();
        if (d == 64 && dv == 64) c = sweep_occupancy_t<64, 64>();
    }
    return c;
}

template <int D, int DV>
static cudaError_t launch_dq_t(const BwdTcParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                               const CUtensorMap& mv, const CUtensorMap& mdo, cudaStream_t s) {
    using L = DqLayout<D, DV>;
    static_assert(L::ALLOC <= 227 * 1024, "shared memory budget");
    auto fn = bwd_dq_sweep_kernel<D, DV>;
    cudaError_t e = set_smem_attrs(reinterpret_cast<const void*>(fn), L::ALLOC);
    if (e != cudaSuccess) return e;
    fn<<<dim3(p.nr, p.B * p.H), BT, L::ALLOC, s>>>(mq, mk, mv, mdo, p);
    return cudaGetLastError();
}

template <int D, int DV>
static cudaError_t launch_dkdv_t(const BwdTcParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                 const CUtensorMap& mv, const CUtensorMap& mdo, cudaStream_t s) {
    using L = DkvLayout<D, DV>;
    static_assert(L::ALLOC <= 227 * 1024, "shared memory budget");
    auto fn = bwd_dkdv_sweep_kernel<D, DV>;
    cudaError_t e = set_smem_attrs(reinterpret_cast<const void*>(fn), L::ALLOC);
    if (e != cudaSuccess) return e;
    fn<<<dim3(p.nr, p.B * p.H), BT, L::ALLOC, s>>>(mq, mk, mv, mdo, p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq_tc(const BwdTcParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                             const CUtensorMap& mv, const CUtensorMap& mdo, cudaStream_t s) {
    if (p.d == 128 && p.dv_dim == 128) return launch_dq_t<128, 128>(p, mq, mk, mv, mdo, s);
    if (p.d == 128 && p.dv_dim == 64) return launch_dq_t<128, 64>(p, mq, mk, mv, mdo, s);
    if (p.d == 64 && p.dv_dim == 128) return launch_dq_t<64, 128>(p, mq, mk, mv, mdo, s);
    if (p.d == 64 && p.dv_dim == 64) return launch_dq_t<64, 64>(p, mq, mk, mv, mdo, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dkdv_tc(const BwdTcParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                               const CUtensorMap& mv, const CUtensorMap& mdo, cudaStream_t s) {
    if (p.d == 128 && p.dv_dim == 128) return launch_dkdv_t<128, 128>(p, mq, mk, mv, mdo, s);
    if (p.d == 128 && p.dv_dim == 64) return launch_dkdv_t<128, 64>(p, mq, mk, mv, mdo, s);
    if (p.d == 64 && p.dv_dim == 128) return launch_dkdv_t<64, 128>(p, mq, mk, mv, mdo, s);
    if (p.d == 64 && p.dv_dim == 64) return launch_dkdv_t<64, 64>(p, mq, mk, mv, mdo, s);
    return cudaErrorInvalidValue;
}

}  // namespace la
