// Tensor-core (tcgen05 + TMEM + TMA) kernels for bf16 storage, f32 accumulation.
//
//   parts_tc  per-part key-value state sums  A_p = sum_{t in p} phi(k_t) v_t^T,
//             s_p = sum phi(k_t): the "sum of k v over the prompt, formed in
//             parallel" of the prompt mode on the page "Attention_Kernel_Mask"
//             (table "Causal Attention Training and Inferencing" and the note below
//             it). Used for prefill parts and for the range aggregates of the
//             sequence-split forward.
//   fwd_tc    the chunk-sequential forward (that page's "chunk sequential mode",
//             mode 3): per chunk c of 64 tokens
//                S'  = phi(Q_c) [phi(K_c) ; z_{c-1}]^T            (64 x 80, TMEM)
//                P   = S'[:, :64] masked to the lower triangle (bf16, smem)
//                den = S'[:, 64] + rowsum(P) + eps
//                O^T = V_c^T P^T + M_{c-1}^T phi(Q_c)^T          (dv x 64, TMEM)
//                out = O / den
//                M^T += V_c^T phi(K_c),  z += sum phi(K_c)       (state in TMEM / smem)
//             with M^T kept as the f32 accumulator in TMEM and re-cast to bf16 in
//             shared memory once per chunk for the next chunk's inter-chunk MMA.
//
// Roles in a block of 192 threads: warp 0 lane 0 issues TMA loads, warp 1 owns
// TMEM and lane 0 issues tcgen05.mma, warps 2-5 (128 threads) apply phi and run
// the epilogues. TMEM lane quarter q = warp % 4 is accessible to that warp only.
//
// Shared-memory operand layouts (all 128-byte swizzled, 1024-byte aligned atoms of
// 8 rows x 128 bytes, 16-byte chunk c of row r stored at chunk c ^ (r % 8)):
//   Q, K, V tiles as loaded by TMA: [64 tokens][64 features] per atom.
//     phi(Q) / phi(K) read K-major (rows = tokens, K = features) for S' and O^T;
//     phi(K) and V read MN-major (rows = tokens = K) for the state update and P V.
//   P: [64 queries][64 keys] K-major.  M^T (bf16): [128 dv rows][d] K-major.
#include "la_internal.h"

namespace la {

constexpr int CH = 64;                 // tokens per chunk on the tensor-core path
constexpr int ATOM = 64 * 128;         // one 64-row, 128-byte-wide swizzle block column
constexpr int KROWS = 80;              // forward K tile rows: 64 keys, z row, 15 zero rows
constexpr int ATOMK = KROWS * 128;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// AND-reduce a predicate over the `n` threads of named barrier `id`.
__device__ __forceinline__ bool bar_and(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort_flag) {
    *abort_flag = 1;
    if (status) atomicOr(status, STATUS_TIMEOUT);
}

// Bounded wait that ignores the abort flag (used while draining at exit).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
    const unsigned long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > LA_WAIT_CYCLES) return false;
    }
    return true;
}

// phi in place on a [64 x D] bf16 tile (atoms `astride` bytes apart), by the 128
// compute threads. Thread ct owns 16-byte chunk column j = ct % (D/8) of rows
// g, g + RG, ... (g = ct / (D/8)); since RG is a multiple of 8 the swizzled chunk
// position j ^ (row % 8) is the same for all of its rows. Rows >= valid become 0
// when ZERO_TAIL (phi(0) = 1 must not enter the sums). With COLSUM the thread adds
// the bf16-rounded results of its 8 columns into colsum[0..8).
template <int D, bool ZERO_TAIL, bool COLSUM>
__device__ __forceinline__ void phi_tile(uint8_t* tile, int astride, int valid, int ct, float* colsum) {
    constexpr int CPR = D / 8;
    constexpr int RG = 128 / CPR;
    constexpr int RPT = CH / RG;
    const int j = ct % CPR, g = ct / CPR;
    uint8_t* base = tile + (j >> 3) * astride + (((j & 7) ^ (g & 7)) << 4);
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int r = g + i * RG;
        uint4* ptr = reinterpret_cast<uint4*>(base + r * 128);
        uint4 x = *ptr;
        uint32_t w[4] = {x.x, x.y, x.z, x.w};
        const bool live = !ZERO_TAIL || r < valid;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t pk = live ? pack_bf16(phi_f(bf16lo(w[e])), phi_f(bf16hi(w[e]))) : 0u;
            if (COLSUM) {
                colsum[2 * e] += bf16lo(pk);
                colsum[2 * e + 1] += bf16hi(pk);
            }
            w[e] = pk;
        }
        *ptr = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Combine the per-thread column sums of phi_tile into zpart[warp][D] (lanes that hold
// a full warp's sum for chunk column j = lane write columns 8j..8j+7).
template <int D>
__device__ __forceinline__ void colsum_to_smem(float* colsum, float* zpart, int ct) {
    constexpr int CPR = D / 8;
#pragma unroll
    for (int off = CPR; off < 32; off <<= 1)
#pragma unroll
        for (int e = 0; e < 8; ++e) colsum[e] += __shfl_xor_sync(0xffffffffu, colsum[e], off);
    const int lane = ct & 31, w = ct >> 5;
    if (lane < CPR)
#pragma unroll
        for (int e = 0; e < 8; ++e) zpart[w * D + lane * 8 + e] = colsum[e];
}

// ============================================================================ parts_tc
template <int D, int DV>
struct PartsLayout {
    static constexpr int NS = 4;
    static constexpr int KB = D / 64 * ATOM;
    static constexpr int VB = DV / 64 * ATOM;
    static constexpr int STAGE = KB + VB;
    static constexpr int PAD = ATOM;  // an M=128 operand over a 64-wide V tile reads one atom past it
    static constexpr int BAR = NS * STAGE + PAD;
    static constexpr int NBAR = 3 * NS + 1;
    static constexpr int MISC = BAR + 8 * NBAR;          // tmem holder, abort flag
    static constexpr int ZP = MISC + 16;
    static constexpr int TOTAL = ZP + 4 * D * 4;
    static constexpr int ALLOC = TOTAL + 1024;           // slack for 1024-byte alignment
};

template <int D, int DV>
__global__ void __launch_bounds__(192, 1)
    parts_tc_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv, PartsParams p) {
    using L = PartsLayout<D, DV>;
    constexpr int NS = L::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint64_t* empty = full + NS;
    uint64_t* phib = empty + NS;
    uint64_t* done = phib + NS;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
    float* zpart = reinterpret_cast<float*>(sm + L::ZP);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int part = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H;
    const int64_t t_begin = (int64_t)part * p.part_len;
    const int64_t t_end = min64(p.T, t_begin + p.part_len);
    const int nch = (int)((t_end - t_begin + CH - 1) / CH);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&phib[s], 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 128);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int s = c % NS;
                if (c >= NS && !mbar_wait(&empty[s], ((c / NS) - 1) & 1, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    break;
                }
                uint8_t* kb = sm + s * L::STAGE;
                uint8_t* vb = kb + L::KB;
                mbar_expect_tx(&full[s], L::STAGE);
                const int t = (int)(t_begin + (int64_t)c * CH);
#pragma unroll
                for (int a = 0; a < D / 64; ++a) tma_load_4d(kb + a * ATOM, &mk, &full[s], a * 64, t, h, b);
#pragma unroll
                for (int a = 0; a < DV / 64; ++a) tma_load_4d(vb + a * ATOM, &mv, &full[s], a * 64, t, h, b);
                ++issued;
            }
            // no copy may still be in flight when the block exits
            for (int c = max(0, issued - NS); c < issued; ++c) mbar_wait_drain(&full[c % NS], (c / NS) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer: M^T (dv x d) += V_c^T phi(K_c)
            constexpr uint32_t idesc = idesc_bf16(128, D, 1, 1);
            for (int c = 0; c < nch; ++c) {
                const int s = c % NS;
                if (!mbar_wait(&phib[s], (c / NS) & 1, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t kb = smem_u32(sm + s * L::STAGE);
                const uint32_t vb = kb + L::KB;
#pragma unroll
                for (int ks = 0; ks < CH / 16; ++ks)
                    mma_bf16_ss(tmem, sdesc_sw128(vb + ks * 2048, ATOM, 1024), sdesc_sw128(kb + ks * 2048, ATOM, 1024),
                                idesc, (c | ks) != 0);
                mma_commit(&empty[s]);
            }
            mma_commit(done);
            mbar_wait_drain(done, 0);
        }
    } else {  // ------------------------ compute warps
        const int ct = threadIdx.x - 64;
        float colsum[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) colsum[e] = 0.f;
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int s = c % NS;
            ok = bar_and(1, 128, mbar_wait(&full[s], (c / NS) & 1, abort_flag));
            if (!ok) break;
            const int valid = (int)min64(CH, t_end - (t_begin + (int64_t)c * CH));
            phi_tile<D, true, true>(sm + s * L::STAGE, ATOM, valid, ct, colsum);
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (ct == 0) mbar_arrive(&phib[s]);
        }
        if (!ok && ct == 0) record_timeout(p.status, abort_flag);
        ok = bar_and(1, 128, ok && mbar_wait(done, 0, abort_flag));
        colsum_to_smem<D>(colsum, zpart, ct);
        named_bar_sync(1, 128);
        if (ok) {
            tc_fence_after();
            const int64_t rec = (int64_t)bh * p.nparts + part;
            if (ct < D) {
                float zz = zpart[ct] + zpart[D + ct] + zpart[2 * D + ct] + zpart[3 * D + ct];
                if (p.base_z) zz += p.base_z[(int64_t)bh * D + ct];
                p.dst_z[rec * p.rec_z + ct] = zz;
            }
            const int q = warp & 3;
            if (32 * q < DV) {  // warp-uniform
                const int j = 32 * q + lane;
                float* dst = p.dst_M + rec * p.rec_M + j;
                const float* base = p.base_M ? p.base_M + (int64_t)bh * D * DV + j : nullptr;
#pragma unroll 1
                for (int i0 = 0; i0 < D; i0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + i0, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        float m = __uint_as_float(r[e]);
                        if (base) m += base[(i0 + e) * DV];
                        dst[(i0 + e) * DV] = m;
                    }
                }
            }
        } else if (ct == 0) {
            record_timeout(p.status, abort_flag);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

// ============================================================================ fwd_tc
template <int D, int DV>
struct FwdLayout {
    static constexpr int QB = D / 64 * ATOM;
    static constexpr int KB = D / 64 * ATOMK;
    static constexpr int VB = DV / 64 * ATOM;
    static constexpr int Q0 = 0;
    static constexpr int K0 = Q0 + 2 * QB;
    static constexpr int V0 = K0 + 2 * KB;
    static constexpr int MT = V0 + 2 * VB;                 // bf16 M^T, 128 rows x d
    static constexpr int MTB = D / 64 * (128 * 128);
    static constexpr int PT = MT + MTB;                    // P, 64 x 64 bf16
    static constexpr int OT = PT + ATOM;                   // out tile, 64 x dv bf16
    static constexpr int PAD = OT + DV / 64 * ATOM;        // garbage-row reads land here at most
    static constexpr int SMALL = PAD + ATOM;
    static constexpr int RDEN = SMALL;                     // 64 floats
    static constexpr int ZF = RDEN + 64 * 4;               // d floats: z_{c-1}, then z_c
    static constexpr int ZP = ZF + 128 * 4;                // 4 x d floats
    static constexpr int BAR = ZP + 4 * 128 * 4;           // 9 mbarriers
    static constexpr int MISC = BAR + 8 * 9 + 8;
    static constexpr int TOTAL = MISC + 16;
    static constexpr int ALLOC = TOTAL + 1024;
};

template <int D, int DV>
__global__ void __launch_bounds__(192, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                  const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mo, FwdTcParams p) {
    using L = FwdLayout<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    float* rden = reinterpret_cast<float*>(sm + L::RDEN);
    float* zf = reinterpret_cast<float*>(sm + L::ZF);
    float* zpart = reinterpret_cast<float*>(sm + L::ZP);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint64_t* full = bars;          // [2]
    uint64_t* empty = bars + 2;     // [2]
    uint64_t* phi_rdy = bars + 4;
    uint64_t* mma1 = bars + 5;
    uint64_t* p_rdy = bars + 6;
    uint64_t* mma2 = bars + 7;
    uint64_t* drain = bars + 8;     // final MMA commit, waited by the MMA thread only
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H;
    const int64_t nch_total = (p.T + CH - 1) / CH;
    const int64_t c_begin = (int64_t)r * p.chunks_per_range;
    const int nch = (int)min64(p.chunks_per_range, nch_total - c_begin);
    const int64_t t_begin = c_begin * CH;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 9; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
        tma_prefetch_desc(&mo);
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    const uint32_t tM = tmem;          // M^T f32: lanes = dv rows, columns 0..d-1
    const uint32_t tS = tmem + 128;    // S' (80 columns), then O^T (64 columns)

    // ---------------- start state: M_in + sum of the aggregates of earlier ranges
    if (warp >= 2) {
        const int ct = threadIdx.x - 64;
        const int q = warp & 3;
        const int j = 32 * q + lane;
        const float* agg = p.ws ? p.ws + (int64_t)bh * (p.nranges - 1) * p.rec : nullptr;
        if (32 * q < DV) {
            uint8_t* mrow = sm + L::MT + j * 128;
#pragma unroll 1
            for (int i0 = 0; i0 < D; i0 += 16) {
                uint32_t rr[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int i = i0 + e;
                    float m = p.M_in ? p.M_in[((int64_t)bh * D + i) * DV + j] : 0.f;
                    for (int pp = 0; pp < r; ++pp) m += agg[pp * p.rec + i * DV + j];
                    rr[e] = __float_as_uint(m);
                }
                tmem_st16(tM + ((uint32_t)(32 * q) << 16) + i0, rr);
                uint8_t* atom = mrow + (i0 >> 6) * (128 * 128);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int cc = ((i0 & 63) >> 3) + u;
                    const uint32_t* x = rr + 8 * u;
                    *reinterpret_cast<uint4*>(atom + ((cc ^ (j & 7)) << 4)) =
                        make_uint4(pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                   pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                   pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                   pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
                }
            }
            tmem_wait_st();
        } else {
            uint8_t* mrow = sm + L::MT + j * 128;
            for (int a = 0; a < D / 64; ++a)
                for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<uint4*>(mrow + a * (128 * 128) + cc * 16) = make_uint4(0, 0, 0, 0);
        }
        if (ct < D) {
            float zz = p.z_in ? p.z_in[(int64_t)bh * D + ct] : 0.f;
            for (int pp = 0; pp < r; ++pp) zz += agg[pp * p.rec + D * DV + ct];
            zf[ct] = zz;
        }
        // K tile rows 65..79 of both stages stay zero (row 64 carries z each chunk)
        for (int idx = ct; idx < 2 * (D / 64) * 15 * 8; idx += 128) {
            const int cc = idx % 8, row = 65 + (idx / 8) % 15, sa = idx / (8 * 15);
            *reinterpret_cast<uint4*>(sm + L::K0 + sa * ATOMK + row * 128 + cc * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == 0) {
        if (lane == 0) {  // ---------------- TMA producer, 2 stages
            int issued = 0;
            for (int c = 0; c < nch; ++c) {
                const int s = c & 1;
                if (c >= 2 && !mbar_wait(&empty[s], ((c >> 1) - 1) & 1, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    break;
                }
                uint8_t* qb = sm + L::Q0 + s * L::QB;
                uint8_t* kb = sm + L::K0 + s * L::KB;
                uint8_t* vb = sm + L::V0 + s * L::VB;
                mbar_expect_tx(&full[s], (2 * D + DV) * CH * 2);
                const int t = (int)(t_begin + (int64_t)c * CH);
#pragma unroll
                for (int a = 0; a < D / 64; ++a) {
                    tma_load_4d(qb + a * ATOM, &mq, &full[s], a * 64, t, h, b);
                    tma_load_4d(kb + a * ATOMK, &mk, &full[s], a * 64, t, h, b);
                }
#pragma unroll
                for (int a = 0; a < DV / 64; ++a) tma_load_4d(vb + a * ATOM, &mv, &full[s], a * 64, t, h, b);
                ++issued;
            }
            for (int c = max(0, issued - 2); c < issued; ++c) mbar_wait_drain(&full[c & 1], (c >> 1) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {  // ---------------- MMA issuer
            constexpr uint32_t id_s = idesc_bf16(128, KROWS, 0, 0);   // S' = phiQ [phiK; z]^T
            constexpr uint32_t id_u = idesc_bf16(128, D, 1, 1);       // M^T += V^T phiK
            constexpr uint32_t id_pv = idesc_bf16(128, CH, 1, 0);     // O^T = V^T P^T
            constexpr uint32_t id_in = idesc_bf16(128, CH, 0, 0);     // O^T += M^T phiQ^T
            const uint32_t mt = smem_u32(sm + L::MT);
            const uint32_t pt = smem_u32(sm + L::PT);
            for (int c = 0; c < nch; ++c) {
                const int s = c & 1;
                const uint32_t qb = smem_u32(sm + L::Q0 + s * L::QB);
                const uint32_t kb = smem_u32(sm + L::K0 + s * L::KB);
                const uint32_t vb = smem_u32(sm + L::V0 + s * L::VB);
                if (!mbar_wait(phi_rdy, c & 1, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks & 3) * 32;
                    mma_bf16_ss(tS, sdesc_sw128(qb + (ks >> 2) * ATOM + off, 16, 1024),
                                sdesc_sw128(kb + (ks >> 2) * ATOMK + off, 16, 1024), id_s, ks != 0);
                }
#pragma unroll
                for (int ks = 0; ks < CH / 16; ++ks)
                    mma_bf16_ss(tM, sdesc_sw128(vb + ks * 2048, ATOM, 1024), sdesc_sw128(kb + ks * 2048, ATOMK, 1024),
                                id_u, 1);
                mma_commit(mma1);
                if (!mbar_wait(p_rdy, c & 1, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < CH / 16; ++ks)
                    mma_bf16_ss(tS, sdesc_sw128(vb + ks * 2048, ATOM, 1024), sdesc_sw128(pt + ks * 32, 16, 1024),
                                id_pv, ks != 0);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks & 3) * 32;
                    mma_bf16_ss(tS, sdesc_sw128(mt + (ks >> 2) * (128 * 128) + off, 16, 1024),
                                sdesc_sw128(qb + (ks >> 2) * ATOM + off, 16, 1024), id_in, 1);
                }
                mma_commit(mma2);
                mma_commit(&empty[s]);
            }
            mma_commit(drain);
            mbar_wait_drain(drain, 0);  // no MMA may still run when TMEM is released
        }
    } else {  // ------------------------ compute warps
        const int ct = threadIdx.x - 64;
        const int q = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const bool is_store = (ct == 0);
        bool ok = true;
        int c = 0;
        for (; c < nch; ++c) {
            const int s = c & 1;
            uint8_t* qb = sm + L::Q0 + s * L::QB;
            uint8_t* kb = sm + L::K0 + s * L::KB;
            const int valid = (int)min64(CH, p.T - (t_begin + (int64_t)c * CH));
            ok = bar_and(1, 128, mbar_wait(&full[s], (c >> 1) & 1, abort_flag));
            if (!ok) break;
            // z_{c-1} into K row 64 (row 64 % 8 == 0: no swizzle offset), then phi
            if (ct < D)
                *reinterpret_cast<__nv_bfloat16*>(kb + (ct >> 6) * ATOMK + 64 * 128 + (ct & 63) * 2) =
                    __float2bfloat16_rn(zf[ct]);
            float colsum[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) colsum[e] = 0.f;
            phi_tile<D, false, false>(qb, ATOM, CH, ct, nullptr);
            phi_tile<D, true, true>(kb, ATOMK, valid, ct, colsum);
            colsum_to_smem<D>(colsum, zpart, ct);
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (ct == 0) mbar_arrive(phi_rdy);
            if (ct < D) zf[ct] += zpart[ct] + zpart[D + ct] + zpart[2 * D + ct] + zpart[3 * D + ct];

            // ---- S' epilogue: P (bf16, masked) and 1 / den
            ok = bar_and(1, 128, mbar_wait(mma1, c & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            if (q < 2) {
                const int t = 32 * q + lane;
                uint32_t rs[KROWS];
                tmem_ld32(tS + lane_base + 0, rs);
                tmem_ld32(tS + lane_base + 32, rs + 32);
                tmem_ld16(tS + lane_base + 64, rs + 64);
                tmem_wait_ld();
                float rowsum = 0.f;
                uint32_t pk[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const float s0 = (2 * jj <= t) ? __uint_as_float(rs[2 * jj]) : 0.f;
                    const float s1 = (2 * jj + 1 <= t) ? __uint_as_float(rs[2 * jj + 1]) : 0.f;
                    const uint32_t pp = pack_bf16(s0, s1);
                    rowsum += bf16lo(pp) + bf16hi(pp);
                    pk[jj] = pp;
                }
                uint8_t* prow = sm + L::PT + t * 128;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc)
                    *reinterpret_cast<uint4*>(prow + ((cc ^ (t & 7)) << 4)) =
                        make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
                rden[t] = 1.f / (__uint_as_float(rs[64]) + rowsum + p.eps);
            }
            tc_fence_before();
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (ct == 0) mbar_arrive(p_rdy);

            // ---- O epilogue and M re-cast
            ok = bar_and(1, 128, mbar_wait(mma2, c & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            if (is_store) tma_store_wait_read0();  // previous out tile has been read
            named_bar_sync(1, 128);
            if (32 * q < DV) {
                const int j = 32 * q + lane;
                uint32_t ro[CH];
                tmem_ld32(tS + lane_base + 0, ro);
                tmem_ld32(tS + lane_base + 32, ro + 32);
                tmem_wait_ld();
                uint8_t* obase = sm + L::OT + (j >> 6) * ATOM + (j & 7) * 2;
                const int cc = (j & 63) >> 3;
#pragma unroll
                for (int t = 0; t < CH; ++t)
                    *reinterpret_cast<__nv_bfloat16*>(obase + t * 128 + ((cc ^ (t & 7)) << 4)) =
                        __float2bfloat16_rn(__uint_as_float(ro[t]) * rden[t]);
                uint8_t* mrow = sm + L::MT + j * 128;
#pragma unroll 1
                for (int i0 = 0; i0 < D; i0 += 32) {
                    uint32_t rm[32];
                    tmem_ld32(tM + lane_base + i0, rm);
                    tmem_wait_ld();
                    uint8_t* atom = mrow + (i0 >> 6) * (128 * 128);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int c2 = ((i0 & 63) >> 3) + u;
                        const uint32_t* x = rm + 8 * u;
                        *reinterpret_cast<uint4*>(atom + ((c2 ^ (j & 7)) << 4)) =
                            make_uint4(pack_bf16(__uint_as_float(x[0]), __uint_as_float(x[1])),
                                       pack_bf16(__uint_as_float(x[2]), __uint_as_float(x[3])),
                                       pack_bf16(__uint_as_float(x[4]), __uint_as_float(x[5])),
                                       pack_bf16(__uint_as_float(x[6]), __uint_as_float(x[7])));
                    }
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (is_store) {
                const int t = (int)(t_begin + (int64_t)c * CH);
#pragma unroll
                for (int a = 0; a < DV / 64; ++a) tma_store_4d(&mo, sm + L::OT + a * ATOM, a * 64, t, h, b);
                tma_store_commit();
            }
        }
        if (!ok && ct == 0) record_timeout(p.status, abort_flag);
        // ---- final state (last range only)
        if (ok && r == p.nranges - 1) {
            if (p.M_out && 32 * q < DV) {
                const int j = 32 * q + lane;
                float* dst = p.M_out + (int64_t)bh * D * DV + j;
#pragma unroll 1
                for (int i0 = 0; i0 < D; i0 += 32) {
                    uint32_t rm[32];
                    tmem_ld32(tM + lane_base + i0, rm);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) dst[(i0 + e) * DV] = __uint_as_float(rm[e]);
                }
            }
            if (p.z_out && ct < D) p.z_out[(int64_t)bh * D + ct] = zf[ct];
        }
        if (is_store) tma_store_wait_all0();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// ============================================================================ launchers
template <int D, int DV>
static cudaError_t launch_parts_tc_t(const PartsParams& p, const CUtensorMap& mk, const CUtensorMap& mv,
                                     cudaStream_t s) {
    using L = PartsLayout<D, DV>;
    auto fn = parts_tc_kernel<D, DV>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    dim3 grid(p.nparts, p.B * p.H);
    fn<<<grid, 192, L::ALLOC, s>>>(mk, mv, p);
    return cudaGetLastError();
}

cudaError_t launch_parts_tc(const PartsParams& p, const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t s) {
    if (p.d == 128 && p.dv == 128) return launch_parts_tc_t<128, 128>(p, mk, mv, s);
    if (p.d == 128 && p.dv == 64) return launch_parts_tc_t<128, 64>(p, mk, mv, s);
    if (p.d == 64 && p.dv == 128) return launch_parts_tc_t<64, 128>(p, mk, mv, s);
    if (p.d == 64 && p.dv == 64) return launch_parts_tc_t<64, 64>(p, mk, mv, s);
    return cudaErrorInvalidValue;
}

template <int D, int DV>
static cudaError_t launch_fwd_tc_t(const FwdTcParams& p, int B, const CUtensorMap& mq, const CUtensorMap& mk,
                                   const CUtensorMap& mv, const CUtensorMap& mo, cudaStream_t s) {
    using L = FwdLayout<D, DV>;
    auto fn = fwd_tc_kernel<D, DV>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    dim3 grid(p.nranges, B * p.H);
    fn<<<grid, 192, L::ALLOC, s>>>(mq, mk, mv, mo, p);
    return cudaGetLastError();
}

cudaError_t launch_fwd_tc(const FwdTcParams& p, int d, int dv, int B, const CUtensorMap& mq, const CUtensorMap& mk,
                          const CUtensorMap& mv, const CUtensorMap& mo, cudaStream_t s) {
    if (d == 128 && dv == 128) return launch_fwd_tc_t<128, 128>(p, B, mq, mk, mv, mo, s);
    if (d == 128 && dv == 64) return launch_fwd_tc_t<128, 64>(p, B, mq, mk, mv, mo, s);
    if (d == 64 && dv == 128) return launch_fwd_tc_t<64, 128>(p, B, mq, mk, mv, mo, s);
    if (d == 64 && dv == 64) return launch_fwd_tc_t<64, 64>(p, B, mq, mk, mv, mo, s);
    return cudaErrorInvalidValue;
}

}  // namespace la
