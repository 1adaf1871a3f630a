// Tensor-core (tcgen05 + TMEM + TMA) per-part state sums for bf16 storage:
//
//   parts_tc  A_p = sum_{t in p} phi(k_t) v_t^T (f32, d x dv) and s_p = sum phi(k_t)
//             over a part of the sequence: the key-value sum of the prompt mode on
//             the page "Attention_Kernel_Mask" (table "Causal Attention Training and
//             Inferencing" and the note below it: only the final state is needed,
//             and its sum can be formed in parallel pieces). Used for prefill parts
//             and for the range aggregates of the sequence-split forward.
//
// Roles in a block of 320 threads (two blocks per SM): warp 0 lane 0 issues TMA loads
// into a 3-stage ring, warp 1 owns TMEM and lane 0 issues tcgen05.mma (M^T (dv x d) += V_c^T phi(K_c),
// f32 accumulator in TMEM), warps 2-9 (two per sub-partition) apply phi in place and
// keep column sums of phi(K) for s_p, then write the record. TMEM lane quarter
// q = warp % 4 is accessible to that warp only.
//
// Operand layouts (128-byte swizzled, 1024-byte aligned atoms of 8 rows x 128 bytes,
// 16-byte chunk c of row r stored at chunk c ^ (r % 8)): K and V tiles exactly as TMA
// loads them, [64 tokens][64 features] per atom, both read MN-major (K dimension =
// tokens).
#include "la_tc_common.cuh"

namespace la {

// ============================================================================ parts_tc
constexpr int PARTS_FW = 8;  // phi warps
constexpr int PARTS_THREADS = 64 + 32 * PARTS_FW;

template <int D, int DV>
struct PartsLayout {
    static constexpr int NS = 3;   // 3 stages keep two blocks on an SM (~109 KB each)
    static constexpr int KB = D / 64 * ATOM;
    static constexpr int VB = DV / 64 * ATOM;
    static constexpr int STAGE = KB + VB;
    static constexpr int PAD = ATOM;  // an M=128 operand over a 64-wide V tile reads one atom past it
    static constexpr int BAR = NS * STAGE + PAD;
    static constexpr int NBAR = 3 * NS + 1;
    static constexpr int MISC = BAR + 8 * NBAR;          // tmem holder, abort flag
    static constexpr int ZP = MISC + 16;
    static constexpr int TOTAL = ZP + PARTS_FW * D * 4;
    static constexpr int ALLOC = TOTAL + 1024;           // slack for 1024-byte alignment
};

template <int D, int DV>
__global__ void __launch_bounds__(PARTS_THREADS, 2)
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
            const uint64_t pol = l2_evict_first_policy();  // k, v are read once
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
                for (int a = 0; a < D / 64; ++a) tma_load_4d_hint(kb + a * ATOM, &mk, &full[s], a * 64, t, h, b, pol);
#pragma unroll
                for (int a = 0; a < DV / 64; ++a) tma_load_4d_hint(vb + a * ATOM, &mv, &full[s], a * 64, t, h, b, pol);
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
    } else {  // ------------------------ phi warps
        constexpr int NT = 32 * PARTS_FW;
        const int ct = threadIdx.x - 64;
        float colsum[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) colsum[e] = 0.f;
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int s = c % NS;
            ok = bar_and(1, NT, mbar_wait(&full[s], (c / NS) & 1, abort_flag));
            if (!ok) break;
            const int valid = (int)min64(CH, t_end - (t_begin + (int64_t)c * CH));
            phi_tile<D, NT>(sm + s * L::STAGE, ATOM, valid, ct, colsum, p.phi_ident);
            fence_proxy_async_smem();
            named_bar_sync(1, NT);
            if (ct == 0) mbar_arrive(&phib[s]);
        }
        if (!ok && ct == 0) record_timeout(p.status, abort_flag);
        ok = bar_and(1, NT, ok && mbar_wait(done, 0, abort_flag));
        colsum_to_smem<D>(colsum, zpart, ct);
        named_bar_sync(1, NT);
        if (ok) {
            tc_fence_after();
            const int64_t rec = (int64_t)bh * p.nparts + part;
            if (ct < D) {
                float zz = 0.f;
#pragma unroll
                for (int w = 0; w < PARTS_FW; ++w) zz += zpart[w * D + ct];
                if (p.base_z) zz += p.base_z[(int64_t)bh * D + ct];
                p.dst_z[rec * p.rec_z + ct] = zz;
            }
            // warps 2-5 write columns [0, 64) of the record's rows, warps 6-9 columns [64, 128)
            const int q = warp & 3;
            const int c_lo = (warp - 2) / 4 * 64;
            if (32 * q < DV && c_lo < D) {  // warp-uniform
                const int j = 32 * q + lane;
                float* dst = p.dst_M + rec * p.rec_M + j;
                const float* base = p.base_M ? p.base_M + (int64_t)bh * D * DV + j : nullptr;
#pragma unroll 1
                for (int i0 = c_lo; i0 < c_lo + 64; i0 += 32) {
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

// ============================================================================ launchers
template <int D, int DV>
static cudaError_t launch_parts_tc_t(const PartsParams& p, const CUtensorMap& mk, const CUtensorMap& mv,
                                     cudaStream_t s) {
    using L = PartsLayout<D, DV>;
    auto fn = parts_tc_kernel<D, DV>;
    cudaError_t e = set_smem_attrs(reinterpret_cast<const void*>(fn), L::ALLOC);
    if (e != cudaSuccess) return e;
    dim3 grid(p.nparts, p.B * p.H);
    fn<<<grid, PARTS_THREADS, L::ALLOC, s>>>(mk, mv, p);
    return cudaGetLastError();
}

cudaError_t launch_parts_tc(const PartsParams& p, const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t s) {
    if (p.d == 128 && p.dv == 128) return launch_parts_tc_t<128, 128>(p, mk, mv, s);
    if (p.d == 128 && p.dv == 64) return launch_parts_tc_t<128, 64>(p, mk, mv, s);
    if (p.d == 64 && p.dv == 128) return launch_parts_tc_t<64, 128>(p, mk, mv, s);
    if (p.d == 64 && p.dv == 64) return launch_parts_tc_t<64, 64>(p, mk, mv, s);
    return cudaErrorInvalidValue;
}

}  // namespace la
