// Tensor-core chunk-sequential causal forward for bf16 storage, f32 accumulation:
// the "chunk sequential mode" (mode 3) of the page "Attention_Kernel_Mask"
// (allenlu2009.github.io), with the normaliser of that page's cumulative-sum
// recurrence split the same way. Per chunk c of 64 tokens:
//     S'  = phi(Q_c) [phi(K_c) ; z_{c-1}]^T              64 x 80 (TMEM)
//     P   = S'[:, :64] masked to the lower triangle incl. the diagonal (bf16, smem)
//     den = S'[:, 64] + rowsum(P) + eps                   (= phi(q_t).z_t + eps)
//     O^T = M_{c-1}^T phi(Q_c)^T + V_c^T P^T              dv x 64 (TMEM)
//     out = O / den
//     M^T += V_c^T phi(K_c) (f32 in TMEM),  z += phi(K_c)^T 1 (f32 in TMEM)
// M^T is re-cast to bf16 after every update into a second TMEM region, which is the A
// operand (read from tensor memory) of the next chunk's inter-chunk MMA; the state
// never passes through shared memory. The key sum z is accumulated on the tensor pipe
// too: phi(K_c)^T (d x 64) times a constant 64 x 16 tile of ones adds the column sums
// of phi(K_c) to a 16-column f32 accumulator (every column the same; column 0 is read).
//
// At dv = 64 the spare lanes 64-127 of the M = 128 products carry the normaliser instead:
// every V stage is followed by an atom of ones, so rows 64-127 of the V^T operand are 1.
// The update then adds the column sums of phi(K_c) to lanes 64-127 of M^T (z^T, with z_in
// placed there at the start), the bf16 re-cast copies z^T into lanes 64-95 of the inter
// operand, so the inter MMA leaves phi(q_t).z_{c-1} in lanes 64-95 of O^T and PV adds
// sum_j P_tj there: lane 64 of O^T is den_t - eps. No key-sum MMA, no z row in the K
// tile (S' is 64 x 64) and no row sums in the P pass; the E warps of lane quarter 2 form
// 1/den. (The row sum is then over the bf16 P that also enters PV.)
//
// One block per (range, head). Warp roles (1024 threads; warp w issues on sub-partition
// w % 4 and may touch only TMEM lane quarter w % 4):
//   warp 0        TMA producer: Q, K, V tiles into a 3-stage ring (5 stages at d = dv = 64)
//   warp 1        TMEM owner; lane 0 issues every tcgen05.mma, software-pipelined one
//                 chunk ahead: PV_c, then S'_{c+1}, inter_{c+1}, update_{c+1} (at d = dv = 64,
//                 where S' does not depend on the state: PV_c, inter_{c+1}, update_{c+1}, S'_{c+2})
//   warps 2,3,18-20,22-24,26-28,30  F: phi in place on Q and K, zero padded keys (none on
//                 sub-partition 1, which the MMA-issuing warp uses; warps 21, 25, 29, 31 idle)
//   warps 4-7     R: after each update, z (bf16) into row 64 of the next chunk's K tile and
//                 the bf16 re-cast of M^T; final M and z to global memory
//   warps 8-15    E: initial state (M^T and z) into TMEM; then out = O / den -> bf16 -> swizzled
//                 smem tile (O^T holds one feature per lane: fragments loaded in the
//                 accumulator layout are stored transposed with stmatrix) -> TMA store;
//                 warps 8-11 take tokens 0-31, 12-15 tokens 32-63
//   warps 16,17   S: P and 1/den from S'
// Each hand-off is an mbarrier; TMEM reads and writes are ordered with tcgen05 fences
// around it.
//
// Segment-wise output (the SEG variant, la_causal_fwd_segments): after the update of the chunk
// that ends a segment, the R warps also write the f32 state (M, z) of that segment boundary;
// the state itself stays in TMEM across the boundary, so a whole segmented sequence is one
// launch.
//
// Sequence split: in the fused two-range schedule (split > 0) range 1 first forms
// the state of chunks [0, split) itself (phi(K) and the update only) while range 0
// runs its main pass over the same chunks. Those state-only chunks go through the ring at
// d = 128; at d = dv = 64 they stream two chunks per stage (one 128-row box per tensor, two
// stages over the ring's Q and K slots): a copy engine moves a 128-row box in little more
// time than a 64-row one, and at that width the boxes, not the bytes, set a stage's pace. With a hand-off area (pub), range 0 writes its
// state after chunk `meet` to it and range 1 forms only the sum of chunks meet+1 .. split-1,
// then adds the published state (a word per head: armed by range 1 at its start, set by
// range 0 once the state is written, cleared by range 1 after reading it; every wait on it
// is bounded, and the grid is launched cooperatively so that both ranges are resident). In
// the parts schedule range r adds the aggregates of ranges < r written by parts_tc.
//
// Operand layouts (128-byte swizzle, 1024-byte aligned atoms, 16-byte chunk c of row
// r at chunk c ^ (r % 8)): Q, K, V tiles as TMA loads them ([64 tokens][64 features]
// per atom; K atoms have 16 extra rows: row 64 holds bf16 z_{c-1}, rows 65-79 zero);
// phi(Q), phi(K) read K-major for S' and inter; phi(K), V read MN-major (K = tokens)
// for the update, the key sum and PV; P [64 queries][64 keys] K-major; the ones tile
// [16][64 tokens] K-major.
#include "la_tc_common.cuh"

namespace la {

constexpr int FWD_THREADS = 1024;
constexpr int NFW = 12;  // F warps

template <int D, int DV>
struct FwdLayout {
    // dv = 64: the key sum and the denominator ride in lanes 64-127 of the M = 128 products
    // whose A operand is V^T (rows 64-127 of that operand read an atom of ones kept after
    // every V stage), so no key-sum MMA and no z row in the K tile
    static constexpr bool ZL = DV == 64;
    // d = dv = 64: the scores S' no longer depend on the state (no z row), so the MMA thread
    // issues them two chunks ahead; a 5-stage ring keeps their operands landed in time
    static constexpr bool AHEAD = D == 64 && DV == 64;
    static constexpr int NST = AHEAD ? 5 : 3;
    // d = dv = 64: state-only chunks (range 1 of the fused schedule) stream in stages of two
    // chunks, one 128-row box per tensor, since an SM's copy engine takes almost as long for a
    // 64-row box as for a 128-row one. Two such stages lie over the ring's Q and K slots (below
    // its ones atoms), which the main chunks take over once their products are done. (At
    // d = 128 two 64 KB stages are too few for the load, phi and update round trip: there the
    // state-only chunks go through the ring itself, 64 rows at a time.)
    static constexpr bool AGG2 = AHEAD;
    static constexpr int AGGR = 2 * CH;
    static constexpr int AKB = D / 64 * AGGR * 128;
    static constexpr int AVB = DV / 64 * AGGR * 128;
    static constexpr int AST = AKB + AVB;
    static constexpr int QB = D / 64 * ATOM;
    static constexpr int KB = D / 64 * ATOMK;
    static constexpr int VB = (ZL ? 2 : DV / 64) * ATOM;
    static constexpr int Q0 = 0;
    static constexpr int K0 = Q0 + NST * QB;     // an M=128 read past the last Q atom lands here
    static constexpr int V0 = K0 + NST * KB;
    static constexpr int PT = V0 + NST * VB;     // P, two buffers
    static constexpr int OT = PT + 2 * ATOM;     // out tile
    static constexpr int ONES = OT + DV / 64 * ATOM;  // 16 x 64 bf16 ones (2 KB, 1024-aligned)
    static constexpr int RDEN = ONES + 2048;          // 2 x 64 floats
    static constexpr int BAR = RDEN + 2 * 64 * 4;
    static constexpr int NBAR = 3 * NST + 20;
    static constexpr int MISC = BAR + 8 * NBAR;
    static constexpr int TOTAL = MISC + 16;
    static constexpr int ALLOC = TOTAL + 1024;
};

// TMEM column map (512 columns allocated)
constexpr uint32_t TM_M = 0;     // M^T f32, d columns
constexpr uint32_t TM_A = 128;   // M^T bf16, two per column: d/2 columns (A operand of inter)
__device__ __forceinline__ uint32_t tm_s(int buf) { return 192u + 80u * buf; }  // S', 80 columns each
__device__ __forceinline__ uint32_t tm_o(int buf) { return 352u + 64u * buf; }  // O^T, 64 columns each
constexpr uint32_t TM_Z = 480;   // z f32, lane = feature, 16 equal columns

// Hand-off words of the fused schedule's state hand-off (arbitrary tags, so that a stale or
// uninitialised word is never taken for either)
constexpr int PUB_ARMED = 0x4C410001;
constexpr int PUB_DONE = 0x4C410002;

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Bounded wait for a hand-off word written by another block of the same (cooperative) grid.
__device__ __forceinline__ bool wait_word(const int* p, int want, volatile int* abort_flag) {
    const unsigned long long t0 = clock64();
    while (ld_acquire_gpu(p) != want) {
        if (*abort_flag) return false;
        if (clock64() - t0 > LA_WAIT_CYCLES) return false;
    }
    return true;
}

// bf16 z_i into row 64 (a multiple of 8: no swizzle offset) of a K tile with atoms ATOMK apart
__device__ __forceinline__ void put_zrow(uint8_t* ktile, int i, float z) {
    *reinterpret_cast<__nv_bfloat16*>(ktile + (i >> 6) * ATOMK + 64 * 128 + (i & 63) * 2) = __float2bfloat16_rn(z);
}

// 16 f32 values -> 8 words of two bf16 (low half = even index)
__device__ __forceinline__ void pack16_bf16(const uint32_t* x, uint32_t* a) {
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = pack_bf16(__uint_as_float(x[2 * k]), __uint_as_float(x[2 * k + 1]));
}

// SEG: the state after every segment is written too; PUB: the fused schedule's state hand-off
// (each compiled separately, so that the other calls run without the bookkeeping)
template <int D, int DV, bool SEG, bool PUB>
__global__ void __launch_bounds__(FWD_THREADS, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                  const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mo,
                  const __grid_constant__ CUtensorMap mk2, const __grid_constant__ CUtensorMap mv2, FwdTcParams p) {
    using L = FwdLayout<D, DV>;
    constexpr int NST = L::NST;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    float* rden = reinterpret_cast<float*>(sm + L::RDEN);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint64_t* full = bars + 0;             // [NST] TMA landed
    uint64_t* empty = bars + NST;          // [NST] stage free (MMA commit)
    uint64_t* phib = bars + 2 * NST;       // [NST] phi applied (F)
    uint64_t* s_full = bars + 3 * NST;     // [2] S' ready (MMA commit)
    uint64_t* s_free = s_full + 2;         // [2] S' read (S)
    uint64_t* p_full = s_full + 4;         // [2] P and 1/den written (S)
    uint64_t* o_full = s_full + 6;         // [2] O^T ready (MMA commit)
    uint64_t* o_free = s_full + 8;         // [2] O^T and 1/den read (E)
    uint64_t* upd_done = s_full + 10;      // state update finished (MMA commit)
    uint64_t* mt_ready = s_full + 11;      // bf16 M^T written and TMEM M read (R)
    uint64_t* drain = s_full + 12;         // all MMAs finished (MMA thread only)
    uint64_t* zrow_ready = s_full + 13;    // z before the next main chunk in its K tile's row 64 (E, then R)
    uint64_t* afull = s_full + 14;         // [2] state-only stage landed (TMA)
    uint64_t* aempty = afull + 2;          // [2] state-only stage free (MMA commit)
    uint64_t* aphib = afull + 4;           // [2] phi applied to its keys (F)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H;
    const int nch = (int)((p.T + CH - 1) / CH);
    // Fused schedule with a hand-off (pub set): range 0 publishes its state after chunk meet,
    // and range 1 sums only chunks meet+1 .. split-1 before adding it (blocks co-resident: the
    // grid is launched cooperatively).
    const bool publish = PUB && p.split > 0;
    int main_begin, main_end, n_agg = 0, nws = 0, agg_begin = 0;
    if (p.split > 0) {
        main_begin = r == 0 ? 0 : p.split;
        main_end = r == 0 ? p.split : nch;
        n_agg = r == 0 ? 0 : (publish ? p.split - p.meet - 1 : p.split);
        agg_begin = publish ? p.meet + 1 : 0;
    } else {
        main_begin = r * p.chunks_per_range;
        main_end = min(nch, main_begin + p.chunks_per_range);
        nws = r;
    }
    const int n_main = main_end - main_begin;
    const int n_ast = L::AGG2 ? (n_agg + 1) / 2 : 0;  // state-only stages of two chunks
    const int n_ring_agg = L::AGG2 ? 0 : n_agg;       // state-only chunks through the ring
    const int nchunks = n_ring_agg + n_main;          // chunks streamed through the ring
    static_assert(!L::AGG2 || 2 * L::AST <= L::V0, "state-only stages over the ring's Q and K slots");
    const bool writes_state = (r == p.nranges - 1);
    const float* agg = p.ws ? p.ws + (int64_t)bh * (p.nranges - 1) * p.rec : nullptr;

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::NBAR; ++i) mbar_init(&bars[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
        tma_prefetch_desc(&mo);
        if (n_agg > 0) {
            tma_prefetch_desc(&mk2);
            tma_prefetch_desc(&mv2);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_holder, 512);
        tmem_relinquish();
    }
    if (warp >= 2 && warp < 6) {  // the ones tile of the key-sum MMA: 2048 bytes of bf16 1.0
        const uint32_t one2 = 0x3F803F80u;
        reinterpret_cast<uint4*>(sm + L::ONES)[threadIdx.x - 64] = make_uint4(one2, one2, one2, one2);
        fence_proxy_async_smem();
    }
    if constexpr (L::ZL) {  // the ones atoms after the V stages
        const uint32_t one2 = 0x3F803F80u;
        for (int i = threadIdx.x; i < NST * (ATOM / 16); i += FWD_THREADS)
            *reinterpret_cast<uint4*>(sm + L::V0 + (i / (ATOM / 16)) * L::VB + ATOM + (i % (ATOM / 16)) * 16) =
                make_uint4(one2, one2, one2, one2);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // Launched as a programmatic dependent of the previous kernel in the stream: the set-up
    // above may overlap that kernel's tail, but nothing in global memory is read or written
    // before it has completed. This block lets the next such launch start its own set-up.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
    if (publish && r == 1 && threadIdx.x == 0) atomicExch(&p.pub_flag[bh], PUB_ARMED);

    if (warp == 0) {
        // ======================================================== TMA producer
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();  // q, k, v are read once
            // state-only stages: keys and values of chunks agg_begin + 2a and + 2a + 1 (when n_agg
            // is odd the last stage's second chunk, chunk split, is loaded and not used)
            int issued_a = 0;
            for (int a = 0; a < n_ast; ++a) {
                const int s = a & 1;
                if (a >= 2 && !mbar_wait(&aempty[s], ((a >> 1) - 1) & 1, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    break;
                }
                const int t = (agg_begin + 2 * a) * CH;
                uint8_t* st = sm + L::Q0 + s * L::AST;
                mbar_expect_tx(&afull[s], (D + DV) * L::AGGR * 2);
#pragma unroll
                for (int a2 = 0; a2 < D / 64; ++a2)
                    tma_load_4d_hint(st + a2 * L::AGGR * 128, &mk2, &afull[s], a2 * 64, t, h, b, pol);
#pragma unroll
                for (int a2 = 0; a2 < DV / 64; ++a2)
                    tma_load_4d_hint(st + L::AKB + a2 * L::AGGR * 128, &mv2, &afull[s], a2 * 64, t, h, b, pol);
                ++issued_a;
            }
            // the ring lies over those stages: their products must be done before it is loaded
            bool ok_a = issued_a == n_ast;
            for (int a = max(0, issued_a - 2); a < issued_a; ++a) {
                if (ok_a && !mbar_wait(&aempty[a & 1], (a >> 1) & 1, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    ok_a = false;
                }
                if (!ok_a) mbar_wait_drain(&afull[a & 1], (a >> 1) & 1);
            }
            int issued = 0;
            for (int g = 0; ok_a && g < nchunks; ++g) {
                const int s = g % NST;
                if (g >= NST && !mbar_wait(&empty[s], ((g / NST) - 1) & 1, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    break;
                }
                const bool is_main = g >= n_ring_agg;
                const int t = (is_main ? main_begin + g - n_ring_agg : agg_begin + g) * CH;
                mbar_expect_tx(&full[s], ((is_main ? D : 0) + D + DV) * CH * 2);
#pragma unroll
                for (int a = 0; a < D / 64; ++a) {
                    if (is_main)
                        tma_load_4d_hint(sm + L::Q0 + s * L::QB + a * ATOM, &mq, &full[s], a * 64, t, h, b, pol);
                    tma_load_4d_hint(sm + L::K0 + s * L::KB + a * ATOMK, &mk, &full[s], a * 64, t, h, b, pol);
                }
#pragma unroll
                for (int a = 0; a < DV / 64; ++a)
                    tma_load_4d_hint(sm + L::V0 + s * L::VB + a * ATOM, &mv, &full[s], a * 64, t, h, b, pol);
                ++issued;
            }
            for (int g = max(0, issued - NST); g < issued; ++g) mbar_wait_drain(&full[g % NST], (g / NST) & 1);
        }
    } else if (warp == 1) {
        // ======================================================== MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16(128, L::ZL ? CH : KROWS, 0, 0);  // S' = phiQ [phiK; z]^T
            constexpr uint32_t id_u = idesc_bf16(128, D, 1, 1);      // M^T += V^T phiK
            constexpr uint32_t id_pv = idesc_bf16(128, CH, 1, 0);    // O^T += V^T P^T
            constexpr uint32_t id_in = idesc_bf16(128, CH, 0, 0);    // O^T = M^T phiQ^T
            constexpr uint32_t id_z = idesc_bf16(128, 16, 1, 0);     // z (x16) += phiK^T 1
            // Descriptors of stage 0 / buffer 0; others differ only in the start-address field
            // (bits 0-13, address >> 4), which stays below 2^14 for any shared-memory address,
            // so an offset is added to the descriptor directly.
            const uint64_t dq0 = sdesc_sw128(smem_u32(sm + L::Q0), 16, 1024);     // phiQ, K-major
            const uint64_t dk0 = sdesc_sw128(smem_u32(sm + L::K0), 16, 1024);     // [phiK; z], K-major
            const uint64_t dku0 = sdesc_sw128(smem_u32(sm + L::K0), ATOMK, 1024); // phiK, MN-major
            const uint64_t dv0 = sdesc_sw128(smem_u32(sm + L::V0), ATOM, 1024);   // V, MN-major
            const uint64_t dp0 = sdesc_sw128(smem_u32(sm + L::PT), 16, 1024);     // P, K-major
            const uint64_t d1 = sdesc_sw128(smem_u32(sm + L::ONES), 16, 1024);    // ones, K-major
            auto off = [](uint32_t bytes) { return (uint64_t)(bytes >> 4); };
            const uint32_t ones0 = smem_u32(sm + L::V0 + ATOM);  // the ring's first ones atom (dv = 64)
            bool ok = true;
            int mt_waits = 0;
            auto wait = [&](uint64_t* bar, uint32_t parity) {
                if (ok && !mbar_wait(bar, parity, abort_flag)) {
                    record_timeout(p.status, abort_flag);
                    ok = false;
                }
                return ok;
            };
            auto update = [&](int s) {
                const uint64_t va = dv0 + off(s * L::VB), kb = dku0 + off(s * L::KB);
#pragma unroll
                for (int ks = 0; ks < CH / 16; ++ks)
                    mma_bf16_ss(tmem + TM_M, va + off(ks * 2048), kb + off(ks * 2048), id_u, 1);
                if constexpr (!L::ZL) {
#pragma unroll
                    for (int ks = 0; ks < CH / 16; ++ks)
                        mma_bf16_ss(tmem + TM_Z, kb + off(ks * 2048), d1 + off(ks * 32), id_z, 1);
                }
            };
            // the update over nk 16-token steps of state-only stage s: the 64-feature blocks of
            // V^T and phi(K) lie AGGR rows apart; at dv = 64 the second block of V^T is the ring's
            // first ones atom (64 rows of ones, read again for the stage's second chunk)
            auto update_agg = [&](int s, int nk) {
                const uint32_t ka = smem_u32(sm + L::Q0 + s * L::AST), va = ka + L::AKB;
                for (int kk = 0; kk < nk; ++kk) {
                    const uint32_t vrow = va + kk * 2048, krow = ka + kk * 2048;
                    const uint64_t vd = sdesc_sw128(vrow, L::ZL ? ones0 + (kk & 3) * 2048 - vrow : L::AGGR * 128, 1024);
                    const uint64_t kd = sdesc_sw128(krow, L::AGGR * 128, 1024);
                    mma_bf16_ss(tmem + TM_M, vd, kd, id_u, 1);
                    if constexpr (!L::ZL) mma_bf16_ss(tmem + TM_Z, kd, d1 + off((kk & 3) * 32), id_z, 1);
                }
            };
            // S'_m of main chunk m
            auto scores = [&](int m) {
                const int g = n_ring_agg + m, s = g % NST, buf = m & 1;
                const uint64_t qd = dq0 + off(s * L::QB), kd = dk0 + off(s * L::KB);
                if (!wait(&phib[s], (g / NST) & 1)) return false;
                if (m >= 2 && !wait(&s_free[buf], ((m >> 1) - 1) & 1)) return false;
                if (!L::ZL && !wait(zrow_ready, m & 1)) return false;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_bf16_ss(tmem + tm_s(buf), qd + off((ks >> 2) * ATOM + (ks & 3) * 32),
                                kd + off((ks >> 2) * ATOMK + (ks & 3) * 32), id_s, ks != 0);
                mma_commit(&s_full[buf]);
                return true;
            };
            // inter_m and update_m of main chunk m
            auto state_part = [&](int m) {
                const int g = n_ring_agg + m, s = g % NST, buf = m & 1;
                const uint64_t qd = dq0 + off(s * L::QB);
                if (!wait(mt_ready, mt_waits++ & 1)) return false;
                if (m >= 2 && !wait(&o_free[buf], ((m >> 1) - 1) & 1)) return false;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_bf16_ts(tmem + tm_o(buf), tmem + TM_A + ks * 8, qd + off((ks >> 2) * ATOM + (ks & 3) * 32),
                                id_in, ks != 0);
                update(s);
                mma_commit(upd_done);
                return true;
            };
            auto front = [&](int m) { return scores(m) && state_part(m); };
            if (n_agg > 0) {
                wait(mt_ready, mt_waits++ & 1);  // initial state in TMEM
                tc_fence_after();
                for (int a = 0; ok && a < n_ast; ++a) {
                    const int s = a & 1;
                    if (!wait(&aphib[s], (a >> 1) & 1)) break;
                    tc_fence_after();
                    update_agg(s, min(2, n_agg - 2 * a) * (CH / 16));
                    mma_commit(&aempty[s]);
                }
                for (int g = 0; ok && g < n_ring_agg; ++g) {
                    const int s = g % NST;
                    if (!wait(&phib[s], (g / NST) & 1)) break;
                    tc_fence_after();
                    update(s);
                    mma_commit(&empty[s]);
                }
                if (ok) mma_commit(upd_done);
            }
            if constexpr (L::AHEAD) {
                if (ok && n_main > 0) ok = scores(0) && state_part(0) && (n_main < 2 || scores(1));
            } else {
                if (ok && n_main > 0) front(0);
            }
            for (int m = 0; ok && m < n_main; ++m) {
                const int g = n_ring_agg + m, s = g % NST, buf = m & 1;
                if (!wait(&p_full[buf], (m >> 1) & 1)) break;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < CH / 16; ++ks)
                    mma_bf16_ss(tmem + tm_o(buf), dv0 + off(s * L::VB + ks * 2048), dp0 + off(buf * ATOM + ks * 32),
                                id_pv, 1);
                mma_commit(&o_full[buf]);
                mma_commit(&empty[s]);
                if constexpr (L::AHEAD) {  // the state chain first; the scores two chunks ahead
                    if (m + 1 < n_main && !state_part(m + 1)) break;
                    if (m + 2 < n_main && !scores(m + 2)) break;
                } else {
                    if (m + 1 < n_main && !front(m + 1)) break;
                }
            }
            mma_commit(drain);
            mbar_wait_drain(drain, 0);
        }
    } else if (warp >= 4 && warp < 8) {
        // ======================================================== R: z row and state re-cast
        const int ct = threadIdx.x - 128;
        const int q = warp & 3;
        const int j = 32 * q + lane;              // dv row of M^T; feature of z
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const bool has_row = 32 * q < DV;         // warp-uniform
        const bool has_z = 32 * q < D;            // warp-uniform
        const bool zlanes = L::ZL && q == 2;      // lanes 64-95 of M^T hold z^T (dv = 64)
        auto recast = [&]() {
            if (!has_row && !zlanes) return;
#pragma unroll 1
            for (int i0 = 0; i0 < D; i0 += 16) {
                uint32_t x[16], a[8];
                tmem_ld16(tmem + TM_M + lane_base + i0, x);
                tmem_wait_ld();
                pack16_bf16(x, a);
                tmem_st8(tmem + TM_A + lane_base + i0 / 2, a);
            }
            tmem_wait_st();
        };
        // the f32 state (M^T and z in TMEM) to [D][DV] and [D] arrays (either may be null);
        // two TMEM loads in flight per wait
        auto store_state = [&](float* Md, float* zd) {
            if (L::ZL && zd && zlanes) {  // every lane of the quarter holds all of z
#pragma unroll 1
                for (int i0 = 0; i0 < D; i0 += 32) {
                    uint32_t x[16], y[16];
                    tmem_ld16(tmem + TM_M + lane_base + i0, x);
                    tmem_ld16(tmem + TM_M + lane_base + i0 + 16, y);
                    tmem_wait_ld();
                    if (lane == 0) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            zd[i0 + e] = __uint_as_float(x[e]);
                            zd[i0 + 16 + e] = __uint_as_float(y[e]);
                        }
                    }
                }
            } else if (!L::ZL && zd && has_z) {
                const uint32_t zb = tmem_ld1(tmem + TM_Z + lane_base);
                tmem_wait_ld();
                zd[j] = __uint_as_float(zb);
            }
            if (Md && has_row) {
#pragma unroll 1
                for (int i0 = 0; i0 < D; i0 += 32) {
                    uint32_t x[16], y[16];
                    tmem_ld16(tmem + TM_M + lane_base + i0, x);
                    tmem_ld16(tmem + TM_M + lane_base + i0 + 16, y);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        Md[(int64_t)(i0 + e) * DV + j] = __uint_as_float(x[e]);
                        Md[(int64_t)(i0 + 16 + e) * DV + j] = __uint_as_float(y[e]);
                    }
                }
            }
        };
        // the f32 state of another block ([D][DV] and [D], read through L2) added into TMEM
        auto add_state = [&](const float* Mp, const float* zp) {
            if (has_row) {
#pragma unroll 1
                for (int i0 = 0; i0 < D; i0 += 16) {
                    uint32_t x[16];
                    tmem_ld16(tmem + TM_M + lane_base + i0, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        x[e] = __float_as_uint(__uint_as_float(x[e]) + __ldcg(Mp + (int64_t)(i0 + e) * DV + j));
                    tmem_st16(tmem + TM_M + lane_base + i0, x);
                }
            }
            if (L::ZL && zlanes) {  // z^T in every lane of the quarter
#pragma unroll 1
                for (int i0 = 0; i0 < D; i0 += 16) {
                    uint32_t x[16];
                    tmem_ld16(tmem + TM_M + lane_base + i0, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = __float_as_uint(__uint_as_float(x[e]) + __ldcg(zp + i0 + e));
                    tmem_st16(tmem + TM_M + lane_base + i0, x);
                }
            } else if (!L::ZL && has_z) {
                const uint32_t zb = tmem_ld1(tmem + TM_Z + lane_base);
                tmem_wait_ld();
                tmem_st1(tmem + TM_Z + lane_base, __float_as_uint(__uint_as_float(zb) + __ldcg(zp + j)));
            }
            tmem_wait_st();
        };
        // SEG: the state after the chunk that ends a segment (or the sequence) is written before
        // the re-cast. The next such chunk and its segment are tracked incrementally (no integer
        // division on the update -> re-cast path).
        int seg_next = 0, seg_idx = 0;
        if constexpr (SEG) {
            seg_next = (main_begin / p.seg_chunks + 1) * p.seg_chunks - 1;
            seg_idx = main_begin / p.seg_chunks;
        }
        bool ok = true;
        int upd = 0;
        const int n_upd = (n_agg > 0 ? 1 : 0) + n_main;
        for (int u = 0; u < n_upd; ++u) {
            ok = bar_and(4, 128, mbar_wait(upd_done, upd++ & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            if (publish && r == 1 && u == 0) {
                // range 1, its sum of chunks meet+1 .. split-1 done: add range 0's state after
                // chunk meet, then clear the hand-off word for the next call (which re-arms it)
                bool got = true;
                if (ct == 0) {
                    got = wait_word(p.pub_flag + bh, PUB_DONE, abort_flag);
                    if (!got) record_timeout(p.status, abort_flag);
                }
                ok = bar_and(4, 128, got);
                if (!ok) break;
                const float* pm = p.pub + (int64_t)bh * p.rec;
                add_state(pm, pm + D * DV);
                named_bar_sync(4, 128);
                if (ct == 0) atomicExch(p.pub_flag + bh, 0);
            }
            // range 0: its state after chunk meet, published once the re-cast below is done
            const bool pub_here = publish && r == 0 && u == p.meet;
            if (pub_here) {
                float* pm = p.pub + (int64_t)bh * p.rec;
                store_state(pm, pm + D * DV);
                __threadfence();
            }
            if constexpr (SEG) {  // (range 1's state-only chunks: no output)
                if (n_agg == 0 || u > 0) {
                    const int c = main_begin + (n_agg > 0 ? u - 1 : u);
                    if (c == seg_next || c == nch - 1) {
                        const int64_t sb = (int64_t)seg_idx * gridDim.y + bh;
                        store_state(p.M_seg ? p.M_seg + sb * D * DV : nullptr, p.z_seg ? p.z_seg + sb * D : nullptr);
                        seg_next += p.seg_chunks;
                        ++seg_idx;
                    }
                }
            }
            if (L::ZL && u + 1 < n_upd) {
                recast();  // z^T rides along in lanes 64-95
                tc_fence_before();
                named_bar_sync(4, 128);
                if (ct == 0) mbar_arrive(mt_ready);
            } else if (u + 1 < n_upd) {
                // the main chunk after this update: its S' reads z from row 64 of its K tile
                const int mnext = n_agg > 0 ? u : u + 1;
                if (has_z) {
                    const uint32_t zb = tmem_ld1(tmem + TM_Z + lane_base);
                    tmem_wait_ld();
                    put_zrow(sm + L::K0 + ((n_ring_agg + mnext) % NST) * L::KB, j, __uint_as_float(zb));
                    fence_proxy_async_smem();
                }
                named_bar_sync(4, 128);
                if (ct == 0) mbar_arrive(zrow_ready);
                recast();
                tc_fence_before();
                named_bar_sync(4, 128);
                if (ct == 0) mbar_arrive(mt_ready);
            } else if (writes_state) {
                store_state(p.M_out ? p.M_out + (int64_t)bh * D * DV : nullptr,
                            p.z_out ? p.z_out + (int64_t)bh * D : nullptr);
            }
            // (the branch above ended with a barrier of the R warps, after every thread's fence;
            // range 1 armed the word at its start)
            if (pub_here && ct == 0) {
                __threadfence();
                if (wait_word(p.pub_flag + bh, PUB_ARMED, abort_flag))
                    st_release_gpu(p.pub_flag + bh, PUB_DONE);
                else
                    record_timeout(p.status, abort_flag);
            }
        }
        if (!ok && ct == 0) record_timeout(p.status, abort_flag);
    } else if (warp >= 8 && warp < 16) {
        // ======================================================== E: initial state, then out = O / den
        const int ct = threadIdx.x - 256;
        const int q = warp & 3;
        const int hf = (warp - 8) >> 2;           // rows 64hf.. of the initial state; tokens 32hf.. of a chunk
        const int j = 32 * q + lane;              // dv index: row of O^T and of M^T
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const bool has_row = 32 * q < DV;         // warp-uniform
        if (has_row) {
            // column j of the initial state M_in (+ range aggregates), rows [64hf, 64hf + 64)
            // (range 1 with a hand-off starts from zero: range 0's published state holds M_in)
            const float* src = p.M_in && !(publish && r == 1) ? p.M_in + (int64_t)bh * D * DV + j : nullptr;
#pragma unroll 1
            for (int i0 = 64 * hf; i0 < D && i0 < 64 * hf + 64; i0 += 16) {
                uint32_t x[16], a[8];
                if (src) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = __float_as_uint(__ldg(src + (int64_t)(i0 + e) * DV));
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = 0u;
                }
#pragma unroll 1
                for (int pp = 0; pp < nws; ++pp) {
                    const float* ag = agg + pp * p.rec + (int64_t)i0 * DV + j;
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = __float_as_uint(__uint_as_float(x[e]) + __ldg(ag + e * DV));
                }
                tmem_st16(tmem + TM_M + lane_base + i0, x);
                pack16_bf16(x, a);
                tmem_st8(tmem + TM_A + lane_base + i0 / 2, a);
            }
            tmem_wait_st();
        }
        if (L::ZL && q == 2) {
            // z_in (+ range aggregates) as the row z^T in every lane 64-95 of M^T (f32 and
            // bf16), columns [64hf, 64hf + 64)
#pragma unroll 1
            for (int i0 = 64 * hf; i0 < D && i0 < 64 * hf + 64; i0 += 16) {
                uint32_t x[16], a[8];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float zz = p.z_in && !(publish && r == 1) ? p.z_in[(int64_t)bh * D + i0 + e] : 0.f;
                    for (int pp = 0; pp < nws; ++pp) zz += agg[pp * p.rec + D * DV + i0 + e];
                    x[e] = __float_as_uint(zz);
                }
                tmem_st16(tmem + TM_M + lane_base + i0, x);
                pack16_bf16(x, a);
                tmem_st8(tmem + TM_A + lane_base + i0 / 2, a);
            }
            tmem_wait_st();
        }
        if (!L::ZL && hf == 0 && 32 * q < D) {
            // z_in (+ range aggregates) into TMEM; with no state-only chunks before the first
            // main chunk it is also z before that chunk (row 64 of its K tile, stage 0)
            float zz = p.z_in && !(publish && r == 1) ? p.z_in[(int64_t)bh * D + j] : 0.f;
            for (int pp = 0; pp < nws; ++pp) zz += agg[pp * p.rec + D * DV + j];
            tmem_st1(tmem + TM_Z + lane_base, __float_as_uint(zz));
            tmem_wait_st();
            if (n_agg == 0) {
                put_zrow(sm + L::K0, j, zz);
                fence_proxy_async_smem();
            }
        }
        tc_fence_before();
        named_bar_sync(3, 256);
        if (ct == 0) {
            mbar_arrive(mt_ready);
            if (!L::ZL && n_agg == 0) mbar_arrive(zrow_ready);
        }

        // Thread l of the warp stores, per stmatrix, row (l % 8) of matrix l / 8: features
        // f0 .. f0+7 (f0 = 32q + 8(l / 8)) of token 32hf + 8i + (l % 8), i = 0..3; the row's
        // 16-byte chunk of the swizzled [token][feature] tile:
        const int f0 = 32 * q + 8 * (lane >> 3);
        const uint32_t ot_row = smem_u32(sm + L::OT + (f0 >> 6) * ATOM) + (uint32_t)((((f0 & 63) >> 3) ^ (lane & 7)) << 4);
        const uint64_t pol = l2_evict_first_policy();  // out is written once
        bool ok = true;
        for (int m = 0; m < n_main; ++m) {
            const int buf = m & 1;
            // (with z in lanes 64-127 the E warps form 1/den themselves and read nothing the S
            // warps write, and PV_m's commit already follows P_m. Nor do the S warps wait for E
            // there, so P_{m+2} may complete p_full[buf]'s next phase before E looks at it: E
            // does not wait on p_full at all then.)
            ok = bar_and(3, 256, mbar_wait(&o_full[buf], (m >> 1) & 1, abort_flag) &&
                                     (L::ZL || mbar_wait(&p_full[buf], (m >> 1) & 1, abort_flag)));
            if (!ok) break;
            tc_fence_after();
            if (L::ZL && q == 2) {
                // lanes 64-95 of O^T all hold phi(q_t).z + sum_j P_tj for token t = 32hf + column;
                // in the fragment layout threads 0-3 hold the 32 tokens between them
                uint32_t x[16];
                tmem_ld16x256_x4(tmem + tm_o(buf) + lane_base + 32 * hf, x);
                tmem_wait_ld();
                if (lane < 4) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        float* rd = rden + buf * 64 + 32 * hf + 8 * k + 2 * lane;
                        rd[0] = 1.f / (__uint_as_float(x[4 * k]) + p.eps);
                        rd[1] = 1.f / (__uint_as_float(x[4 * k + 1]) + p.eps);
                    }
                }
            }
            if (ct == 0) tma_store_wait_read0();  // previous out tile read by the TMA unit
            named_bar_sync(3, 256);
            if (has_row) {
                // O^T lanes 32q + 16lb + {0..15}, tokens 32hf + {0..31}: two loads in the fragment layout
                uint32_t x[2][16];
                tmem_ld16x256_x4(tmem + tm_o(buf) + lane_base + 32 * hf, x[0]);
                tmem_ld16x256_x4(tmem + tm_o(buf) + lane_base + (16u << 16) + 32 * hf, x[1]);
                const float2* rd2 = reinterpret_cast<const float2*>(rden + buf * 64 + 32 * hf + 2 * (lane & 3));
                float2 rd[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) rd[i] = rd2[4 * i];  // tokens 8i + 2(l % 4) + {0, 1}
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t w[4];  // matrix m = 2lb + hh: features 32q + 16lb + 8hh + {0..7}, tokens 8i + {0..7}
                    const uint64_t rdi = f2_pack(rd[i].x, rd[i].y);
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        const uint32_t* r = x[m >> 1] + 4 * i + 2 * (m & 1);
                        const uint64_t o = f2_mul(f2_pack(__uint_as_float(r[0]), __uint_as_float(r[1])), rdi);
                        w[m] = pack_bf16(f2_lo(o), f2_hi(o));
                    }
                    stmatrix_x4_trans(ot_row + (uint32_t)((32 * hf + 8 * i + (lane & 7)) * 128), w);
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            named_bar_sync(3, 256);
            if (ct == 0) {
                mbar_arrive(&o_free[buf]);
                const int t = (main_begin + m) * CH;
#pragma unroll
                for (int a = 0; a < DV / 64; ++a)
                    tma_store_4d_hint(&mo, sm + L::OT + a * ATOM, a * 64, t, h, b, pol);
                tma_store_commit();
            }
        }
        if (!ok && ct == 0) record_timeout(p.status, abort_flag);
        if (ct == 0) tma_store_wait_all0();
    } else if (warp >= 16 && warp < 18) {
        // ======================================================== S: P and 1/den
        const int ct = threadIdx.x - 512;
        const int q = warp & 3;                   // 0 or 1
        const int t = 32 * q + lane;              // query row in the chunk
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        bool ok = true;
        for (int m = 0; m < n_main; ++m) {
            const int buf = m & 1;
            bool w = mbar_wait(&s_full[buf], (m >> 1) & 1, abort_flag);
            if (!L::ZL && m >= 2) w = w && mbar_wait(&o_free[buf], ((m - 2) >> 1) & 1, abort_flag);  // rden[buf] consumed
            ok = bar_and(2, 64, w);
            if (!ok) break;
            tc_fence_after();
            uint8_t* prow = sm + L::PT + buf * ATOM + t * 128;
            uint64_t rowsum2 = 0;  // (even keys, odd keys) partial sums of the f32 scores
            const uint32_t srow = tmem + tm_s(buf) + lane_base;
            // keys 32h .. 32h+31 of the row from x[0..32): P as bf16 into the swizzled tile, row sum
            auto half = [&](const uint32_t* x, int h, bool diag) {
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    uint32_t pk[4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int c0 = 32 * h + 8 * g8 + 2 * jj;
                        float s0 = __uint_as_float(x[8 * g8 + 2 * jj]);
                        float s1 = __uint_as_float(x[8 * g8 + 2 * jj + 1]);
                        if (diag) {
                            s0 = (c0 <= t) ? s0 : 0.f;
                            s1 = (c0 + 1 <= t) ? s1 : 0.f;
                        }
                        pk[jj] = pack_bf16(s0, s1);
                        rowsum2 = f2_add(rowsum2, f2_pack(s0, s1));
                    }
                    *reinterpret_cast<uint4*>(prow + (((4 * h + g8) ^ (t & 7)) << 4)) =
                        make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            };
            uint32_t zq = 0;
            if (q == 0) {  // rows 0-31: keys 32-63 all lie after the row
                uint32_t x[32];
                tmem_ld32(srow, x);
                if constexpr (!L::ZL) zq = tmem_ld1(srow + 64);
                tmem_wait_ld();
                half(x, 0, true);
#pragma unroll
                for (int g8 = 4; g8 < 8; ++g8)
                    *reinterpret_cast<uint4*>(prow + ((g8 ^ (t & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
            } else {       // rows 32-63: keys 0-31 all lie before the row
                uint32_t x[32], y[32];
                tmem_ld32(srow, x);
                tmem_ld32(srow + 32, y);
                if constexpr (!L::ZL) zq = tmem_ld1(srow + 64);
                tmem_wait_ld();
                half(x, 0, false);
                half(y, 1, true);
            }
            if constexpr (!L::ZL)  // (dv = 64: the E warps form 1/den from lanes 64-95 of O^T)
                rden[buf * 64 + t] = 1.f / (__uint_as_float(zq) + (f2_lo(rowsum2) + f2_hi(rowsum2)) + p.eps);
            tc_fence_before();
            fence_proxy_async_smem();
            named_bar_sync(2, 64);
            if (ct == 0) {
                mbar_arrive(&s_free[buf]);
                mbar_arrive(&p_full[buf]);
            }
        }
        if (!ok && ct == 0) record_timeout(p.status, abort_flag);
    } else if (warp != 21 && warp != 25 && warp != 29 && warp != 31) {
        // ======================================================== F: phi (warps 2, 3, 18-30 but 21, 25, 29)
        const int fi = warp < 4 ? warp - 2 : 2 + (warp - 18) - (warp - 17) / 4;
        const int ct = fi * 32 + lane;
        // rows 65-79 of the K atoms feed only columns of S' that are never read; they are zeroed
        // unless the state-only stages of two chunks lie over them
        if (n_ast == 0) {
            for (int idx = ct; idx < NST * (D / 64) * 15 * 8; idx += 32 * NFW) {
                const int c16 = idx % 8, row = 65 + (idx / 8) % 15, sa = idx / (8 * 15);
                *reinterpret_cast<uint4*>(sm + L::K0 + sa * ATOMK + row * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
            }
        }
        bool ok = true;
        for (int a = 0; a < n_ast; ++a) {  // state-only stages of two chunks: phi on their keys (full chunks)
            const int s = a & 1;
            ok = bar_and(1, 32 * NFW, mbar_wait(&afull[s], (a >> 1) & 1, abort_flag));
            if (!ok) break;
            uint8_t* kt = sm + L::Q0 + s * L::AST;
            phi_tile<D, 32 * NFW>(kt, L::AGGR * 128, CH, ct, nullptr, p.phi_ident);
            if (2 * a + 1 < n_agg) phi_tile<D, 32 * NFW>(kt + CH * 128, L::AGGR * 128, CH, ct, nullptr, p.phi_ident);
            fence_proxy_async_smem();
            named_bar_sync(1, 32 * NFW);
            if (ct == 0) mbar_arrive(&aphib[s]);
        }
        for (int g = 0; ok && g < nchunks; ++g) {
            const int s = g % NST;
            const bool is_main = g >= n_ring_agg;
            ok = bar_and(1, 32 * NFW, mbar_wait(&full[s], (g / NST) & 1, abort_flag));
            if (!ok) break;
            const int64_t t0 = (int64_t)(is_main ? main_begin + g - n_ring_agg : agg_begin + g) * CH;
            const int valid = (int)min64(CH, p.T - t0);
            if (is_main) phi_tile<D, 32 * NFW>(sm + L::Q0 + s * L::QB, ATOM, CH, ct, nullptr, p.phi_ident);
            phi_tile<D, 32 * NFW>(sm + L::K0 + s * L::KB, ATOMK, valid, ct, nullptr, p.phi_ident);
            fence_proxy_async_smem();
            named_bar_sync(1, 32 * NFW);
            if (ct == 0) mbar_arrive(&phib[s]);
        }
        if (!ok && ct == 0) record_timeout(p.status, abort_flag);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D, int DV, bool SEG, bool PUB>
static cudaError_t launch_t(const FwdTcParams& p, int B, const CUtensorMap& mq, const CUtensorMap& mk,
                            const CUtensorMap& mv, const CUtensorMap& mo, const CUtensorMap& mk2,
                            const CUtensorMap& mv2, cudaStream_t s) {
    using L = FwdLayout<D, DV>;
    static_assert(L::ALLOC <= 227 * 1024, "shared memory budget");
    auto fn = fwd_tc_kernel<D, DV, SEG, PUB>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.nranges, B * p.H);
    cfg.blockDim = dim3(FWD_THREADS);
    cfg.dynamicSmemBytes = L::ALLOC;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // the state hand-off between the two ranges of a head needs every block resident at once
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = PUB ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, fn, mq, mk, mv, mo, mk2, mv2, p);
}

cudaError_t launch_fwd_tc(const FwdTcParams& p, int d, int dv, int B, const CUtensorMap& mq, const CUtensorMap& mk,
                          const CUtensorMap& mv, const CUtensorMap& mo, const CUtensorMap& mk2, const CUtensorMap& mv2,
                          cudaStream_t s) {
    const bool seg = p.M_seg || p.z_seg;
    const bool pub = p.pub != nullptr && p.split > 0;
    if (seg && p.seg_chunks <= 0) return cudaErrorInvalidValue;
    if (pub && (!p.pub_flag || p.meet < 0 || p.meet > p.split - 2)) return cudaErrorInvalidValue;
#define LA_FWD_SHAPE(DD, DDV)                                                                         \
    if (d == DD && dv == DDV) {                                                                       \
        if (seg) return pub ? launch_t<DD, DDV, true, true>(p, B, mq, mk, mv, mo, mk2, mv2, s)                  \
                            : launch_t<DD, DDV, true, false>(p, B, mq, mk, mv, mo, mk2, mv2, s);                \
        return pub ? launch_t<DD, DDV, false, true>(p, B, mq, mk, mv, mo, mk2, mv2, s)                          \
                   : launch_t<DD, DDV, false, false>(p, B, mq, mk, mv, mo, mk2, mv2, s);                        \
    }
    LA_FWD_SHAPE(128, 128)
    LA_FWD_SHAPE(128, 64)
    LA_FWD_SHAPE(64, 128)
    LA_FWD_SHAPE(64, 64)
#undef LA_FWD_SHAPE
    return cudaErrorInvalidValue;
}

}  // namespace la
