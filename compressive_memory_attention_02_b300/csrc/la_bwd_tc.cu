// Tensor-core (tcgen05 + TMEM + TMA) chunk kernels of the training backward, bf16
// storage, f32 accumulation. The page "Attention_Kernel_Mask" names the training-
// backward mode (table "Causal Attention Training and Inferencing") but prints no
// formula; these kernels apply the chain rule to the chunk form of that page's "chunk
// sequential mode" (mode 3), as the float32 kernels of la_bwd.cu do. For chunk c with
// the state (M, z) of every token before it and S = phi(Q_c) phi(K_c)^T kept for keys at
// or before the query:
//   D_t = phi(q_t).z + sum_j S_tj + eps,   out_t = (phi(q_t)^T M + sum_j S_tj v_j) / D_t
//   g_t = dout_t / D_t,   e_t = -(g_t . out_t),   dA_tj = g_t . v_j + e_t   (j <= t)
//   dphi(q_t) = M g_t + e_t z + sum_j dA_tj phi(k_j)
//   dphi(k_j) = sum_{t >= j} dA_tj phi(q_t) + R v_j + r,   dv_j = sum_{t >= j} S_tj g_t + R^T phi(k_j)
// with (R, r) the state gradient from every token after the chunk, and dx = dphi(x) phi'(x),
// phi'(x) = min(phi(x), 1).
//
//   bwd_dq_tc    one block per (chunk, b*H + h): S', O = phi(Q) M + P V, g, e, dA, dq, and
//                the chunk's share of the state gradient, phi(Q)^T G and phi(Q)^T e
//   bwd_dkdv_tc  one block per (chunk, b*H + h): S^T, dA^T, dv and dk
// The states before each chunk and (R, r) after it come from the ordered scans of
// la_bwd.cu over per-chunk records; G (bf16) and e (f32) pass from the first kernel to
// the second through the workspace.
//
// G, P and dA are formed in f32 inside the kernels; each enters its products as two bf16
// operands, a high part and the rounded remainder (x = hi + lo to ~16 bits), so that the
// cancellations in dq (M g + e z against the intra-chunk sum, and g . v_j + e inside dA)
// act on f32-accurate values; the other operands (phi, V, dout, the states) are bf16.
//
// Each block runs its steps in sequence (load, phi, MMAs, element-wise passes), with
// several blocks per SM overlapping each other. 256 threads: warp w may touch only TMEM
// lane quarter w % 4; per-token passes use warps 0 and 1 (lanes 0-63 = the chunk's
// tokens), per-feature passes all eight warps. Thread 0 issues the MMAs and their
// commits; every wait is a bounded mbarrier wait.
//
// Operand layouts (128-byte swizzle, 1024-byte aligned): token tiles [64 tokens][64
// features] per atom as TMA loads them (the dq kernel's K tile has 80 rows per atom: row
// 64 holds bf16 z, rows 65-79 zero); the state tile (M or R, bf16) [d rows][64 dv] per
// block of d * 128 bytes, read MN-major (K = d) and K-major (K = dv); P, dA and their
// transposes [64][64] K-major; the high and low parts of G, P and dA in adjacent tiles.
// Every A-operand tile of 64 rows is followed by at least one atom of shared memory (an
// M = 128 MMA reads 64 rows past it; those rows of the result are never used).
#include "la_bwd.h"
#include "la_tc_common.cuh"

namespace la {
namespace {

constexpr int BT = 256;  // threads per block

// f32 state record [D][DV] row-major (16-byte aligned) -> bf16 tile in the layout above.
template <int D, int DV>
__device__ __forceinline__ void state_to_tile(const float* rec, uint8_t* tile, int tid) {
    constexpr int N = D * DV / 8;  // 16-byte bf16 chunks
#pragma unroll 2
    for (int c = tid; c < N; c += BT) {
        const int i = c / (DV / 8), j0 = (c % (DV / 8)) * 8;
        const float4 a = __ldg(reinterpret_cast<const float4*>(rec + (int64_t)i * DV + j0));
        const float4 b = __ldg(reinterpret_cast<const float4*>(rec + (int64_t)i * DV + j0 + 4));
        const uint4 w = make_uint4(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w), pack_bf16(b.x, b.y), pack_bf16(b.z, b.w));
        *reinterpret_cast<uint4*>(tile + (j0 >> 6) * (D * 128) + i * 128 + ((((j0 & 63) >> 3) ^ (i & 7)) << 4)) = w;
    }
}

// Two f32 values as bf16 high parts (hi) and bf16 remainders (lo): x = hi + lo to ~16 bits.
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = pack_bf16(a, b);
    lo = pack_bf16(a - bf16lo(hi), b - bf16hi(hi));
}

// bf16 element (row, col) of a tile with 64-column atoms `astride` bytes apart
__device__ __forceinline__ uint32_t tile_off(int row, int col, int astride) {
    return (col >> 6) * astride + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + (col & 7) * 2;
}

__device__ __forceinline__ float tile_get(const uint8_t* tile, int row, int col, int astride) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + tile_off(row, col, astride)));
}

// Bounded wait by every thread of the block on the MMA-completion barrier; false (and the
// status recorded) if it ran out.
__device__ __forceinline__ bool block_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* status) {
    const bool ok = mbar_wait(bar, parity, abort_flag);
    if (!ok) record_timeout(status, abort_flag);
    return __syncthreads_and(ok) != 0;
}

// 16 f32 columns of TMEM (this thread's lane) starting at column col
__device__ __forceinline__ void ld16f(uint32_t taddr, float* x) {
    uint32_t r[16];
    tmem_ld16(taddr, r);
    tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) x[e] = __uint_as_float(r[e]);
}

}  // namespace

// ================================================================================ dq
template <int D, int DV>
struct DqLayout {
    static constexpr int QT = 0;                          // phi(Q), D/64 atoms (+ read-past room: KT)
    static constexpr int KT = QT + D / 64 * ATOM;         // [phi(K); z], D/64 atoms of 80 rows
    static constexpr int VT = KT + D / 64 * ATOMK;        // V, DV/64 atoms
    static constexpr int OT = VT + DV / 64 * ATOM;        // dout, DV/64 atoms
    static constexpr int PT = OT + DV / 64 * ATOM;        // P high, then low part [64][64]
    static constexpr int GT = PT + 2 * ATOM;              // G high (DV/64 atoms), then low part
    static constexpr int AT = GT + 2 * (DV / 64) * ATOM;  // dA high, then low part
    static constexpr int MT = AT + 2 * ATOM;              // state M (bf16), DV/64 blocks of D*128 bytes
    static constexpr int DEN = MT + D * DV * 2;           // 64 floats: D_t
    static constexpr int EV = DEN + 256;                  // 64 floats: e_t
    static constexpr int ZF = EV + 256;                   // D floats: z
    static constexpr int BAR = ZF + 512;
    static constexpr int MISC = BAR + 16;
    static constexpr int ALLOC = MISC + 16 + 1024;
    // TMEM columns
    static constexpr uint32_t TS = 0;                     // S' (80), later dA (64)
    static constexpr uint32_t TO = 128;                   // O (DV), later dphi(Q) (D)
    static constexpr uint32_t TR = TO + (D > DV ? D : DV);  // phi(Q)^T G (DV)
    static constexpr uint32_t NCOL = TR + DV <= 256 ? 256 : 512;
};

template <int D, int DV>
__global__ void __launch_bounds__(BT, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                     const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mdo,
                     BwdTcParams p) {
    using L = DqLayout<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint64_t* ld_full = bars + 0;   // TMA landed
    uint64_t* mma_done = bars + 1;  // the issued MMAs completed (one phase per step)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
    float* den = reinterpret_cast<float*>(sm + L::DEN);
    float* ev = reinterpret_cast<float*>(sm + L::EV);
    float* zf = reinterpret_cast<float*>(sm + L::ZF);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H;
    const int64_t t0 = (int64_t)c * CH;
    const int valid = (int)min64(CH, p.T - t0);
    const float* state = p.states + ((int64_t)bh * p.nch + c) * p.rec;

    if (tid == 0) {
        mbar_init(ld_full, 1);
        mbar_init(mma_done, 1);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (tid == 0) {
        const uint64_t pol = l2_evict_first_policy();
        mbar_expect_tx(ld_full, (2 * D + 2 * DV) * CH * 2);
        for (int a = 0; a < D / 64; ++a) {
            tma_load_4d_hint(sm + L::QT + a * ATOM, &mq, ld_full, a * 64, (int)t0, h, b, pol);
            tma_load_4d_hint(sm + L::KT + a * ATOMK, &mk, ld_full, a * 64, (int)t0, h, b, pol);
        }
        for (int a = 0; a < DV / 64; ++a) {
            tma_load_4d_hint(sm + L::VT + a * ATOM, &mv, ld_full, a * 64, (int)t0, h, b, pol);
            tma_load_4d_hint(sm + L::OT + a * ATOM, &mdo, ld_full, a * 64, (int)t0, h, b, pol);
        }
    }
    // meanwhile: the state before the chunk as bf16 tiles, z as f32 and as row 64 of the K
    // tile, rows 65-79 of the K tile zero
    state_to_tile<D, DV>(state, sm + L::MT, tid);
    if (tid < D) {
        const float z = state[D * DV + tid];
        zf[tid] = z;
        *reinterpret_cast<__nv_bfloat16*>(sm + L::KT + (tid >> 6) * ATOMK + 64 * 128 + (tid & 63) * 2) =
            __float2bfloat16_rn(z);
    }
    for (int i = tid; i < (D / 64) * 15 * 8; i += BT) {
        const int c16 = i % 8, row = 65 + (i / 8) % 15, a = i / (8 * 15);
        *reinterpret_cast<uint4*>(sm + L::KT + a * ATOMK + row * 128 + c16 * 16) = make_uint4(0, 0, 0, 0);
    }
    bool ok = block_wait(ld_full, 0, abort_flag, p.status);
    if (ok) {
        // phi in place; query and key rows past the end become 0 (they then add nothing to
        // any sum over tokens, and their g and e are 0 since dout is zero-filled there)
        phi_tile<D, BT>(sm + L::QT, ATOM, valid, tid, nullptr);
        phi_tile<D, BT>(sm + L::KT, ATOMK, valid, tid, nullptr);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    auto off = [](uint32_t bytes) { return (uint64_t)(bytes >> 4); };
    const uint64_t dQk = sdesc_sw128(smem_u32(sm + L::QT), 16, 1024);      // phi(Q), K-major
    const uint64_t dQm = sdesc_sw128(smem_u32(sm + L::QT), ATOM, 1024);    // phi(Q), MN-major (M or N = d)
    const uint64_t dKk = sdesc_sw128(smem_u32(sm + L::KT), 16, 1024);      // [phi(K); z], K-major
    const uint64_t dKm = sdesc_sw128(smem_u32(sm + L::KT), ATOMK, 1024);   // phi(K), MN-major
    const uint64_t dVk = sdesc_sw128(smem_u32(sm + L::VT), 16, 1024);      // V, K-major (K = dv)
    const uint64_t dVm = sdesc_sw128(smem_u32(sm + L::VT), ATOM, 1024);    // V, MN-major (K = keys)
    const uint64_t dMm = sdesc_sw128(smem_u32(sm + L::MT), D * 128, 1024); // M, MN-major (K = d, N = dv)
    const uint64_t dMk = sdesc_sw128(smem_u32(sm + L::MT), 16, 1024);      // M, K-major (N = d, K = dv)
    const uint64_t dPk = sdesc_sw128(smem_u32(sm + L::PT), 16, 1024);
    const uint64_t dGk = sdesc_sw128(smem_u32(sm + L::GT), 16, 1024);      // G, K-major (K = dv)
    const uint64_t dGm = sdesc_sw128(smem_u32(sm + L::GT), ATOM, 1024);    // G, MN-major (K = tokens)
    const uint64_t dAk = sdesc_sw128(smem_u32(sm + L::AT), 16, 1024);
    uint32_t phase = 0;

    // ---- S' = phi(Q) [phi(K); z]^T, O = phi(Q) M
    if (ok && tid == 0) {
        constexpr uint32_t id_s = idesc_bf16(128, KROWS, 0, 0);
        constexpr uint32_t id_o = idesc_bf16(128, DV, 0, 1);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t qo = (ks >> 2) * ATOM + (ks & 3) * 32;
            mma_bf16_ss(tmem + L::TS, dQk + off(qo), dKk + off((ks >> 2) * ATOMK + (ks & 3) * 32), id_s, ks != 0);
            mma_bf16_ss(tmem + L::TO, dQk + off(qo), dMm + off(ks * 2048), id_o, ks != 0);
        }
        mma_commit(mma_done);
    }
    ok = ok && block_wait(mma_done, phase++ & 1, abort_flag, p.status);
    tc_fence_after();
    // ---- P = S' masked (bf16), D_t = phi(q_t).z + row sum + eps: token rows (warps 0, 1)
    if (ok && warp < 2) {
        const int t = tid;
        const uint32_t srow = tmem + L::TS + ((uint32_t)(32 * warp) << 16);
        uint8_t* prow = sm + L::PT + t * 128;
        float rs = 0.f;
#pragma unroll
        for (int k0 = 0; k0 < 64; k0 += 16) {
            float x[16];
            ld16f(srow + k0, x);
            uint32_t ph[8], pl[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float s0 = (k0 + 2 * e <= t) ? x[2 * e] : 0.f;
                const float s1 = (k0 + 2 * e + 1 <= t) ? x[2 * e + 1] : 0.f;
                split2(s0, s1, ph[e], pl[e]);
                rs += s0 + s1;
            }
            const int ch = k0 >> 3;  // 16-byte chunks ch, ch + 1 of the row
            const uint32_t c0 = (ch ^ (t & 7)) << 4, c1 = ((ch + 1) ^ (t & 7)) << 4;
            *reinterpret_cast<uint4*>(prow + c0) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
            *reinterpret_cast<uint4*>(prow + c1) = make_uint4(ph[4], ph[5], ph[6], ph[7]);
            *reinterpret_cast<uint4*>(prow + ATOM + c0) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
            *reinterpret_cast<uint4*>(prow + ATOM + c1) = make_uint4(pl[4], pl[5], pl[6], pl[7]);
        }
        const float zq = __uint_as_float(tmem_ld1(srow + 64));
        tmem_wait_ld();
        den[t] = zq + rs + p.eps;
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- O += P V
    if (ok && tid == 0) {
        constexpr uint32_t id_pv = idesc_bf16(128, DV, 0, 1);
#pragma unroll
        for (int ks = 0; ks < CH / 16; ++ks) {
            mma_bf16_ss(tmem + L::TO, dPk + off(ks * 32), dVm + off(ks * 2048), id_pv, 1);
            mma_bf16_ss(tmem + L::TO, dPk + off(ATOM + ks * 32), dVm + off(ks * 2048), id_pv, 1);
        }
        mma_commit(mma_done);
    }
    ok = ok && block_wait(mma_done, phase++ & 1, abort_flag, p.status);
    tc_fence_after();
    // ---- g = dout / D, e = -(g . out): token rows; G as bf16 tile and to the workspace
    if (ok && warp < 2) {
        const int t = tid;
        const uint32_t orow = tmem + L::TO + ((uint32_t)(32 * warp) << 16);
        const float rd = t < valid ? 1.f / den[t] : 0.f;  // rows past the end: g = e = 0
        float dot = 0.f;
        // workspace: the high parts of G as [B*H][T][dv] bf16, the low parts right after them
        __nv_bfloat16* gout = reinterpret_cast<__nv_bfloat16*>(p.G) + ((int64_t)bh * p.T + t0 + t) * DV;
        const int64_t glo = (int64_t)p.B * p.H * p.T * DV;
#pragma unroll 1
        for (int j0 = 0; j0 < DV; j0 += 16) {
            float o[16];
            ld16f(orow + j0, o);
            uint32_t gh[8], gl[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t dw = *reinterpret_cast<const uint32_t*>(sm + L::OT + tile_off(t, j0 + 2 * e, ATOM));
                const float g0 = bf16lo(dw) * rd, g1 = bf16hi(dw) * rd;
                dot += g0 * o[2 * e] + g1 * o[2 * e + 1];
                split2(g0, g1, gh[e], gl[e]);
            }
            uint8_t* grow = sm + L::GT + (j0 >> 6) * ATOM + t * 128;
            const int ch = (j0 & 63) >> 3;
            const uint32_t c0 = (ch ^ (t & 7)) << 4, c1 = ((ch + 1) ^ (t & 7)) << 4;
            const uint4 h0 = make_uint4(gh[0], gh[1], gh[2], gh[3]), h1 = make_uint4(gh[4], gh[5], gh[6], gh[7]);
            const uint4 l0 = make_uint4(gl[0], gl[1], gl[2], gl[3]), l1 = make_uint4(gl[4], gl[5], gl[6], gl[7]);
            *reinterpret_cast<uint4*>(grow + c0) = h0;
            *reinterpret_cast<uint4*>(grow + c1) = h1;
            *reinterpret_cast<uint4*>(grow + (DV / 64) * ATOM + c0) = l0;
            *reinterpret_cast<uint4*>(grow + (DV / 64) * ATOM + c1) = l1;
            if (t < valid) {
                *reinterpret_cast<uint4*>(gout + j0) = h0;
                *reinterpret_cast<uint4*>(gout + j0 + 8) = h1;
                *reinterpret_cast<uint4*>(gout + glo + j0) = l0;
                *reinterpret_cast<uint4*>(gout + glo + j0 + 8) = l1;
            }
        }
        const float e = -dot * rd;  // g . out = (g . O) / D
        ev[t] = e;
        if (t < valid) p.E[(int64_t)bh * p.T + t0 + t] = e;
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- dA = G V^T, dphi(Q) = G M^T, phi(Q)^T G
    if (ok && tid == 0) {
        constexpr uint32_t id_a = idesc_bf16(128, CH, 0, 0);
        constexpr uint32_t id_q = idesc_bf16(128, D, 0, 0);
        constexpr uint32_t id_r = idesc_bf16(128, DV, 1, 1);
        constexpr uint32_t GLO = (DV / 64) * ATOM;  // offset of the low parts of G
#pragma unroll
        for (int ks = 0; ks < DV / 16; ++ks) {
            const uint32_t go = (ks >> 2) * ATOM + (ks & 3) * 32;
            const uint64_t mo = off((ks >> 2) * (D * 128) + (ks & 3) * 32);
            mma_bf16_ss(tmem + L::TS, dGk + off(go), dVk + off(go), id_a, ks != 0);
            mma_bf16_ss(tmem + L::TS, dGk + off(GLO + go), dVk + off(go), id_a, 1);
            mma_bf16_ss(tmem + L::TO, dGk + off(go), dMk + mo, id_q, ks != 0);
            mma_bf16_ss(tmem + L::TO, dGk + off(GLO + go), dMk + mo, id_q, 1);
        }
#pragma unroll
        for (int ks = 0; ks < CH / 16; ++ks) {
            mma_bf16_ss(tmem + L::TR, dQm + off(ks * 2048), dGm + off(ks * 2048), id_r, ks != 0);
            mma_bf16_ss(tmem + L::TR, dQm + off(ks * 2048), dGm + off(GLO + ks * 2048), id_r, 1);
        }
        mma_commit(mma_done);
    }
    ok = ok && block_wait(mma_done, phase++ & 1, abort_flag, p.status);
    tc_fence_after();
    // ---- dA + e, masked to keys at or before the query, as bf16: token rows
    if (ok && warp < 2) {
        const int t = tid;
        const uint32_t arow = tmem + L::TS + ((uint32_t)(32 * warp) << 16);
        const float e = ev[t];
        uint8_t* row = sm + L::AT + t * 128;
#pragma unroll
        for (int k0 = 0; k0 < 64; k0 += 16) {
            float x[16];
            ld16f(arow + k0, x);
            uint32_t ah[8], al[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float a0 = (k0 + 2 * q <= t) ? x[2 * q] + e : 0.f;
                const float a1 = (k0 + 2 * q + 1 <= t) ? x[2 * q + 1] + e : 0.f;
                split2(a0, a1, ah[q], al[q]);
            }
            const int ch = k0 >> 3;
            const uint32_t c0 = (ch ^ (t & 7)) << 4, c1 = ((ch + 1) ^ (t & 7)) << 4;
            *reinterpret_cast<uint4*>(row + c0) = make_uint4(ah[0], ah[1], ah[2], ah[3]);
            *reinterpret_cast<uint4*>(row + c1) = make_uint4(ah[4], ah[5], ah[6], ah[7]);
            *reinterpret_cast<uint4*>(row + ATOM + c0) = make_uint4(al[0], al[1], al[2], al[3]);
            *reinterpret_cast<uint4*>(row + ATOM + c1) = make_uint4(al[4], al[5], al[6], al[7]);
        }
        fence_proxy_async_smem();
    }
    // ---- the chunk's state-gradient record: phi(Q)^T G (lanes = features) and phi(Q)^T e
    if (ok) {
        float* rrec = p.rev + ((int64_t)bh * p.nch + c) * p.rec;
        const int q4 = warp & 3, half = warp >> 2;  // lane quarter; columns [half*DV/2, +DV/2)
        const int i = 32 * q4 + lane;
        if (32 * q4 < D) {
            const uint32_t rrow = tmem + L::TR + ((uint32_t)(32 * q4) << 16);
#pragma unroll 1
            for (int j0 = half * (DV / 2); j0 < (half + 1) * (DV / 2); j0 += 16) {
                float x[16];
                ld16f(rrow + j0, x);
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                    *reinterpret_cast<float4*>(rrec + (int64_t)i * DV + j0 + e) =
                        make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
            }
        }
        if (tid < D) {
            float s = 0.f;
            for (int t = 0; t < CH; ++t) s += tile_get(sm + L::QT, t, tid, ATOM) * ev[t];
            rrec[D * DV + tid] = s;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- dphi(Q) += dA phi(K)
    if (ok && tid == 0) {
        constexpr uint32_t id_q = idesc_bf16(128, D, 0, 1);
#pragma unroll
        for (int ks = 0; ks < CH / 16; ++ks) {
            mma_bf16_ss(tmem + L::TO, dAk + off(ks * 32), dKm + off(ks * 2048), id_q, 1);
            mma_bf16_ss(tmem + L::TO, dAk + off(ATOM + ks * 32), dKm + off(ks * 2048), id_q, 1);
        }
        mma_commit(mma_done);
    }
    ok = ok && block_wait(mma_done, phase++ & 1, abort_flag, p.status);
    tc_fence_after();
    // ---- dq = (dphi(Q) + e z) phi'(q): token rows (the TMEM loads are warp-wide; only rows
    // inside the sequence are stored)
    if (ok && warp < 2) {
        const int t = tid;
        const bool store = t < valid;
        const uint32_t qrow = tmem + L::TO + ((uint32_t)(32 * warp) << 16);
        const float e = ev[t];
        __nv_bfloat16* dq = reinterpret_cast<__nv_bfloat16*>(p.dq) + ((int64_t)bh * p.T + t0 + t) * D;
#pragma unroll 1
        for (int i0 = 0; i0 < D; i0 += 16) {
            float x[16];
            ld16f(qrow + i0, x);
            uint32_t w[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint32_t fw = *reinterpret_cast<const uint32_t*>(sm + L::QT + tile_off(t, i0 + 2 * q, ATOM));
                const float d0 = (x[2 * q] + e * zf[i0 + 2 * q]) * fminf(bf16lo(fw), 1.f);
                const float d1 = (x[2 * q + 1] + e * zf[i0 + 2 * q + 1]) * fminf(bf16hi(fw), 1.f);
                w[q] = pack_bf16(d0, d1);
            }
            if (store) {
                *reinterpret_cast<uint4*>(dq + i0) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(dq + i0 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, L::NCOL);
    }
}

// ================================================================================ dk, dv
template <int D, int DV>
struct DkvLayout {
    static constexpr int QT = 0;                          // phi(Q), D/64 atoms
    static constexpr int KT = QT + D / 64 * ATOM;         // phi(K), D/64 atoms (+ read past: VT)
    static constexpr int VT = KT + D / 64 * ATOM;         // V, DV/64 atoms (+ read past: GT)
    static constexpr int GT = VT + DV / 64 * ATOM;        // G high (DV/64 atoms), then low part
    static constexpr int PT = GT + 2 * (DV / 64) * ATOM;  // P^T [64 keys][64 queries] high, then low
    static constexpr int AT = PT + 2 * ATOM;              // dA^T high, then low
    static constexpr int RT = AT + 2 * ATOM;              // R (bf16), DV/64 blocks of D*128 bytes
    static constexpr int EV = RT + D * DV * 2;            // 64 floats: e_t
    static constexpr int RV = EV + 256;                   // D floats: r
    static constexpr int BAR = RV + 512;
    static constexpr int MISC = BAR + 16;
    static constexpr int ALLOC = MISC + 16 + 1024;
    static constexpr uint32_t TS = 0;                     // S^T (64)
    static constexpr uint32_t TA = 64;                    // dA^T (64)
    static constexpr uint32_t TV = 128;                   // dv (DV)
    static constexpr uint32_t TK = TV + DV;               // dphi(K) (D)
    static constexpr uint32_t NCOL = TK + D <= 256 ? 256 : 512;
};

template <int D, int DV>
__global__ void __launch_bounds__(BT, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mk,
                       const __grid_constant__ CUtensorMap mv, const __grid_constant__ CUtensorMap mg,
                       const __grid_constant__ CUtensorMap mgl, BwdTcParams p) {
    using L = DkvLayout<D, DV>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint64_t* ld_full = bars + 0;
    uint64_t* mma_done = bars + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
    float* ev = reinterpret_cast<float*>(sm + L::EV);
    float* rv = reinterpret_cast<float*>(sm + L::RV);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int c = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H;
    const int64_t t0 = (int64_t)c * CH;
    const int valid = (int)min64(CH, p.T - t0);
    const float* rrec = p.rev + ((int64_t)bh * p.nch + c) * p.rec;

    if (tid == 0) {
        mbar_init(ld_full, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mq);
        tma_prefetch_desc(&mk);
        tma_prefetch_desc(&mv);
        tma_prefetch_desc(&mg);
        tma_prefetch_desc(&mgl);
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, L::NCOL);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (tid == 0) {
        const uint64_t pol = l2_evict_first_policy();
        mbar_expect_tx(ld_full, (2 * D + 3 * DV) * CH * 2);
        for (int a = 0; a < D / 64; ++a) {
            tma_load_4d_hint(sm + L::QT + a * ATOM, &mq, ld_full, a * 64, (int)t0, h, b, pol);
            tma_load_4d_hint(sm + L::KT + a * ATOM, &mk, ld_full, a * 64, (int)t0, h, b, pol);
        }
        for (int a = 0; a < DV / 64; ++a) {
            tma_load_4d_hint(sm + L::VT + a * ATOM, &mv, ld_full, a * 64, (int)t0, h, b, pol);
            tma_load_4d_hint(sm + L::GT + a * ATOM, &mg, ld_full, a * 64, (int)t0, h, b, pol);
            tma_load_4d_hint(sm + L::GT + (DV / 64 + a) * ATOM, &mgl, ld_full, a * 64, (int)t0, h, b, pol);
        }
    }
    state_to_tile<D, DV>(rrec, sm + L::RT, tid);
    if (tid < D) rv[tid] = rrec[D * DV + tid];
    if (tid < CH) ev[tid] = tid < valid ? p.E[(int64_t)bh * p.T + t0 + tid] : 0.f;
    bool ok = block_wait(ld_full, 0, abort_flag, p.status);
    if (ok) {
        phi_tile<D, BT>(sm + L::QT, ATOM, valid, tid, nullptr);
        phi_tile<D, BT>(sm + L::KT, ATOM, valid, tid, nullptr);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    auto off = [](uint32_t bytes) { return (uint64_t)(bytes >> 4); };
    const uint64_t dQk = sdesc_sw128(smem_u32(sm + L::QT), 16, 1024);      // phi(Q), K-major (K = d)
    const uint64_t dQm = sdesc_sw128(smem_u32(sm + L::QT), ATOM, 1024);    // phi(Q), MN-major (K = queries)
    const uint64_t dKk = sdesc_sw128(smem_u32(sm + L::KT), 16, 1024);      // phi(K), K-major (K = d)
    const uint64_t dVk = sdesc_sw128(smem_u32(sm + L::VT), 16, 1024);      // V, K-major (K = dv)
    const uint64_t dGk = sdesc_sw128(smem_u32(sm + L::GT), 16, 1024);      // G, K-major (K = dv)
    const uint64_t dGm = sdesc_sw128(smem_u32(sm + L::GT), ATOM, 1024);    // G, MN-major (K = queries)
    const uint64_t dRm = sdesc_sw128(smem_u32(sm + L::RT), D * 128, 1024); // R, MN-major (K = d, N = dv)
    const uint64_t dRk = sdesc_sw128(smem_u32(sm + L::RT), 16, 1024);      // R, K-major (N = d, K = dv)
    const uint64_t dPk = sdesc_sw128(smem_u32(sm + L::PT), 16, 1024);
    const uint64_t dAk = sdesc_sw128(smem_u32(sm + L::AT), 16, 1024);
    uint32_t phase = 0;

    // ---- S^T = phi(K) phi(Q)^T, dA^T = V G^T (lanes = keys, columns = queries)
    if (ok && tid == 0) {
        constexpr uint32_t id_t = idesc_bf16(128, CH, 0, 0);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t o = (ks >> 2) * ATOM + (ks & 3) * 32;
            mma_bf16_ss(tmem + L::TS, dKk + off(o), dQk + off(o), id_t, ks != 0);
        }
#pragma unroll
        for (int ks = 0; ks < DV / 16; ++ks) {
            const uint32_t o = (ks >> 2) * ATOM + (ks & 3) * 32;
            mma_bf16_ss(tmem + L::TA, dVk + off(o), dGk + off(o), id_t, ks != 0);
            mma_bf16_ss(tmem + L::TA, dVk + off(o), dGk + off((DV / 64) * ATOM + o), id_t, 1);
        }
        mma_commit(mma_done);
    }
    ok = ok && block_wait(mma_done, phase++ & 1, abort_flag, p.status);
    tc_fence_after();
    // ---- P^T and dA^T + e, masked to queries at or after the key (bf16): key rows
    if (ok && warp < 2) {
        const int j = threadIdx.x;
        const uint32_t lb = (uint32_t)(32 * warp) << 16;
        uint8_t* prow = sm + L::PT + j * 128;
        uint8_t* arow = sm + L::AT + j * 128;
#pragma unroll 1
        for (int k0 = 0; k0 < 64; k0 += 16) {
            float s[16], a[16];
            ld16f(tmem + L::TS + lb + k0, s);
            ld16f(tmem + L::TA + lb + k0, a);
            uint32_t ph[8], pl[8], ah[8], al[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int tq = k0 + 2 * q;
                const bool m0 = tq >= j, m1 = tq + 1 >= j;
                split2(m0 ? s[2 * q] : 0.f, m1 ? s[2 * q + 1] : 0.f, ph[q], pl[q]);
                split2(m0 ? a[2 * q] + ev[tq] : 0.f, m1 ? a[2 * q + 1] + ev[tq + 1] : 0.f, ah[q], al[q]);
            }
            const int ch = k0 >> 3;
            const uint32_t c0 = (ch ^ (j & 7)) << 4, c1 = ((ch + 1) ^ (j & 7)) << 4;
            *reinterpret_cast<uint4*>(prow + c0) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
            *reinterpret_cast<uint4*>(prow + c1) = make_uint4(ph[4], ph[5], ph[6], ph[7]);
            *reinterpret_cast<uint4*>(prow + ATOM + c0) = make_uint4(pl[0], pl[1], pl[2], pl[3]);
            *reinterpret_cast<uint4*>(prow + ATOM + c1) = make_uint4(pl[4], pl[5], pl[6], pl[7]);
            *reinterpret_cast<uint4*>(arow + c0) = make_uint4(ah[0], ah[1], ah[2], ah[3]);
            *reinterpret_cast<uint4*>(arow + c1) = make_uint4(ah[4], ah[5], ah[6], ah[7]);
            *reinterpret_cast<uint4*>(arow + ATOM + c0) = make_uint4(al[0], al[1], al[2], al[3]);
            *reinterpret_cast<uint4*>(arow + ATOM + c1) = make_uint4(al[4], al[5], al[6], al[7]);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- dv = P^T G + phi(K) R,  dphi(K) = dA^T phi(Q) + V R^T
    if (ok && tid == 0) {
        constexpr uint32_t id_vg = idesc_bf16(128, DV, 0, 1);
        constexpr uint32_t id_kq = idesc_bf16(128, D, 0, 1);
        constexpr uint32_t id_kr = idesc_bf16(128, D, 0, 0);
        constexpr uint32_t GLO = (DV / 64) * ATOM;
#pragma unroll
        for (int ks = 0; ks < CH / 16; ++ks) {
            // P^T G with both split: hi.hi + lo.hi + hi.lo
            mma_bf16_ss(tmem + L::TV, dPk + off(ks * 32), dGm + off(ks * 2048), id_vg, ks != 0);
            mma_bf16_ss(tmem + L::TV, dPk + off(ATOM + ks * 32), dGm + off(ks * 2048), id_vg, 1);
            mma_bf16_ss(tmem + L::TV, dPk + off(ks * 32), dGm + off(GLO + ks * 2048), id_vg, 1);
            mma_bf16_ss(tmem + L::TK, dAk + off(ks * 32), dQm + off(ks * 2048), id_kq, ks != 0);
            mma_bf16_ss(tmem + L::TK, dAk + off(ATOM + ks * 32), dQm + off(ks * 2048), id_kq, 1);
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
            mma_bf16_ss(tmem + L::TV, dKk + off((ks >> 2) * ATOM + (ks & 3) * 32), dRm + off(ks * 2048), id_vg, 1);
#pragma unroll
        for (int ks = 0; ks < DV / 16; ++ks)
            mma_bf16_ss(tmem + L::TK, dVk + off((ks >> 2) * ATOM + (ks & 3) * 32),
                        dRk + off((ks >> 2) * (D * 128) + (ks & 3) * 32), id_kr, 1);
        mma_commit(mma_done);
    }
    ok = ok && block_wait(mma_done, phase++ & 1, abort_flag, p.status);
    tc_fence_after();
    // ---- dk = (dphi(K) + r) phi'(k), dv: key rows; warps 0-1 take dk, warps 4-5 dv
    if (ok && (warp & 3) < 2) {
        const int j = 32 * (warp & 3) + (threadIdx.x & 31);
        const uint32_t lb = (uint32_t)(32 * (warp & 3)) << 16;
        const bool store = j < valid;  // the TMEM loads are warp-wide; only key rows inside the sequence are stored
        {
            if (warp < 4) {
                __nv_bfloat16* dk = reinterpret_cast<__nv_bfloat16*>(p.dk) + ((int64_t)bh * p.T + t0 + j) * D;
#pragma unroll 1
                for (int i0 = 0; i0 < D; i0 += 16) {
                    float x[16];
                    ld16f(tmem + L::TK + lb + i0, x);
                    uint32_t w[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint32_t fw =
                            *reinterpret_cast<const uint32_t*>(sm + L::KT + tile_off(j, i0 + 2 * q, ATOM));
                        w[q] = pack_bf16((x[2 * q] + rv[i0 + 2 * q]) * fminf(bf16lo(fw), 1.f),
                                         (x[2 * q + 1] + rv[i0 + 2 * q + 1]) * fminf(bf16hi(fw), 1.f));
                    }
                    if (store) {
                        *reinterpret_cast<uint4*>(dk + i0) = make_uint4(w[0], w[1], w[2], w[3]);
                        *reinterpret_cast<uint4*>(dk + i0 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            } else {
                __nv_bfloat16* dvp = reinterpret_cast<__nv_bfloat16*>(p.dv) + ((int64_t)bh * p.T + t0 + j) * DV;
#pragma unroll 1
                for (int j0 = 0; j0 < DV; j0 += 16) {
                    float x[16];
                    ld16f(tmem + L::TV + lb + j0, x);
                    uint32_t w[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) w[q] = pack_bf16(x[2 * q], x[2 * q + 1]);
                    if (store) {
                        *reinterpret_cast<uint4*>(dvp + j0) = make_uint4(w[0], w[1], w[2], w[3]);
                        *reinterpret_cast<uint4*>(dvp + j0 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, L::NCOL);
    }
}

// ================================================================================ launchers
template <int D, int DV>
static cudaError_t launch_dq_t(const BwdTcParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                               const CUtensorMap& mv, const CUtensorMap& mdo, cudaStream_t s) {
    using L = DqLayout<D, DV>;
    static_assert(L::ALLOC <= 227 * 1024, "shared memory budget");
    auto fn = bwd_dq_tc_kernel<D, DV>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    fn<<<dim3(p.nch, p.B * p.H), BT, L::ALLOC, s>>>(mq, mk, mv, mdo, p);
    return cudaGetLastError();
}

template <int D, int DV>
static cudaError_t launch_dkdv_t(const BwdTcParams& p, const CUtensorMap& mq, const CUtensorMap& mk,
                                 const CUtensorMap& mv, const CUtensorMap& mg, const CUtensorMap& mgl,
                                 cudaStream_t s) {
    using L = DkvLayout<D, DV>;
    static_assert(L::ALLOC <= 227 * 1024, "shared memory budget");
    auto fn = bwd_dkdv_tc_kernel<D, DV>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    fn<<<dim3(p.nch, p.B * p.H), BT, L::ALLOC, s>>>(mq, mk, mv, mg, mgl, p);
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
                               const CUtensorMap& mv, const CUtensorMap& mg, const CUtensorMap& mgl,
                               cudaStream_t s) {
    if (p.d == 128 && p.dv_dim == 128) return launch_dkdv_t<128, 128>(p, mq, mk, mv, mg, mgl, s);
    if (p.d == 128 && p.dv_dim == 64) return launch_dkdv_t<128, 64>(p, mq, mk, mv, mg, mgl, s);
    if (p.d == 64 && p.dv_dim == 128) return launch_dkdv_t<64, 128>(p, mq, mk, mv, mg, mgl, s);
    if (p.d == 64 && p.dv_dim == 64) return launch_dkdv_t<64, 64>(p, mq, mk, mv, mg, mgl, s);
    return cudaErrorInvalidValue;
}

}  // namespace la
