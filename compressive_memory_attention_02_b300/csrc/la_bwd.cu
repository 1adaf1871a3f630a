// Training backward of causal linear attention, float32 arithmetic (SIMT).
//
// The page "Attention_Kernel_Mask" names a training-backward mode (table "Causal
// Attention Training and Inferencing") but prints no formula. This is the chain rule on
// the chunk form of that page's "chunk sequential mode" (mode 3). For chunk c, with the
// state (M_{c-1}, z_{c-1}) of every token before it and S = phi(Q_c) phi(K_c)^T kept
// for keys at or before the query:
//   D_t   = phi(q_t) . z_{c-1} + sum_j S_tj + eps
//   out_t = (phi(q_t)^T M_{c-1} + sum_j S_tj v_j) / D_t
//   g_t = dout_t / D_t,   e_t = -(g_t . out_t),   dA_tj = g_t . v_j + e_t   (j <= t)
//   dphi(q_t) = M_{c-1} g_t + e_t z_{c-1} + sum_j dA_tj phi(k_j)
//   R_c = dM_out + sum over chunks c' > c of phi(Q_c')^T G_c'   (r_c the same with e)
//   dphi(k_j) = sum_{t >= j} dA_tj phi(q_t) + R_c v_j + r_c
//   dv_j      = sum_{t >= j} S_tj g_t + R_c^T phi(k_j)
//   dM_in = dM_out + sum over all chunks of phi(Q_c)^T G_c   (dz_in the same with e)
// and dx = dphi(x) phi'(x), where phi'(x) = min(phi(x), 1): 1 for x > 0, exp(x) otherwise.
//
// Launches (la_api.cu): 64-token key-value sums (bwd_sums) -> exclusive prefix scan
// (the state before each chunk) -> bwd_dq (dq, G, E and the chunk sums phi(Q)^T G,
// phi(Q)^T e) -> exclusive reverse scan (R_c; the totals are dM_in, dz_in) -> bwd_dk ->
// bwd_dv. A chunk kernel runs one block of 256 threads per (chunk, b*H + h) with every
// operand of the chunk in shared memory (tile rows padded by one float so that strided
// reads by consecutive threads fall in distinct banks); its products run through Tile,
// a register-tiled micro-kernel.
#include <type_traits>

#include "la_bwd.h"

namespace la {
namespace {

template <typename T>
__device__ __forceinline__ float bld(const T* p);
template <>
__device__ __forceinline__ float bld<float>(const float* p) {
    return *p;
}
template <>
__device__ __forceinline__ float bld<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}
template <typename T>
__device__ __forceinline__ void bst(T* p, float x);
template <>
__device__ __forceinline__ void bst<float>(float* p, float x) {
    *p = x;
}
template <>
__device__ __forceinline__ void bst<__nv_bfloat16>(__nv_bfloat16* p, float x) {
    *p = __float2bfloat16_rn(x);
}

constexpr int NT = 256;
constexpr int C = BWD_CH;
constexpr int LDS = C + 1;  // row stride of the C x C score tiles

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// 16 bytes of storage elements -> floats (8 for bf16, 4 for float32).
__device__ __forceinline__ void unpack16(const uint4& u, float* x, const __nv_bfloat16*) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = __uint_as_float(w[e] << 16);
        x[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
    }
}
__device__ __forceinline__ void unpack16(const uint4& u, float* x, const float*) {
    x[0] = __uint_as_float(u.x), x[1] = __uint_as_float(u.y), x[2] = __uint_as_float(u.z), x[3] = __uint_as_float(u.w);
}

// Rows 0..C-1 of a contiguous [rows, n] slice (16-byte aligned, n a multiple of 8) into a
// tile with row stride ld, phi applied when asked; rows >= nv become 0. Every thread
// issues all of its 16-byte loads (at most 8) before it uses any of them.
template <typename TI>
__device__ void load_rows(float* dst, int ld, const TI* src, int n, int nv, bool apply_phi) {
    constexpr int VE = 16 / (int)sizeof(TI);
    const int vpr = n / VE, nvec = C * vpr;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4 buf[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int idx = (int)threadIdx.x + u * NT;
        buf[u] = make_uint4(0u, 0u, 0u, 0u);
        if (idx < nvec && idx / vpr < nv) buf[u] = __ldg(s4 + idx);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int idx = (int)threadIdx.x + u * NT;
        if (idx >= nvec) break;
        const int t = idx / vpr, c0 = (idx - t * vpr) * VE;
        float x[8];
        unpack16(buf[u], x, src);
        const bool f = apply_phi && t < nv;
#pragma unroll
        for (int e = 0; e < VE; ++e) dst[t * ld + c0 + e] = f ? phi_f(x[e]) : x[e];
    }
}

// A state record (M row-major d x dv, then z; 16-byte aligned) into Ms (row stride ld) and zs.
__device__ void load_record(float* Ms, int ld, float* zs, const float* rec, int d, int dv) {
    const int nvec = d * dv / 4, vpr = dv / 4;
    const float4* s4 = reinterpret_cast<const float4*>(rec);
    for (int base = 0; base < nvec; base += 8 * NT) {
        float4 buf[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = base + (int)threadIdx.x + u * NT;
            if (idx < nvec) buf[u] = __ldg(s4 + idx);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = base + (int)threadIdx.x + u * NT;
            if (idx >= nvec) break;
            const int i = idx / vpr, j = (idx - i * vpr) * 4;
            float* m = Ms + i * ld + j;
            m[0] = buf[u].x, m[1] = buf[u].y, m[2] = buf[u].z, m[3] = buf[u].w;
        }
    }
    for (int i = threadIdx.x; i < d; i += NT) zs[i] = rec[(int64_t)d * dv + i];
}

// Register-tiled product over shared-memory operands: out(r, n) += sum_k A(r, k) B(k, n)
// with A(r, k) = A[r*ars + k*aks] and B(k, n) = B[k*bks + n*bns]. Thread (rg, cg) =
// (tid / 16, tid % 16) owns rows r0 + rg + 16i (i < 4; with BLK the four consecutive rows
// r0 + 4rg + i) and columns cg + 16j (j < 8, while below N): per k it loads 4 + (up to) 8
// operands for up to 32 multiply-adds. With FX
// (d and dv fixed at compile time, multiples of 64) every stride, N and K is a constant, so
// the k loop unrolls into loads at constant offsets; otherwise rows past R read row R-1
// (in bounds) and are not stored.
template <bool FX, bool BLK = false>
struct Tile {
    float acc[4][8];
    int rg, cg, nb;
    // row i of this thread (before r0): rows rg + 16i, or with BLK the four rows 4rg .. 4rg+3
    __device__ __forceinline__ int row(int i) const { return BLK ? 4 * rg + i : rg + 16 * i; }
    __device__ __forceinline__ explicit Tile(int N) : rg((int)threadIdx.x >> 4), cg((int)threadIdx.x & 15) {
        nb = FX ? (N >> 4) : ((N - cg + 15) >> 4);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    }
    __device__ __forceinline__ void add(const float* A, int ars, int aks, const float* B, int bks, int bns, int K,
                                        int r0, int R) {
        int ro[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ro[i] = (FX ? r0 + row(i) : min(r0 + row(i), R - 1)) * ars;
        const float* pb = B + cg * bns;
        constexpr int UNROLL = FX ? 4 : 1;  // runtime strides: keep the loop compact
#pragma unroll UNROLL
        for (int k = 0; k < K; ++k) {
            float a[4], b[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = A[ro[i] + k * aks];
#pragma unroll
            for (int j = 0; j < 8; ++j) b[j] = (j < nb) ? pb[k * bks + 16 * j * bns] : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < nb) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    // The same product over k in [kb, ke) only, for a C-row product (r0 = 0, R = C): with BLK,
    // a causal mask bounds k per thread (keys up to the thread's last row, or queries from
    // its first row on) and the masked terms are skipped instead of multiplied by zero.
    __device__ __forceinline__ void add_range(const float* A, int ars, int aks, const float* B, int bks, int bns,
                                              int kb, int ke) {
        int ro[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ro[i] = row(i) * ars;
        const float* pb = B + cg * bns;
        constexpr int UNROLL = FX ? 4 : 1;
#pragma unroll UNROLL
        for (int k = kb; k < ke; ++k) {
            float a[4], b[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = A[ro[i] + k * aks];
#pragma unroll
            for (int j = 0; j < 8; ++j) b[j] = (j < nb) ? pb[k * bks + 16 * j * bns] : 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < nb) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
    }
    // f(row, col, value) for every owned element with row < R
    template <class F>
    __device__ __forceinline__ void store(int r0, int R, F f) const {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = r0 + row(i);
            if (r >= R) continue;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < nb) f(r, cg + 16 * j, acc[i][j]);
        }
    }
};

// S_tj = phi(q_t) . phi(k_j) for j <= t, else 0 (the C x C product, then the mask).
template <bool FX>
__device__ __forceinline__ void scores(float* Ss, const float* Qf, const float* Kf, int ldq, int d) {
    Tile<FX> tl(C);
    tl.add(Qf, ldq, 1, Kf, 1, ldq, d, 0, C);
    tl.store(0, C, [&](int t, int j, float x) { Ss[t * LDS + j] = (j <= t) ? x : 0.f; });
}

// dA_tj = g_t . v_j + e_t for j <= t, else 0.
template <bool FX>
__device__ __forceinline__ void score_grads(float* dA, const float* Gs, const float* Vs, const float* ee, int ldv,
                                            int dv) {
    Tile<FX> tl(C);
    tl.add(Gs, ldv, 1, Vs, 1, ldv, dv, 0, C);
    tl.store(0, C, [&](int t, int j, float x) { dA[t * LDS + j] = (j <= t) ? x + ee[t] : 0.f; });
}

// ------------------------------------------------------------------ 64-token key-value sums
// Record (bh, c) = [sum_t phi(k_t) v_t^T (d x dv row-major) | sum_t phi(k_t)] over the chunk.
// Shared memory (float): Kf [C][d+1], Vs [C][dv+1].
template <typename TI, int DT, int DVT>
__global__ void __launch_bounds__(NT) bwd_sums_kernel(BwdParams p) {
    extern __shared__ float sm[];
    constexpr bool FX = DT > 0;  // d, dv fixed at compile time
    const int d = FX ? DT : p.d, dv = FX ? DVT : p.dv_dim;
    const int ldq = d + 1, ldv = dv + 1;
    const int c = blockIdx.x, bh = blockIdx.y;
    const int64_t t0 = (int64_t)c * C;
    const int nv = (int)min64(C, p.T - t0);
    float* Kf = sm;
    float* Vs = Kf + C * ldq;
    const int64_t row0 = (int64_t)bh * p.T + t0;
    load_rows(Kf, ldq, static_cast<const TI*>(p.k) + row0 * d, d, nv, true);
    load_rows(Vs, ldv, static_cast<const TI*>(p.v) + row0 * dv, dv, nv, false);
    __syncthreads();
    float* rec = p.states + ((int64_t)bh * p.nch + c) * p.rec;
    for (int r0 = 0; r0 < d; r0 += 64) {
        Tile<FX> tl(dv);
        tl.add(Kf, 1, ldq, Vs, ldv, 1, FX ? C : nv, r0, d);
        tl.store(r0, d, [&](int i, int n, float x) { rec[i * dv + n] = x; });
    }
    for (int i = threadIdx.x; i < d; i += NT) {
        float acc = 0.f;
        for (int t = 0; t < nv; ++t) acc += Kf[t * ldq + i];
        rec[(int64_t)d * dv + i] = acc;
    }
}

// ------------------------------------------------------------------ dq, G, E, chunk sums
// Shared memory (float): Qf, Kf [C][d+1]; Vs, Os [C][dv+1]; Ms [d][dv+1]; Ss [C][C+1];
// zs [d]; den, ee [C]. Os holds out, then g.
template <typename TI, int DT, int DVT>
__global__ void __launch_bounds__(NT) bwd_dq_kernel(BwdParams p) {
    extern __shared__ float sm[];
    constexpr bool FX = DT > 0;  // d, dv fixed at compile time
    const int d = FX ? DT : p.d, dv = FX ? DVT : p.dv_dim;
    const int ldq = d + 1, ldv = dv + 1;
    const int c = blockIdx.x, bh = blockIdx.y;
    const int64_t t0 = (int64_t)c * C;
    const int nv = (int)min64(C, p.T - t0);
    float* Qf = sm;
    float* Kf = Qf + C * ldq;
    float* Vs = Kf + C * ldq;
    float* Os = Vs + C * ldv;
    float* Ms = Os + C * ldv;
    float* Ss = Ms + d * ldv;
    float* zs = Ss + C * LDS;
    float* den = zs + d;
    float* ee = den + C;
    const int64_t row0 = (int64_t)bh * p.T + t0;
    const TI* dout = static_cast<const TI*>(p.dout) + row0 * dv;
    TI* dq = static_cast<TI*>(p.dq) + row0 * d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // dout rows warp + 8r, columns lane + 32m of this thread's g/e pass, requested first
    float dreg[C / 8][4];
#pragma unroll
    for (int r = 0; r < C / 8; ++r)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int t = warp + 8 * r, n = lane + 32 * m;
            dreg[r][m] = (t < nv && n < dv) ? bld(dout + (int64_t)t * dv + n) : 0.f;
        }

    load_rows(Qf, ldq, static_cast<const TI*>(p.q) + row0 * d, d, nv, true);
    load_rows(Kf, ldq, static_cast<const TI*>(p.k) + row0 * d, d, nv, true);
    load_rows(Vs, ldv, static_cast<const TI*>(p.v) + row0 * dv, dv, nv, false);
    load_record(Ms, ldv, zs, p.states + ((int64_t)bh * p.nch + c) * p.rec, d, dv);
    __syncthreads();
    scores<FX>(Ss, Qf, Kf, ldq, d);
    __syncthreads();
    for (int t = warp; t < C; t += NT / 32) {  // D_t
        float s = 0.f;
        for (int i = lane; i < d; i += 32) s = fmaf(Qf[t * ldq + i], zs[i], s);
        for (int j = lane; j <= t; j += 32) s += Ss[t * LDS + j];
        s = warp_sum(s);
        if (lane == 0) den[t] = s + p.eps;
    }
    __syncthreads();
    {  // out_t = (phi(q_t)^T M + sum_j S_tj v_j) / D_t
        Tile<FX, true> tl(dv);
        tl.add(Qf, ldq, 1, Ms, ldv, 1, d, 0, C);
        tl.add_range(Ss, LDS, 1, Vs, ldv, 1, 0, 4 * tl.rg + 4);  // keys j <= t
        tl.store(0, C, [&](int t, int n, float x) { Os[t * ldv + n] = (t < nv) ? x / den[t] : 0.f; });
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < C / 8; ++r) {  // g_t and e_t
        const int t = warp + 8 * r;
        float s = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int n = lane + 32 * m;
            if (n >= dv) break;
            const float g = (t < nv) ? dreg[r][m] / den[t] : 0.f;
            s = fmaf(g, Os[t * ldv + n], s);
            Os[t * ldv + n] = g;
            if (t < nv) p.G[(row0 + t) * dv + n] = g;
        }
        s = warp_sum(s);
        if (lane == 0) {
            ee[t] = -s;
            if (t < nv) p.E[row0 + t] = -s;
        }
    }
    __syncthreads();
    score_grads<FX>(Ss, Os, Vs, ee, ldv, dv);
    __syncthreads();
    {  // dq_t = (M g_t + e_t z + sum_j dA_tj phi(k_j)) phi'(q_t)
        Tile<FX, true> tl(d);
        tl.add(Os, ldv, 1, Ms, 1, ldv, dv, 0, C);
        tl.add_range(Ss, LDS, 1, Kf, ldq, 1, 0, 4 * tl.rg + 4);  // keys j <= t
        tl.store(0, nv, [&](int t, int i, float x) {
            bst(dq + (int64_t)t * d + i, (x + ee[t] * zs[i]) * fminf(Qf[t * ldq + i], 1.f));
        });
    }
    // chunk sums phi(Q)^T G and phi(Q)^T e (no barrier needed: Qf, Os, ee are unchanged)
    float* rv = p.rev + ((int64_t)bh * p.nch + c) * p.rec;
    for (int r0 = 0; r0 < d; r0 += 64) {
        Tile<FX> tl(dv);
        tl.add(Qf, 1, ldq, Os, ldv, 1, FX ? C : nv, r0, d);
        tl.store(r0, d, [&](int i, int n, float x) { rv[i * dv + n] = x; });
    }
    for (int i = threadIdx.x; i < d; i += NT) {
        float acc = 0.f;
        for (int t = 0; t < nv; ++t) acc = fmaf(Qf[t * ldq + i], ee[t], acc);
        rv[(int64_t)d * dv + i] = acc;
    }
}

// G and E rows of the chunk (rows >= nv become 0).
__device__ void load_g(float* Gs, int ldv, float* ee, const BwdParams& p, int64_t row0, int nv) {
    load_rows(Gs, ldv, p.G + row0 * p.dv_dim, p.dv_dim, nv, false);
    if (ee)
        for (int t = threadIdx.x; t < C; t += NT) ee[t] = (t < nv) ? p.E[row0 + t] : 0.f;
}

// ------------------------------------------------------------------ dk
// Shared memory (float): Qf, Kf [C][d+1]; Vs, Gs [C][dv+1]; Rs [d][dv+1]; dA [C][C+1];
// rs [d]; ee [C].
template <typename TI, int DT, int DVT>
__global__ void __launch_bounds__(NT) bwd_dk_kernel(BwdParams p) {
    extern __shared__ float sm[];
    constexpr bool FX = DT > 0;  // d, dv fixed at compile time
    const int d = FX ? DT : p.d, dv = FX ? DVT : p.dv_dim;
    const int ldq = d + 1, ldv = dv + 1;
    const int c = blockIdx.x, bh = blockIdx.y;
    const int64_t t0 = (int64_t)c * C;
    const int nv = (int)min64(C, p.T - t0);
    float* Qf = sm;
    float* Kf = Qf + C * ldq;
    float* Vs = Kf + C * ldq;
    float* Gs = Vs + C * ldv;
    float* Rs = Gs + C * ldv;
    float* dA = Rs + d * ldv;
    float* rs = dA + C * LDS;
    float* ee = rs + d;
    const int64_t row0 = (int64_t)bh * p.T + t0;
    TI* dk = static_cast<TI*>(p.dk) + row0 * d;

    load_rows(Qf, ldq, static_cast<const TI*>(p.q) + row0 * d, d, nv, true);
    load_rows(Kf, ldq, static_cast<const TI*>(p.k) + row0 * d, d, nv, true);
    load_rows(Vs, ldv, static_cast<const TI*>(p.v) + row0 * dv, dv, nv, false);
    load_g(Gs, ldv, ee, p, row0, nv);
    load_record(Rs, ldv, rs, p.rev + ((int64_t)bh * p.nch + c) * p.rec, d, dv);
    __syncthreads();
    score_grads<FX>(dA, Gs, Vs, ee, ldv, dv);
    __syncthreads();
    // dk_j = (sum_{t >= j} dA_tj phi(q_t) + R v_j + r) phi'(k_j)
    Tile<FX, true> tl(d);
    tl.add_range(dA, 1, LDS, Qf, ldq, 1, 4 * tl.rg, FX ? C : nv);  // queries t >= j
    tl.add(Vs, ldv, 1, Rs, 1, ldv, dv, 0, C);
    tl.store(0, nv, [&](int j, int i, float x) {
        bst(dk + (int64_t)j * d + i, (x + rs[i]) * fminf(Kf[j * ldq + i], 1.f));
    });
}

// ------------------------------------------------------------------ dv
// Shared memory (float): Qf, Kf [C][d+1]; Gs [C][dv+1]; Rs [d][dv+1]; Ss [C][C+1]; rs [d].
template <typename TI, int DT, int DVT>
__global__ void __launch_bounds__(NT) bwd_dv_kernel(BwdParams p) {
    extern __shared__ float sm[];
    constexpr bool FX = DT > 0;  // d, dv fixed at compile time
    const int d = FX ? DT : p.d, dv = FX ? DVT : p.dv_dim;
    const int ldq = d + 1, ldv = dv + 1;
    const int c = blockIdx.x, bh = blockIdx.y;
    const int64_t t0 = (int64_t)c * C;
    const int nv = (int)min64(C, p.T - t0);
    float* Qf = sm;
    float* Kf = Qf + C * ldq;
    float* Gs = Kf + C * ldq;
    float* Rs = Gs + C * ldv;
    float* Ss = Rs + d * ldv;
    float* rs = Ss + C * LDS;
    const int64_t row0 = (int64_t)bh * p.T + t0;
    TI* dvo = static_cast<TI*>(p.dv) + row0 * dv;

    load_rows(Qf, ldq, static_cast<const TI*>(p.q) + row0 * d, d, nv, true);
    load_rows(Kf, ldq, static_cast<const TI*>(p.k) + row0 * d, d, nv, true);
    load_g(Gs, ldv, nullptr, p, row0, nv);
    load_record(Rs, ldv, rs, p.rev + ((int64_t)bh * p.nch + c) * p.rec, d, dv);
    __syncthreads();
    scores<FX>(Ss, Qf, Kf, ldq, d);
    __syncthreads();
    // dv_j = sum_{t >= j} S_tj g_t + R^T phi(k_j)
    Tile<FX, true> tl(dv);
    tl.add_range(Ss, 1, LDS, Gs, ldv, 1, 4 * tl.rg, FX ? C : nv);  // queries t >= j
    tl.add(Kf, ldq, 1, Rs, ldv, 1, d, 0, C);
    tl.store(0, nv, [&](int j, int n, float x) { bst(dvo + (int64_t)j * dv + n, x); });
}

// ------------------------------------------------------------------ exclusive scans over chunks
// grid (ceil(len / 4 / NT), B*H); thread e walks elements 4e..4e+3 of every record of its bh in chunk
// order (reverse order when asked), replacing each record by the running sum before it.
__global__ void __launch_bounds__(NT) scan_states_kernel(ScanParams p) {
    // four consecutive elements per thread (len = d (dv + 1) and d * dv are multiples of 8,
    // so a group never straddles M and z and the records' float4 slots are aligned); the
    // loads of up to G records are issued together, then the exclusive sums are stored
    constexpr int G = 8;
    const int64_t n4 = p.len / 4;
    const int64_t e4 = (int64_t)blockIdx.x * NT + threadIdx.x;
    if (e4 >= n4) return;
    const int bh = blockIdx.y;
    const int64_t dd = (int64_t)p.d * p.dv, e = 4 * e4;
    float run[4] = {0.f, 0.f, 0.f, 0.f};
    const float* base = e < dd ? (p.base_M ? p.base_M + (int64_t)bh * dd + e : nullptr)
                               : (p.base_z ? p.base_z + (int64_t)bh * p.d + (e - dd) : nullptr);
    if (base)
#pragma unroll
        for (int u = 0; u < 4; ++u) run[u] = base[u];
    float4* r = reinterpret_cast<float4*>(p.rec + (int64_t)bh * p.nch * p.len) + e4;
    for (int i = 0; i < p.nch; i += G) {
        float4 x[G];
#pragma unroll
        for (int u = 0; u < G; ++u)
            if (i + u < p.nch) x[u] = r[(int64_t)(p.reverse ? p.nch - 1 - (i + u) : i + u) * n4];
#pragma unroll
        for (int u = 0; u < G; ++u)
            if (i + u < p.nch) {
                r[(int64_t)(p.reverse ? p.nch - 1 - (i + u) : i + u) * n4] = make_float4(run[0], run[1], run[2], run[3]);
                run[0] += x[u].x, run[1] += x[u].y, run[2] += x[u].z, run[3] += x[u].w;
            }
    }
    float* tot = e < dd ? (p.total_M ? p.total_M + (int64_t)bh * dd + e : nullptr)
                        : (p.total_z ? p.total_z + (int64_t)bh * p.d + (e - dd) : nullptr);
    if (tot)
#pragma unroll
        for (int u = 0; u < 4; ++u) tot[u] = run[u];
}

size_t dq_smem(int d, int dv) {
    return sizeof(float) * (2 * (size_t)C * (d + 1) + 2 * (size_t)C * (dv + 1) + (size_t)d * (dv + 1) +
                            (size_t)C * LDS + d + 2 * C);
}
size_t dk_smem(int d, int dv) {
    return sizeof(float) * (2 * (size_t)C * (d + 1) + 2 * (size_t)C * (dv + 1) + (size_t)d * (dv + 1) +
                            (size_t)C * LDS + d + C);
}
size_t dv_smem(int d, int dv) {
    return sizeof(float) * (2 * (size_t)C * (d + 1) + (size_t)C * (dv + 1) + (size_t)d * (dv + 1) +
                            (size_t)C * LDS + d);
}
size_t sums_smem(int d, int dv) { return sizeof(float) * ((size_t)C * (d + 1) + (size_t)C * (dv + 1)); }

template <typename F32Fn, typename BF16Fn>
cudaError_t launch_chunk_kernel(F32Fn f32, BF16Fn bf, const BwdParams& p, bool bf16, size_t smem, cudaStream_t s) {
    const void* fn = bf16 ? (const void*)bf : (const void*)f32;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.nch, p.B * p.H);
    if (bf16)
        bf<<<grid, NT, smem, s>>>(p);
    else
        f32<<<grid, NT, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_floats(int64_t BH, int64_t T, int d, int dv, size_t* off_rev, size_t* off_G, size_t* off_E) {
    const int64_t nch = (T + C - 1) / C;
    const size_t rec = (size_t)d * dv + d;
    auto up = [](size_t n) { return (n + 63) & ~(size_t)63; };  // 256-byte multiples
    const size_t s_rec = up((size_t)BH * nch * rec);
    const size_t s_G = up((size_t)BH * T * dv);
    const size_t s_E = up((size_t)BH * T);
    *off_rev = s_rec;
    *off_G = 2 * s_rec;
    *off_E = 2 * s_rec + s_G;
    return 2 * s_rec + s_G + s_E;
}

cudaError_t launch_scan_states(const ScanParams& p, cudaStream_t s) {
    if (p.len % 8 != 0) return cudaErrorInvalidValue;  // d, dv multiples of 8
    dim3 grid((unsigned)((p.len / 4 + NT - 1) / NT), p.BH);
    scan_states_kernel<<<grid, NT, 0, s>>>(p);
    return cudaGetLastError();
}

// Calls f with the compile-time shape (D, DV) of the specialised kernels, or (0, 0).
template <class F>
cudaError_t by_shape(const BwdParams& p, F f) {
    using I64 = std::integral_constant<int, 64>;
    using I128 = std::integral_constant<int, 128>;
    if (p.d == 64 && p.dv_dim == 64) return f(I64{}, I64{});
    if (p.d == 128 && p.dv_dim == 128) return f(I128{}, I128{});
    if (p.d == 64 && p.dv_dim == 128) return f(I64{}, I128{});
    if (p.d == 128 && p.dv_dim == 64) return f(I128{}, I64{});
    return f(std::integral_constant<int, 0>{}, std::integral_constant<int, 0>{});
}

cudaError_t launch_bwd_sums(const BwdParams& p, bool bf16, cudaStream_t s) {
    return by_shape(p, [&](auto D, auto DV) {
        return launch_chunk_kernel(bwd_sums_kernel<float, D(), DV()>, bwd_sums_kernel<__nv_bfloat16, D(), DV()>, p,
                                   bf16, sums_smem(p.d, p.dv_dim), s);
    });
}

cudaError_t launch_bwd_dq(const BwdParams& p, bool bf16, cudaStream_t s) {
    return by_shape(p, [&](auto D, auto DV) {
        return launch_chunk_kernel(bwd_dq_kernel<float, D(), DV()>, bwd_dq_kernel<__nv_bfloat16, D(), DV()>, p, bf16,
                                   dq_smem(p.d, p.dv_dim), s);
    });
}

cudaError_t launch_bwd_dk(const BwdParams& p, bool bf16, cudaStream_t s) {
    return by_shape(p, [&](auto D, auto DV) {
        return launch_chunk_kernel(bwd_dk_kernel<float, D(), DV()>, bwd_dk_kernel<__nv_bfloat16, D(), DV()>, p, bf16,
                                   dk_smem(p.d, p.dv_dim), s);
    });
}

cudaError_t launch_bwd_dv(const BwdParams& p, bool bf16, cudaStream_t s) {
    return by_shape(p, [&](auto D, auto DV) {
        return launch_chunk_kernel(bwd_dv_kernel<float, D(), DV()>, bwd_dv_kernel<__nv_bfloat16, D(), DV()>, p, bf16,
                                   dv_smem(p.d, p.dv_dim), s);
    });
}

}  // namespace la
