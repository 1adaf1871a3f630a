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
// Launches (la_api.cu): 64-token key-value sums (parts_simt) -> exclusive prefix scan
// (the state before each chunk) -> bwd_dq (dq, G, E and the chunk sums phi(Q)^T G,
// phi(Q)^T e) -> exclusive reverse scan (R_c; the totals are dM_in, dz_in) -> bwd_dk ->
// bwd_dv. A chunk kernel runs one block of 256 threads per (chunk, b*H + h) with every
// operand of the chunk in shared memory; tile rows are padded by one float so that
// column-wise reads by consecutive threads fall in distinct banks.
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

// Rows 0..C-1 of a contiguous [rows, n] slice into a tile with row stride ld (phi applied
// when asked); rows >= nv become 0.
template <typename TI>
__device__ void load_rows(float* dst, int ld, const TI* src, int n, int nv, bool apply_phi) {
    for (int idx = threadIdx.x; idx < C * n; idx += NT) {
        const int t = idx / n, i = idx - t * n;
        float x = 0.f;
        if (t < nv) {
            x = bld(src + (int64_t)t * n + i);
            if (apply_phi) x = phi_f(x);
        }
        dst[t * ld + i] = x;
    }
}

// A state record (M row-major d x dv, then z) into Ms (row stride ld) and zs.
__device__ void load_record(float* Ms, int ld, float* zs, const float* rec, int d, int dv) {
    for (int idx = threadIdx.x; idx < d * dv; idx += NT) {
        const int i = idx / dv, j = idx - i * dv;
        Ms[i * ld + j] = rec[idx];
    }
    for (int i = threadIdx.x; i < d; i += NT) zs[i] = rec[(int64_t)d * dv + i];
}

// S_tj = phi(q_t) . phi(k_j) for j <= t, else 0.
__device__ void scores(float* Ss, const float* Qf, const float* Kf, int ldq, int d) {
    for (int o = threadIdx.x; o < C * C; o += NT) {
        const int t = o / C, j = o - t * C;
        float acc = 0.f;
        if (j <= t) {
            const float* a = Qf + t * ldq;
            const float* b = Kf + j * ldq;
            for (int i = 0; i < d; ++i) acc = fmaf(a[i], b[i], acc);
        }
        Ss[t * LDS + j] = acc;
    }
}

// dA_tj = g_t . v_j + e_t for j <= t, else 0.
__device__ void score_grads(float* dA, const float* Gs, const float* Vs, const float* ee, int ldv, int dv) {
    for (int o = threadIdx.x; o < C * C; o += NT) {
        const int t = o / C, j = o - t * C;
        float acc = 0.f;
        if (j <= t) {
            const float* a = Gs + t * ldv;
            const float* b = Vs + j * ldv;
            for (int n = 0; n < dv; ++n) acc = fmaf(a[n], b[n], acc);
            acc += ee[t];
        }
        dA[t * LDS + j] = acc;
    }
}

// ------------------------------------------------------------------ dq, G, E, chunk sums
// Shared memory (float): Qf, Kf [C][d+1]; Vs, Os [C][dv+1]; Ms [d][dv+1]; Ss [C][C+1];
// zs [d]; den, ee [C]. Os holds the numerator, then out, then g.
template <typename TI>
__global__ void __launch_bounds__(NT) bwd_dq_kernel(BwdParams p) {
    extern __shared__ float sm[];
    const int d = p.d, dv = p.dv_dim;
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
    const TI* q = static_cast<const TI*>(p.q) + row0 * d;
    const TI* k = static_cast<const TI*>(p.k) + row0 * d;
    const TI* v = static_cast<const TI*>(p.v) + row0 * dv;
    const TI* dout = static_cast<const TI*>(p.dout) + row0 * dv;
    TI* dq = static_cast<TI*>(p.dq) + row0 * d;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    load_rows(Qf, ldq, q, d, nv, true);
    load_rows(Kf, ldq, k, d, nv, true);
    load_rows(Vs, ldv, v, dv, nv, false);
    load_record(Ms, ldv, zs, p.states + ((int64_t)bh * p.nch + c) * p.rec, d, dv);
    __syncthreads();
    scores(Ss, Qf, Kf, ldq, d);
    __syncthreads();
    for (int t = warp; t < C; t += NT / 32) {  // D_t
        float s = 0.f;
        for (int i = lane; i < d; i += 32) s = fmaf(Qf[t * ldq + i], zs[i], s);
        for (int j = lane; j <= t; j += 32) s += Ss[t * LDS + j];
        s = warp_sum(s);
        if (lane == 0) den[t] = s + p.eps;
    }
    __syncthreads();
    for (int o = threadIdx.x; o < C * dv; o += NT) {  // out_t
        const int t = o / dv, n = o - t * dv;
        const float* a = Qf + t * ldq;
        const float* s = Ss + t * LDS;
        float acc = 0.f;
        for (int i = 0; i < d; ++i) acc = fmaf(a[i], Ms[i * ldv + n], acc);
        for (int j = 0; j <= t; ++j) acc = fmaf(s[j], Vs[j * ldv + n], acc);
        Os[t * ldv + n] = (t < nv) ? acc / den[t] : 0.f;
    }
    __syncthreads();
    for (int t = warp; t < C; t += NT / 32) {  // g_t and e_t
        float s = 0.f;
        for (int n = lane; n < dv; n += 32) {
            const float g = (t < nv) ? bld(dout + (int64_t)t * dv + n) / den[t] : 0.f;
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
    score_grads(Ss, Os, Vs, ee, ldv, dv);
    __syncthreads();
    for (int o = threadIdx.x; o < C * d; o += NT) {  // dq_t
        const int t = o / d, i = o - t * d;
        if (t >= nv) continue;
        const float* g = Os + t * ldv;
        const float* m = Ms + i * ldv;
        const float* s = Ss + t * LDS;
        float acc = ee[t] * zs[i];
        for (int n = 0; n < dv; ++n) acc = fmaf(m[n], g[n], acc);
        for (int j = 0; j <= t; ++j) acc = fmaf(s[j], Kf[j * ldq + i], acc);
        bst(dq + (int64_t)t * d + i, acc * fminf(Qf[t * ldq + i], 1.f));
    }
    // chunk sums phi(Q)^T G and phi(Q)^T e (no barrier needed: Qf, Os, ee are unchanged)
    float* rv = p.rev + ((int64_t)bh * p.nch + c) * p.rec;
    for (int o = threadIdx.x; o < d * dv; o += NT) {
        const int i = o / dv, n = o - i * dv;
        float acc = 0.f;
        for (int t = 0; t < nv; ++t) acc = fmaf(Qf[t * ldq + i], Os[t * ldv + n], acc);
        rv[o] = acc;
    }
    for (int i = threadIdx.x; i < d; i += NT) {
        float acc = 0.f;
        for (int t = 0; t < nv; ++t) acc = fmaf(Qf[t * ldq + i], ee[t], acc);
        rv[(int64_t)d * dv + i] = acc;
    }
}

// G and E rows of the chunk (rows >= nv become 0).
__device__ void load_g(float* Gs, int ldv, float* ee, const BwdParams& p, int64_t row0, int nv) {
    const int dv = p.dv_dim;
    for (int idx = threadIdx.x; idx < C * dv; idx += NT) {
        const int t = idx / dv, n = idx - t * dv;
        Gs[t * ldv + n] = (t < nv) ? p.G[(row0 + t) * dv + n] : 0.f;
    }
    for (int t = threadIdx.x; t < C; t += NT) ee[t] = (t < nv) ? p.E[row0 + t] : 0.f;
}

// ------------------------------------------------------------------ dk
// Shared memory (float): Qf, Kf [C][d+1]; Vs, Gs [C][dv+1]; Rs [d][dv+1]; dA [C][C+1];
// rs [d]; ee [C].
template <typename TI>
__global__ void __launch_bounds__(NT) bwd_dk_kernel(BwdParams p) {
    extern __shared__ float sm[];
    const int d = p.d, dv = p.dv_dim;
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
    const TI* q = static_cast<const TI*>(p.q) + row0 * d;
    const TI* k = static_cast<const TI*>(p.k) + row0 * d;
    const TI* v = static_cast<const TI*>(p.v) + row0 * dv;
    TI* dk = static_cast<TI*>(p.dk) + row0 * d;

    load_rows(Qf, ldq, q, d, nv, true);
    load_rows(Kf, ldq, k, d, nv, true);
    load_rows(Vs, ldv, v, dv, nv, false);
    load_g(Gs, ldv, ee, p, row0, nv);
    load_record(Rs, ldv, rs, p.rev + ((int64_t)bh * p.nch + c) * p.rec, d, dv);
    __syncthreads();
    score_grads(dA, Gs, Vs, ee, ldv, dv);
    __syncthreads();
    for (int o = threadIdx.x; o < C * d; o += NT) {
        const int j = o / d, i = o - j * d;
        if (j >= nv) continue;
        const float* r = Rs + i * ldv;
        const float* vj = Vs + j * ldv;
        float acc = rs[i];
        for (int n = 0; n < dv; ++n) acc = fmaf(r[n], vj[n], acc);
        for (int t = j; t < nv; ++t) acc = fmaf(dA[t * LDS + j], Qf[t * ldq + i], acc);
        bst(dk + (int64_t)j * d + i, acc * fminf(Kf[j * ldq + i], 1.f));
    }
}

// ------------------------------------------------------------------ dv
// Shared memory (float): Qf, Kf [C][d+1]; Gs [C][dv+1]; Rs [d][dv+1]; Ss [C][C+1]; rs [d],
// ee [C] (loaded with G, unused here).
template <typename TI>
__global__ void __launch_bounds__(NT) bwd_dv_kernel(BwdParams p) {
    extern __shared__ float sm[];
    const int d = p.d, dv = p.dv_dim;
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
    float* ee = rs + d;
    const int64_t row0 = (int64_t)bh * p.T + t0;
    const TI* q = static_cast<const TI*>(p.q) + row0 * d;
    const TI* k = static_cast<const TI*>(p.k) + row0 * d;
    TI* dvo = static_cast<TI*>(p.dv) + row0 * dv;

    load_rows(Qf, ldq, q, d, nv, true);
    load_rows(Kf, ldq, k, d, nv, true);
    load_g(Gs, ldv, ee, p, row0, nv);
    load_record(Rs, ldv, rs, p.rev + ((int64_t)bh * p.nch + c) * p.rec, d, dv);
    __syncthreads();
    scores(Ss, Qf, Kf, ldq, d);
    __syncthreads();
    for (int o = threadIdx.x; o < C * dv; o += NT) {
        const int j = o / dv, n = o - j * dv;
        if (j >= nv) continue;
        const float* kj = Kf + j * ldq;
        float acc = 0.f;
        for (int i = 0; i < d; ++i) acc = fmaf(kj[i], Rs[i * ldv + n], acc);
        for (int t = j; t < nv; ++t) acc = fmaf(Ss[t * LDS + j], Gs[t * ldv + n], acc);
        bst(dvo + (int64_t)j * dv + n, acc);
    }
}

// ------------------------------------------------------------------ exclusive scans over chunks
// grid (ceil(len / NT), B*H); thread e walks element e of every record of its bh in chunk
// order (reverse order when asked), replacing each record by the running sum before it.
__global__ void __launch_bounds__(NT) scan_states_kernel(ScanParams p) {
    const int64_t e = (int64_t)blockIdx.x * NT + threadIdx.x;
    if (e >= p.len) return;
    const int bh = blockIdx.y;
    const int64_t dd = (int64_t)p.d * p.dv;
    float run = 0.f;
    if (e < dd) {
        if (p.base_M) run = p.base_M[(int64_t)bh * dd + e];
    } else if (p.base_z) {
        run = p.base_z[(int64_t)bh * p.d + (e - dd)];
    }
    float* r = p.rec + (int64_t)bh * p.nch * p.len + e;
    auto at = [&](int i) -> float& { return r[(int64_t)(p.reverse ? p.nch - 1 - i : i) * p.len]; };
    int i = 0;
    for (; i + 8 <= p.nch; i += 8) {  // eight loads in flight, then eight stores
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = at(i + u);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            at(i + u) = run;
            run += x[u];
        }
    }
    for (; i < p.nch; ++i) {
        const float x = at(i);
        at(i) = run;
        run += x;
    }
    if (e < dd) {
        if (p.total_M) p.total_M[(int64_t)bh * dd + e] = run;
    } else if (p.total_z) {
        p.total_z[(int64_t)bh * p.d + (e - dd)] = run;
    }
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
                            (size_t)C * LDS + d + C);
}

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
    dim3 grid((unsigned)((p.len + NT - 1) / NT), p.BH);
    scan_states_kernel<<<grid, NT, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdParams& p, bool bf16, cudaStream_t s) {
    return launch_chunk_kernel(bwd_dq_kernel<float>, bwd_dq_kernel<__nv_bfloat16>, p, bf16, dq_smem(p.d, p.dv_dim), s);
}

cudaError_t launch_bwd_dk(const BwdParams& p, bool bf16, cudaStream_t s) {
    return launch_chunk_kernel(bwd_dk_kernel<float>, bwd_dk_kernel<__nv_bfloat16>, p, bf16, dk_smem(p.d, p.dv_dim), s);
}

cudaError_t launch_bwd_dv(const BwdParams& p, bool bf16, cudaStream_t s) {
    return launch_chunk_kernel(bwd_dv_kernel<float>, bwd_dv_kernel<__nv_bfloat16>, p, bf16, dv_smem(p.d, p.dv_dim), s);
}

}  // namespace la
