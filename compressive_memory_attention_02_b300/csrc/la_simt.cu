// SIMT (CUDA-core) kernels:
//   * fwd_simt      chunked causal forward in float32 arithmetic for any supported
//                   d, dv, chunk and for float32 or bf16 storage. It is the path of
//                   LA_F32 (whose 1e-4 tolerance rules out bf16 or tf32 tensor-core
//                   operands) and of bf16 shapes the tensor-core kernels do not take.
//   * parts_simt    per-part key-value sums (prefill partial states) in float32.
//   * reduce_parts  ordered sum of per-part states onto the initial state.
//   * prefill_out   last-token read-out from a final state.
//   * decode_step   one recurrent token per (stream, head): memory-bound RMW of M, z.
// All follow the token recurrence of the page "Attention_Kernel_Mask"
// (section "Implementing Causality with Cumulative Sums") with phi = elu + 1;
// fwd_simt uses that page's chunk-sequential (mode 3) split of each chunk into
// an inter-chunk term read from the carried state and a masked intra-chunk term.
#include "la_internal.h"

namespace la {

template <typename T>
__device__ __forceinline__ float ldf(const T* p);
template <>
__device__ __forceinline__ float ldf<float>(const float* p) {
    return __ldg(p);
}
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void stf(T* p, float x);
template <>
__device__ __forceinline__ void stf<float>(float* p, float x) {
    *p = x;
}
template <>
__device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16* p, float x) {
    *p = __float2bfloat16_rn(x);
}

// phi = elu + 1, or the value itself when q and k hold feature values already
__device__ __forceinline__ float phi_x(float x, int ident) { return ident ? x : phi_f(x); }

// ------------------------------------------------------------------ forward
// One block per (b, h). Shared memory (float): M[d*dv] z[d] Q[C*d] K[C*d] V[C*dv] S[C*C] den[C].
template <typename TI>
__global__ void __launch_bounds__(256) fwd_simt_kernel(FwdParams p) {
    extern __shared__ float sm[];
    const int d = p.d, dv = p.dv, C = p.chunk;
    const int bh = blockIdx.x;
    const int b = bh / p.H, h = bh % p.H;
    const int tid = threadIdx.x, nt = blockDim.x;
    float* Ms = sm;
    float* zs = Ms + d * dv;
    float* Qs = zs + d;
    float* Ks = Qs + C * d;
    float* Vs = Ks + C * d;
    float* Ss = Vs + C * dv;
    float* ds = Ss + C * C;
    // element offsets of this head in q, k, v, out (every access is checked against the
    // buffer's extent in the checked build)
    const TI* q = static_cast<const TI*>(p.q);
    const TI* k = static_cast<const TI*>(p.k);
    const TI* v = static_cast<const TI*>(p.v);
    TI* o = static_cast<TI*>(p.out);
    const int64_t qh = b * p.st.q_sb + h * p.st.q_sh, kh = b * p.st.k_sb + h * p.st.k_sh;
    const int64_t vh = b * p.st.v_sb + h * p.st.v_sh, oh = b * p.st.o_sb + h * p.st.o_sh;

    for (int i = tid; i < d * dv; i += nt) {
        const int64_t e = (int64_t)bh * d * dv + i;
        Ms[i] = p.M_in && inb(e, 1, p.ext.M_in, p.status) ? p.M_in[e] : 0.f;
    }
    for (int i = tid; i < d; i += nt) {
        const int64_t e = (int64_t)bh * d + i;
        zs[i] = p.z_in && inb(e, 1, p.ext.z_in, p.status) ? p.z_in[e] : 0.f;
    }

    for (int64_t c0 = 0; c0 < p.T; c0 += C) {
        const int n = (int)min64(C, p.T - c0);
        __syncthreads();
        for (int idx = tid; idx < C * d; idx += nt) {
            const int t = idx / d, i = idx % d;
            float qf = 0.f, kf = 0.f;
            if (t < n) {
                const int64_t iq = qh + (c0 + t) * p.st.q_st + i, ik = kh + (c0 + t) * p.st.k_st + i;
                if (inb(iq, 1, p.ext.q, p.status)) qf = phi_x(ldf(q + iq), p.phi_ident);
                if (inb(ik, 1, p.ext.k, p.status)) kf = phi_x(ldf(k + ik), p.phi_ident);
            }
            Qs[idx] = qf;
            Ks[idx] = kf;  // rows past the end stay 0: phi of padding must not enter z
        }
        for (int idx = tid; idx < C * dv; idx += nt) {
            const int t = idx / dv, j = idx % dv;
            const int64_t iv = vh + (c0 + t) * p.st.v_st + j;
            Vs[idx] = (t < n && inb(iv, 1, p.ext.v, p.status)) ? ldf(v + iv) : 0.f;
        }
        __syncthreads();
        // intra-chunk scores, lower triangle with diagonal
        for (int idx = tid; idx < C * C; idx += nt) {
            const int t = idx / C, s = idx % C;
            float acc = 0.f;
            if (s <= t && t < n) {
                const float* qr = Qs + t * d;
                const float* kr = Ks + s * d;
                for (int i = 0; i < d; ++i) acc = fmaf(qr[i], kr[i], acc);
            }
            Ss[idx] = acc;
        }
        __syncthreads();
        // denominator: inter (phi q . z_{c-1}) + intra row sum + eps
        for (int t = tid; t < n; t += nt) {
            float inter = 0.f, intra = 0.f;
            const float* qr = Qs + t * d;
            for (int i = 0; i < d; ++i) inter = fmaf(qr[i], zs[i], inter);
            for (int s = 0; s <= t; ++s) intra += Ss[t * C + s];
            ds[t] = inter + intra + p.eps;
        }
        __syncthreads();
        // numerator: phi q . M_{c-1} + masked S . V
        for (int idx = tid; idx < n * dv; idx += nt) {
            const int t = idx / dv, j = idx % dv;
            float inter = 0.f, intra = 0.f;
            const float* qr = Qs + t * d;
            for (int i = 0; i < d; ++i) inter = fmaf(qr[i], Ms[i * dv + j], inter);
            for (int s = 0; s <= t; ++s) intra = fmaf(Ss[t * C + s], Vs[s * dv + j], intra);
            const int64_t io = oh + (c0 + t) * p.st.o_st + j;
            if (inb(io, 1, p.ext.o, p.status)) stf(o + io, (inter + intra) / ds[t]);
        }
        __syncthreads();
        // state update: M += phi(K)^T V, z += sum phi(K)
        for (int idx = tid; idx < d * dv; idx += nt) {
            const int i = idx / dv, j = idx % dv;
            float acc = 0.f;
            for (int s = 0; s < n; ++s) acc = fmaf(Ks[s * d + i], Vs[s * dv + j], acc);
            Ms[idx] += acc;
        }
        for (int i = tid; i < d; i += nt) {
            float acc = 0.f;
            for (int s = 0; s < n; ++s) acc += Ks[s * d + i];
            zs[i] += acc;
        }
    }
    __syncthreads();
    if (p.M_out)
        for (int i = tid; i < d * dv; i += nt) {
            const int64_t e = (int64_t)bh * d * dv + i;
            if (inb(e, 1, p.ext.M_out, p.status)) p.M_out[e] = Ms[i];
        }
    if (p.z_out)
        for (int i = tid; i < d; i += nt) {
            const int64_t e = (int64_t)bh * d + i;
            if (inb(e, 1, p.ext.z_out, p.status)) p.z_out[e] = zs[i];
        }
}

// ------------------------------------------------------------------ per-part state sums
// grid (nparts, B*H). Part p covers tokens [p*L, min(T, (p+1)*L)). Writes
//   A_p = sum phi(k_t) v_t^T (d x dv) and s_p = sum phi(k_t) (d)
// to dst_M[(bh*nparts + p) * rec], dst_z[...] (rec = record stride in floats), after
// adding base (M_in, z_in of this bh) when base pointers are given. With final_out
// (nparts == 1), also computes out_last from the complete state.
// Shared memory (float): A[d*dv] s[d] K[TILE*d] V[TILE*dv] fq[d]
template <typename TI>
__global__ void __launch_bounds__(256) parts_simt_kernel(PartsParams p) {
    extern __shared__ float sm[];
    constexpr int TILE = 32;
    const int d = p.d, dv = p.dv;
    const int part = blockIdx.x, bh = blockIdx.y;
    const int b = bh / p.H, h = bh % p.H;
    const int tid = threadIdx.x, nt = blockDim.x;
    float* As = sm;
    float* ss = As + d * dv;
    float* Ks = ss + d;
    float* Vs = Ks + TILE * d;
    float* fq = Vs + TILE * dv;
    const TI* k = static_cast<const TI*>(p.k);
    const TI* v = static_cast<const TI*>(p.v);
    const int64_t kh = b * p.st.k_sb + h * p.st.k_sh, vh = b * p.st.v_sb + h * p.st.v_sh;
    const int64_t t_begin = (int64_t)part * p.part_len;
    const int64_t t_end = min64(p.T, t_begin + p.part_len);

    for (int i = tid; i < d * dv; i += nt) As[i] = 0.f;
    for (int i = tid; i < d; i += nt) ss[i] = 0.f;
    for (int64_t t0 = t_begin; t0 < t_end; t0 += TILE) {
        const int n = (int)min64(TILE, t_end - t0);
        __syncthreads();
        for (int idx = tid; idx < TILE * d; idx += nt) {
            const int t = idx / d, i = idx % d;
            const int64_t ik = kh + (t0 + t) * p.st.k_st + i;
            Ks[idx] = (t < n && inb(ik, 1, p.ext.k, p.status)) ? phi_x(ldf(k + ik), p.phi_ident) : 0.f;
        }
        for (int idx = tid; idx < TILE * dv; idx += nt) {
            const int t = idx / dv, j = idx % dv;
            const int64_t iv = vh + (t0 + t) * p.st.v_st + j;
            Vs[idx] = (t < n && inb(iv, 1, p.ext.v, p.status)) ? ldf(v + iv) : 0.f;
        }
        __syncthreads();
        for (int idx = tid; idx < d * dv; idx += nt) {
            const int i = idx / dv, j = idx % dv;
            float acc = As[idx];
            for (int s = 0; s < n; ++s) acc = fmaf(Ks[s * d + i], Vs[s * dv + j], acc);
            As[idx] = acc;
        }
        for (int i = tid; i < d; i += nt) {
            float acc = ss[i];
            for (int s = 0; s < n; ++s) acc += Ks[s * d + i];
            ss[i] = acc;
        }
    }
    __syncthreads();
    if (p.base_M)
        for (int i = tid; i < d * dv; i += nt) {
            const int64_t e = (int64_t)bh * d * dv + i;
            if (inb(e, 1, p.ext.M_in, p.status)) As[i] += p.base_M[e];
        }
    if (p.base_z)
        for (int i = tid; i < d; i += nt) {
            const int64_t e = (int64_t)bh * d + i;
            if (inb(e, 1, p.ext.z_in, p.status)) ss[i] += p.base_z[e];
        }
    __syncthreads();
    const int64_t rec = (int64_t)bh * p.nparts + part;
    if (p.dst_M)
        for (int i = tid; i < d * dv; i += nt) {
            const int64_t e = rec * p.rec_M + i;
            if (inb(e, 1, p.ext.M_out, p.status)) p.dst_M[e] = As[i];
        }
    if (p.dst_z)
        for (int i = tid; i < d; i += nt) {
            const int64_t e = rec * p.rec_z + i;
            if (inb(e, 1, p.ext.z_out, p.status)) p.dst_z[e] = ss[i];
        }
    if (p.out_last) {  // only launched with nparts == 1
        const TI* q = static_cast<const TI*>(p.q);
        const int64_t qt = b * p.st.q_sb + h * p.st.q_sh + (p.T - 1) * p.st.q_st;
        for (int i = tid; i < d; i += nt)
            fq[i] = inb(qt + i, 1, p.ext.q, p.status) ? phi_x(ldf(q + qt + i), p.phi_ident) : 0.f;
        __syncthreads();
        float den = p.eps;
        for (int i = 0; i < d; ++i) den = fmaf(fq[i], ss[i], den);
        TI* o = static_cast<TI*>(p.out_last);
        for (int j = tid; j < dv; j += nt) {
            float num = 0.f;
            for (int i = 0; i < d; ++i) num = fmaf(fq[i], As[i * dv + j], num);
            const int64_t e = (int64_t)bh * dv + j;
            if (inb(e, 1, p.ext.o, p.status)) stf(o + e, num / den);
        }
    }
}

// ------------------------------------------------------------------ ordered reduction of parts
// grid (ceil((d*dv + d)/4 / 256), B*H): element e of [M | z] for this bh is
// base[e] + sum_{p=0}^{nparts-1} part_p[e], summed in part order (deterministic).
__global__ void __launch_bounds__(256) reduce_parts_kernel(ReduceParams p) {
    const int bh = blockIdx.y;
    const int dd = p.d * p.dv;
    const int n4 = (dd + p.d) / 4;
    const int e4 = blockIdx.x * blockDim.x + threadIdx.x;
    if (e4 >= n4) return;
    const int e = e4 * 4;
    const bool isM = e < dd;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t se = isM ? (int64_t)bh * dd + e : (int64_t)bh * p.d + (e - dd);  // state element
    if (isM ? (p.base_M != nullptr) : (p.base_z != nullptr)) {
        const float* src = isM ? p.base_M : p.base_z;
        if (inb(se, 4, isM ? p.ext.M_in : p.ext.z_in, p.status)) acc = *reinterpret_cast<const float4*>(src + se);
    }
    // part records: parts_M / parts_z are the M and z views of one record array of p.ext.ws
    // floats that starts at parts_M
    const float* part = isM ? p.parts_M + (int64_t)bh * p.nparts * p.rec_M + e
                            : p.parts_z + (int64_t)bh * p.nparts * p.rec_z + (e - dd);
    const int64_t stride = isM ? p.rec_M : p.rec_z;
    for (int i = 0; i < p.nparts; ++i) {
        if (!inb((part + i * stride) - p.parts_M, 4, p.ext.ws, p.status)) continue;
        const float4 x = *reinterpret_cast<const float4*>(part + i * stride);
        acc.x += x.x;
        acc.y += x.y;
        acc.z += x.z;
        acc.w += x.w;
    }
    float* dst = isM ? p.dst_M : p.dst_z;
    if (inb(se, 4, isM ? p.ext.M_out : p.ext.z_out, p.status)) *reinterpret_cast<float4*>(dst + se) = acc;
}

// ------------------------------------------------------------------ last-token read-out
// grid B*H, block 128: out[bh, j] = phi(q_T) . M_T[:, j] / (phi(q_T) . z_T + eps)
template <typename TI>
__global__ void __launch_bounds__(128) prefill_out_kernel(PrefillOutParams p) {
    __shared__ float fq[128];
    __shared__ float red[4];
    const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;
    const int tid = threadIdx.x;
    const TI* q = static_cast<const TI*>(p.q);
    const int64_t qt = b * p.st.q_sb + h * p.st.q_sh + (p.T - 1) * p.st.q_st;
    float part = 0.f;
    if (tid < p.d) {
        const int64_t ez = (int64_t)bh * p.d + tid;
        fq[tid] = inb(qt + tid, 1, p.ext.q, p.status) ? phi_f(ldf(q + qt + tid)) : 0.f;
        part = inb(ez, 1, p.ext.z_out, p.status) ? fq[tid] * p.z[ez] : 0.f;
    }
    for (int off = 16; off; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if ((tid & 31) == 0) red[tid >> 5] = part;
    __syncthreads();
    const float den = red[0] + red[1] + red[2] + red[3] + p.eps;
    const int64_t mh = (int64_t)bh * p.d * p.dv;
    for (int j = tid; j < p.dv; j += blockDim.x) {
        float num = 0.f;
        for (int i = 0; i < p.d; ++i) {
            const int64_t e = mh + (int64_t)i * p.dv + j;
            if (inb(e, 1, p.ext.M_out, p.status)) num = fmaf(fq[i], p.M[e], num);
        }
        const int64_t eo = (int64_t)bh * p.dv + j;
        if (inb(eo, 1, p.ext.o, p.status)) stf(static_cast<TI*>(p.out) + eo, num / den);
    }
}

// ------------------------------------------------------------------ decode step
// grid (N*H, ceil(dv/64)), block 256, three blocks per SM. Block (nh, c) updates
// columns [64c, 64c + 64) of M for every row and writes those outputs; it forms the
// full denominator phi(q).(z + phi(k)) itself, and block c = 0 writes z back.
// Thread (rg, cg) owns the float4 column group cg of rows rg, rg + R, ...
// (R = 256 / (width/4), at most 8 rows); a warp covers 256 contiguous bytes of two
// rows, so every load and store of M is a coalesced 128-bit access. The thread's rows
// of M are requested first, before q, k, v and z, so the state stream does not wait
// for the token's round trip; all of them are in flight before any is used.
constexpr int DEC_NT = 256;
constexpr int DEC_CW = 64;  // columns per block

template <typename TI>
__global__ void __launch_bounds__(DEC_NT, 3) decode_kernel(DecodeParams p) {
    constexpr int MAXR = 8;  // d * DEC_CW / (4 * DEC_NT) rows per thread at d = 128
    __shared__ float fq[128], fk[128];
    __shared__ __align__(16) float vv[128];
    __shared__ float4 red[DEC_NT];
    __shared__ float dred[DEC_NT / 32];
    const int nh = blockIdx.x;
    const int c0 = blockIdx.y * DEC_CW;
    const int tid = threadIdx.x;
    const int d = p.d, dv = p.dv;
    const int width = min(DEC_CW, dv - c0);
    const int ncg = width >> 2;
    const int R = DEC_NT / ncg;
    const int cg = tid % ncg, rg = tid / ncg;
    const int nrows = rg < R ? (d - rg + R - 1) / R : 0;  // rows rg, rg+R, ... < d (threads past R*ncg idle)
    const int rs4 = dv >> 2;                               // row stride of M in float4
    const int64_t m0 = (int64_t)nh * d * dv + c0 + 4 * cg;  // element of M at (row 0, this column group)
    float4* M4 = reinterpret_cast<float4*>(p.M + m0);
    float4 m[MAXR];
#pragma unroll
    for (int r = 0; r < MAXR; ++r)
        if (r < nrows && inb(m0 + (int64_t)(rg + r * R) * dv, 4, p.ext.M_out, p.status))
            m[r] = __ldcs(M4 + (int64_t)(rg + r * R) * rs4);
        else
            m[r] = make_float4(0.f, 0.f, 0.f, 0.f);

    const TI* q = static_cast<const TI*>(p.q);
    const TI* k = static_cast<const TI*>(p.k);
    const TI* v = static_cast<const TI*>(p.v);
    const int64_t qk0 = (int64_t)nh * d, v0 = (int64_t)nh * dv + c0;
    float zo = 0.f;
    if (tid < d) {
        if (inb(qk0 + tid, 1, p.ext.z_out, p.status)) zo = p.z[qk0 + tid];
        fq[tid] = inb(qk0 + tid, 1, p.ext.q, p.status) ? phi_f(ldf(q + qk0 + tid)) : 0.f;
        fk[tid] = inb(qk0 + tid, 1, p.ext.k, p.status) ? phi_f(ldf(k + qk0 + tid)) : 0.f;
    }
    if (tid < width) vv[tid] = inb(v0 + tid, 1, p.ext.v, p.status) ? ldf(v + v0 + tid) : 0.f;
    __syncthreads();
    // z <- z + phi(k) (written by the first column block); den = phi(q) . z + eps
    float part = 0.f;
    if (tid < d) {
        const float zn = zo + fk[tid];
        if (blockIdx.y == 0 && inb(qk0 + tid, 1, p.ext.z_out, p.status)) p.z[qk0 + tid] = zn;
        part = fq[tid] * zn;
    }
    for (int off = 16; off; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if ((tid & 31) == 0) dred[tid >> 5] = part;

    const float4 v4 = reinterpret_cast<const float4*>(vv)[cg];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < MAXR; ++r) {
        if (r < nrows) {
            const int i = rg + r * R;
            const float a = fk[i], g = fq[i];
            float4 x = m[r];
            x.x = fmaf(a, v4.x, x.x);
            x.y = fmaf(a, v4.y, x.y);
            x.z = fmaf(a, v4.z, x.z);
            x.w = fmaf(a, v4.w, x.w);
            if (inb(m0 + (int64_t)i * dv, 4, p.ext.M_out, p.status)) __stcs(M4 + (int64_t)i * rs4, x);
            acc.x = fmaf(g, x.x, acc.x);
            acc.y = fmaf(g, x.y, acc.y);
            acc.z = fmaf(g, x.z, acc.z);
            acc.w = fmaf(g, x.w, acc.w);
        }
    }
    red[tid] = acc;
    __syncthreads();
    if (tid < ncg) {
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < R; ++r) {
            const float4 x = red[r * ncg + tid];
            s.x += x.x;
            s.y += x.y;
            s.z += x.z;
            s.w += x.w;
        }
        float den = p.eps;
        for (int w = 0; w < 4; ++w) den += dred[w];  // threads >= d (<= 128) add nothing
        const int64_t eo = (int64_t)nh * dv + c0 + tid * 4;
        TI* o = static_cast<TI*>(p.out) + eo;
        if (inb(eo, 4, p.ext.o, p.status)) {
            stf(o + 0, s.x / den);
            stf(o + 1, s.y / den);
            stf(o + 2, s.z / den);
            stf(o + 3, s.w / den);
        }
    }
}

// ------------------------------------------------------------------ launchers
size_t fwd_simt_smem(int d, int dv, int C) {
    return sizeof(float) * ((size_t)d * dv + d + (size_t)C * (2 * d + dv) + (size_t)C * C + C);
}

size_t parts_simt_smem(int d, int dv) { return sizeof(float) * ((size_t)d * dv + d + 32 * (d + dv) + d); }

template <typename TI>
static cudaError_t set_smem(const void* fn, size_t smem) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

cudaError_t launch_fwd_simt(const FwdParams& p, bool bf16, cudaStream_t s) {
    const size_t smem = fwd_simt_smem(p.d, p.dv, p.chunk);
    const void* fn = bf16 ? (const void*)fwd_simt_kernel<__nv_bfloat16> : (const void*)fwd_simt_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (bf16)
        fwd_simt_kernel<__nv_bfloat16><<<p.B * p.H, 256, smem, s>>>(p);
    else
        fwd_simt_kernel<float><<<p.B * p.H, 256, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_parts_simt(const PartsParams& p, bool bf16, cudaStream_t s) {
    const size_t smem = parts_simt_smem(p.d, p.dv);
    const void* fn = bf16 ? (const void*)parts_simt_kernel<__nv_bfloat16> : (const void*)parts_simt_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(p.nparts, p.B * p.H);
    if (bf16)
        parts_simt_kernel<__nv_bfloat16><<<grid, 256, smem, s>>>(p);
    else
        parts_simt_kernel<float><<<grid, 256, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_reduce_parts(const ReduceParams& p, cudaStream_t s) {
    const int n4 = (p.d * p.dv + p.d) / 4;
    dim3 grid((n4 + 255) / 256, p.BH);
    reduce_parts_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_prefill_out(const PrefillOutParams& p, bool bf16, cudaStream_t s) {
    if (bf16)
        prefill_out_kernel<__nv_bfloat16><<<p.B * p.H, 128, 0, s>>>(p);
    else
        prefill_out_kernel<float><<<p.B * p.H, 128, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, bool bf16, cudaStream_t s) {
    if (bf16)
        decode_kernel<__nv_bfloat16><<<dim3(p.N * p.H, (p.dv + DEC_CW - 1) / DEC_CW), DEC_NT, 0, s>>>(p);
    else
        decode_kernel<float><<<dim3(p.N * p.H, (p.dv + DEC_CW - 1) / DEC_CW), DEC_NT, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace la
