// Helpers shared by the tensor-core kernels: tile geometry, bounded waits that
// unwind consistently, and the in-place phi transform of a TMA-loaded tile.
#pragma once
#include "la_internal.h"

namespace la {

constexpr int CH = 64;                 // tokens per chunk on the tensor-core path
constexpr int ATOM = 64 * 128;         // one 64-row, 128-byte-wide swizzle block column
constexpr int KROWS = 80;              // forward K tile rows: 64 keys, z row, 15 zero rows
constexpr int ATOMK = KROWS * 128;

// Dynamic shared memory of a kernel, with the largest shared-memory carveout preferred:
// without that preference the driver may size the carveout for one block and keep a
// second block of a kernel that fits two per SM off the SM.
static inline cudaError_t set_smem_attrs(const void* fn, int bytes) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
}

// Round the dynamic shared-memory base up to 1024 bytes (the 128-byte swizzle repeats
// every 1024 bytes). Plain pointer arithmetic on the __shared__ array, so the compiler
// still knows every derived pointer is a shared-memory address (ld/st.shared rather
// than generic accesses).
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    return p + ((1024u - (a & 1023u)) & 1023u);
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
    if (mbar_test_wait(bar, parity)) return true;
    const unsigned long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > LA_WAIT_CYCLES) return false;
    }
    return true;
}

// phi on two packed bf16 values: exp(min(x, 0)) in f32 rounded to bf16, plus max(x, 0) in
// bf16. For x <= 0 that is the rounded exponential; for x > 0 the exponential is exactly
// 1 and the bf16 add rounds 1 + x once, so the result equals rounding the f32 value
// exp(min(x, 0)) + max(x, 0) to bf16.
__device__ __forceinline__ uint32_t phi_bf16x2(uint32_t w) {
    const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&w);
    const __nv_bfloat162 zero = __float2bfloat162_rn(0.f);
    const __nv_bfloat162 mn = __hmin2(x, zero);
    const uint32_t m = *reinterpret_cast<const uint32_t*>(&mn);
    constexpr float kLog2e = 1.4426950408889634f;
    const uint64_t y = f2_mul(f2_pack(bf16lo(m), bf16hi(m)), f2_pack(kLog2e, kLog2e));
    const __nv_bfloat162 e = __floats2bfloat162_rn(ex2_approx(f2_lo(y)), ex2_approx(f2_hi(y)));
    const __nv_bfloat162 r = __hadd2(e, __hmax2(x, zero));
    return *reinterpret_cast<const uint32_t*>(&r);
}

// phi in place on a [64 x D] bf16 tile (atoms `astride` bytes apart), by NT threads.
// Thread ct owns 16-byte chunk column j = ct % (D/8) of rows g, g + RG, ... below 64
// (g = ct / (D/8)); since RG is a multiple of 8 the swizzled chunk position
// j ^ (row % 8) is the same for all of its rows. Rows >= valid become 0 (phi(0) = 1
// must not enter the sums; pass valid = 64 to keep all rows). With colsum != nullptr
// the thread adds the bf16-rounded results of its 8 columns into colsum[0..8). With
// ident the tile already holds feature values (another map applied by the caller): rows
// below valid are kept as they are, the others still become 0.
// The row loop is unrolled so that a thread's rows are in flight together.
template <int D, int NT = 128>
__device__ __forceinline__ void phi_tile(uint8_t* tile, int astride, int valid, int ct, float* colsum,
                                         bool ident = false) {
    constexpr int CPR = D / 8;
    constexpr int RG = NT / CPR;
    static_assert(RG % 8 == 0, "rows of a thread share one swizzle phase");
    constexpr int RPT = (CH + RG - 1) / RG;
    const int j = ct % CPR, g = ct / CPR;
    uint4* base = reinterpret_cast<uint4*>(tile + (j >> 3) * astride + (((j & 7) ^ (g & 7)) << 4) + g * 128);
    uint64_t cs[4];  // column sums as f32 pairs
    if (colsum) {
#pragma unroll
        for (int e = 0; e < 4; ++e) cs[e] = f2_pack(colsum[2 * e], colsum[2 * e + 1]);
    }
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        if (CH % RG != 0 && g + i * RG >= CH) break;
        uint4 x = base[i * RG * 8];
        uint32_t w[4] = {x.x, x.y, x.z, x.w};
        if (g + i * RG < valid) {
            if (!ident) {
#pragma unroll
                for (int e = 0; e < 4; ++e) w[e] = phi_bf16x2(w[e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = 0u;
        }
        base[i * RG * 8] = make_uint4(w[0], w[1], w[2], w[3]);
        if (colsum) {
#pragma unroll
            for (int e = 0; e < 4; ++e) cs[e] = f2_add(cs[e], f2_pack(bf16lo(w[e]), bf16hi(w[e])));
        }
    }
    if (colsum) {
#pragma unroll
        for (int e = 0; e < 4; ++e) colsum[2 * e] = f2_lo(cs[e]), colsum[2 * e + 1] = f2_hi(cs[e]);
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

}  // namespace la
