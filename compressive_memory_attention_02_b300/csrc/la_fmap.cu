// Positive random-feature map on the tensor cores, bf16 storage, f32 arithmetic:
//     phi(x) = exp(W x - |x|^2 / 2) / sqrt(m)          x [rows, d], W [m, d] -> [rows, m]
// The page "Attention_Kernel_Mask" lists positive and orthogonal random features among the
// feature maps of its non-causal kernel discussion (without printing them); this is the
// positive random-feature map of that family. Orthogonal random features are the same map
// with W's rows orthogonal within blocks of d (the caller builds W). The mapped q and k
// then go through la_causal_fwd_mapped, the same chunked kernels with the map applied.
//
// One block of 128 threads per 128 rows: TMA loads the x tile (two 64-row halves per
// 64-feature block) and W (m rows), one thread issues the tcgen05 MMAs X W^T into TMEM
// (lane = row, column = feature), and each thread finishes its row: |x|^2 from the x tile,
// then exp(acc - |x|^2 / 2) / sqrt(m) rounded to bf16 and stored. Rows past the end are
// zero-filled by TMA and not stored.
#include "la_tc_common.cuh"

namespace la {

template <int D, int MF>
struct FmapLayout {
    static constexpr int XT = 0;                          // x: D/64 blocks of [128 rows][64] (2 atoms)
    static constexpr int WT = XT + D / 64 * 2 * ATOM;     // W: D/64 blocks of [MF rows][64]
    static constexpr int BAR = WT + D / 64 * (MF / 64) * ATOM;
    static constexpr int MISC = BAR + 16;
    static constexpr int ALLOC = MISC + 16 + 1024;
};

template <int D, int MF>
__global__ void __launch_bounds__(128, 1)
    fmap_prf_kernel(const __grid_constant__ CUtensorMap mx, const __grid_constant__ CUtensorMap mw, void* out,
                    int64_t rows, int* status) {
    using L = FmapLayout<D, MF>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint64_t* ld_full = reinterpret_cast<uint64_t*>(sm + L::BAR);
    uint64_t* mma_done = ld_full + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sm + L::MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + L::MISC + 4);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int64_t r0 = (int64_t)blockIdx.x * 128;

    if (tid == 0) {
        mbar_init(ld_full, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mx);
        tma_prefetch_desc(&mw);
    }
    if (warp == 0) {
        tmem_alloc(tmem_holder, MF);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (tid == 0) {
        mbar_expect_tx(ld_full, (128 + MF) * D * 2);
        for (int a = 0; a < D / 64; ++a) {
            for (int hr = 0; hr < 2; ++hr)
                tma_load_4d(sm + L::XT + (2 * a + hr) * ATOM, &mx, ld_full, a * 64, (int)(r0 + 64 * hr), 0, 0);
            for (int hr = 0; hr < MF / 64; ++hr)
                tma_load_4d(sm + L::WT + (a * (MF / 64) + hr) * ATOM, &mw, ld_full, a * 64, 64 * hr, 0, 0);
        }
    }
    bool ok = mbar_wait(ld_full, 0, abort_flag);
    if (!ok) record_timeout(status, abort_flag);
    ok = __syncthreads_and(ok) != 0;
    if (ok && tid == 0) {
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, MF, 0, 0);
        const uint64_t dx = sdesc_sw128(smem_u32(sm + L::XT), 16, 1024);
        const uint64_t dw = sdesc_sw128(smem_u32(sm + L::WT), 16, 1024);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t kb = ks >> 2, kw = (ks & 3) * 32;
            mma_bf16_ss(tmem, dx + ((kb * 2 * ATOM + kw) >> 4), dw + ((kb * (MF / 64) * ATOM + kw) >> 4), id, ks != 0);
        }
        mma_commit(mma_done);
    }
    // |x|^2 of this thread's row from the swizzled tile while the MMAs run
    const int r = tid;
    float n2 = 0.f;
#pragma unroll 4
    for (int c = 0; c < D / 8; ++c) {
        const uint8_t* row = sm + L::XT + ((c >> 3) * 2 + (r >> 6)) * ATOM + (r & 63) * 128;
        const uint4 x = *reinterpret_cast<const uint4*>(row + (((c & 7) ^ (r & 7)) << 4));
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float a = bf16lo(w[e]), b = bf16hi(w[e]);
            n2 += a * a + b * b;
        }
    }
    if (ok) {
        ok = mbar_wait(mma_done, 0, abort_flag);
        if (!ok) record_timeout(status, abort_flag);
    }
    ok = __syncthreads_and(ok) != 0;
    tc_fence_after();
    if (ok) {  // the TMEM loads are warp-wide; only rows inside the input are stored
        const bool store = r0 + r < rows;
        constexpr float kLog2e = 1.4426950408889634f;
        const float scale = 1.f / sqrtf((float)MF);
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out) + (store ? (r0 + r) * MF : 0);
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
#pragma unroll 1
        for (int j0 = 0; j0 < MF; j0 += 16) {
            uint32_t acc[16];
            tmem_ld16(tmem + lane_base + j0, acc);
            tmem_wait_ld();
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float y0 = ex2_approx((__uint_as_float(acc[2 * e]) - 0.5f * n2) * kLog2e) * scale;
                const float y1 = ex2_approx((__uint_as_float(acc[2 * e + 1]) - 0.5f * n2) * kLog2e) * scale;
                w[e] = pack_bf16(y0, y1);
            }
            if (store) {
                *reinterpret_cast<uint4*>(o + j0) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(o + j0 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, MF);
    }
}

template <int D, int MF>
static cudaError_t launch_fmap_t(const CUtensorMap& mx, const CUtensorMap& mw, void* out, int64_t rows, int* status,
                                 cudaStream_t s) {
    using L = FmapLayout<D, MF>;
    auto fn = fmap_prf_kernel<D, MF>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    fn<<<(unsigned)((rows + 127) / 128), 128, L::ALLOC, s>>>(mx, mw, out, rows, status);
    return cudaGetLastError();
}

cudaError_t launch_fmap_prf(const CUtensorMap& mx, const CUtensorMap& mw, void* out, int64_t rows, int d, int m,
                            int* status, cudaStream_t s) {
    if (d == 64 && m == 64) return launch_fmap_t<64, 64>(mx, mw, out, rows, status, s);
    if (d == 64 && m == 128) return launch_fmap_t<64, 128>(mx, mw, out, rows, status, s);
    if (d == 128 && m == 64) return launch_fmap_t<128, 64>(mx, mw, out, rows, status, s);
    if (d == 128 && m == 128) return launch_fmap_t<128, 128>(mx, mw, out, rows, status, s);
    return cudaErrorInvalidValue;
}

}  // namespace la
