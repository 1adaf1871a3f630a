// la_prefill_state_noalloc: the prefill for callers that cannot allocate device
// memory (contract in include/linattn.h). The scratch of the multi-part schedule is a
// file-scope device array of fixed size instead of a caller workspace; everything
// else is la_prefill_state_ex with that array as its workspace.
#include <mutex>

#include "la_internal.h"

namespace la {

// Shared by every call on a device; holds per-part state sums and, when the caller
// asks only for the last output, the final state. Each call writes every byte it
// later reads, so nothing has to be cleared between calls.
static __device__ __align__(256) unsigned char g_noalloc_scratch[LA_NOALLOC_SCRATCH_BYTES];

constexpr int kNoallocMaxDevices = 64;
struct NoallocSlot {
    unsigned long long ctx_id = 0;  // context the address was looked up in
    void* ptr = nullptr;
};
static NoallocSlot g_noalloc[kNoallocMaxDevices];
static std::mutex g_noalloc_mu;

// Device address of g_noalloc_scratch on the current device. In host code the
// array's name only stands in for the symbol, so the address must be looked up
// (once per device and context, with that device current) before a kernel may be
// given it. A new context on the device (after cudaDeviceReset) loads the module
// anew, so the address is looked up again then.
static int noalloc_scratch(void** ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices) return LA_ERR_CUDA;
    unsigned long long ctx = 0;
    if (current_context_id(&ctx) != LA_OK) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocSlot& slot = g_noalloc[dev];
    if (slot.ctx_id != ctx || !slot.ptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return LA_ERR_CUDA;
        slot.ptr = p;
        slot.ctx_id = ctx;
    }
    *ptr = slot.ptr;
    return LA_OK;
}

}  // namespace la

extern "C" int la_prefill_state_noalloc(const void* q, const void* k, const void* v, void* out_last,
                                        const float* M_in, const float* z_in, float* M_out, float* z_out, int B,
                                        int H, int64_t T, int d, int dv, int segment, float eps, la_dtype dtype,
                                        la_stream_t stream) {
    // argument errors are reported by the prefill itself; only the size limit is checked here
    if (!q || !k || !v || B <= 0 || H <= 0 || T <= 0 || segment < 0) return LA_ERR_INVALID_ARG;
    if (!out_last && !M_out && !z_out) return LA_OK;  // nothing requested
    for (const float* st : {M_in, z_in, static_cast<const float*>(M_out), static_cast<const float*>(z_out)})
        if (reinterpret_cast<uintptr_t>(st) & 15u) return LA_ERR_INVALID_ARG;  // as the prefill requires
    const size_t need = la::prefill_scratch_bytes(B, H, T, d, dv, segment, dtype, out_last, M_out, z_out);
    if (need > LA_NOALLOC_SCRATCH_BYTES) return LA_ERR_SCRATCH_LIMIT;
    void* ws = nullptr;
    const int rc = la::noalloc_scratch(&ws);
    if (rc != LA_OK) return rc;
    return la::prefill_impl(q, k, v, out_last, M_in, z_in, M_out, z_out, B, H, T, d, dv, segment, eps, dtype,
                            nullptr, ws, LA_NOALLOC_SCRATCH_BYTES, false, (cudaStream_t)stream);
}
