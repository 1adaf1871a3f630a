// C ABI of the library (declarations and contracts in include/linattn.h):
// argument validation, path selection, tensor-map construction and launches.
// Host code only; every step of the computation runs in the kernels of
// la_simt.cu, la_tc.cu and la_fwd_tc.cu.
#include <cudaTypedefs.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/linattn.h"
#include "la_bwd.h"
#include "la_internal.h"

namespace la {

__device__ int g_status;  // per-device status word (STATUS_* bits), read by la_get_last_device_status

static thread_local int t_launches = 0;

constexpr int kMaxDevices = 64;
constexpr int kSmemLimit = 227 * 1024;

struct DeviceState {
    unsigned long long ctx_id = 0;  // context the cached addresses belong to (0: none yet)
    int* status = nullptr;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    int sm_count = 0;
};
static DeviceState g_dev[kMaxDevices];
static std::mutex g_mu;

// Driver calls reached through the runtime's entry-point query (the library links
// only the runtime).
template <typename F>
static F driver_fn(const char* name, int version) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
        return reinterpret_cast<F>(p);
    return nullptr;
}

int current_context_id(unsigned long long* id) {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        get_current = driver_fn<GetCurrent>("cuCtxGetCurrent", 4000);
        get_id = driver_fn<GetId>("cuCtxGetId", 12000);
    });
    if (!get_current || !get_id) return LA_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return LA_ERR_CUDA;
    if (!ctx) {
        // no context on this thread yet: a runtime call makes the device's primary context
        // current (this cannot happen inside a stream capture, which needs a context)
        if (cudaFree(nullptr) != cudaSuccess || get_current(&ctx) != CUDA_SUCCESS || !ctx) return LA_ERR_CUDA;
    }
    if (get_id(ctx, id) != CUDA_SUCCESS) return LA_ERR_CUDA;
    return LA_OK;
}

// Per-device state, looked up again whenever the current context is not the one the
// cached addresses were taken in (after cudaDeviceReset the module is loaded anew
// and its device variables may live elsewhere; a registered workspace belonged to
// the old context and is dropped).
static int current_device(DeviceState** st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LA_ERR_CUDA;
    unsigned long long ctx = 0;
    if (current_context_id(&ctx) != LA_OK) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& s = g_dev[dev];
    if (s.ctx_id != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return LA_ERR_CUDA;
        s = DeviceState{};
        s.status = static_cast<int*>(p);
        cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev);
        s.ctx_id = ctx;
    }
    *st = &s;
    return LA_OK;
}

int device_status_word(int** status) {
    DeviceState* ds = nullptr;
    const int rc = current_device(&ds);
    if (rc == LA_OK) *status = ds->status;
    return rc;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] { fn = driver_fn<PFN_cuTensorMapEncodeTiled_v12000>("cuTensorMapEncodeTiled", 12000); });
    return fn;
}

// 4-D bf16 map {inner, T, H, B} over a strided [B, H, T, inner] tensor; 64 x 64 boxes,
// 128-byte swizzle (the operand layout the kernels' descriptors assume), zero fill.
// Tiled map of a [B][H][T][inner] bf16 tensor (element strides st, sh, sb): boxes of 64
// features x `rows` tokens, 128-byte swizzle
static bool make_map(CUtensorMap* m, const void* base, int inner, int64_t T, int H, int B, int64_t st, int64_t sh,
                     int64_t sb, int rows = 64) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)T, (cuuint64_t)H, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)st * 2, (cuuint64_t)sh * 2, (cuuint64_t)sb * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)rows, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static int env_int(const char* name, int dflt) {
    const char* s = std::getenv(name);
    return (s && *s) ? std::atoi(s) : dflt;
}

static bool shape_ok(int d, int dv) { return d >= 8 && dv >= 8 && d <= 128 && dv <= 128 && d % 8 == 0 && dv % 8 == 0; }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static Strides contiguous(int H, int64_t T, int d, int dv) {
    Strides s;
    s.q_st = d, s.q_sh = T * d, s.q_sb = (int64_t)H * T * d;
    s.k_st = d, s.k_sh = T * d, s.k_sb = (int64_t)H * T * d;
    s.v_st = dv, s.v_sh = T * dv, s.v_sb = (int64_t)H * T * dv;
    s.o_st = dv, s.o_sh = T * dv, s.o_sb = (int64_t)H * T * dv;
    return s;
}

static Strides from_array(const int64_t* a) {
    Strides s;
    s.q_sb = a[0], s.q_sh = a[1], s.q_st = a[2];
    s.k_sb = a[3], s.k_sh = a[4], s.k_st = a[5];
    s.v_sb = a[6], s.v_sh = a[7], s.v_st = a[8];
    s.o_sb = a[9], s.o_sh = a[10], s.o_st = a[11];
    return s;
}

static bool strides_valid(const Strides& s, int d, int dv, bool with_out) {
    const int64_t v[12] = {s.q_sb, s.q_sh, s.q_st, s.k_sb, s.k_sh, s.k_st,
                           s.v_sb, s.v_sh, s.v_st, s.o_sb, s.o_sh, s.o_st};
    for (int i = 0; i < (with_out ? 12 : 9); ++i)
        if (v[i] < 0) return false;
    return s.q_st >= d && s.k_st >= d && s.v_st >= dv && (!with_out || s.o_st >= dv);
}

static bool strides_tma(const Strides& s, bool with_out) {
    const int64_t v[12] = {s.q_sb, s.q_sh, s.q_st, s.k_sb, s.k_sh, s.k_st,
                           s.v_sb, s.v_sh, s.v_st, s.o_sb, s.o_sh, s.o_st};
    for (int i = 0; i < (with_out ? 12 : 9); ++i)
        if (v[i] % 8 != 0 || v[i] * 2 >= (int64_t(1) << 40)) return false;
    return true;
}

static int cuda_rc(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

// Elements spanned by a strided [B, H, T, inner] tensor.
static int64_t span(int B, int H, int64_t T, int inner, int64_t sb, int64_t sh, int64_t st) {
    return (int64_t)(B - 1) * sb + (int64_t)(H - 1) * sh + (T - 1) * st + inner;
}

// Extents of the caller's buffers for the checked build's device-side bounds checks. In
// that build only, LA_CHECKS_SHRINK=n declares every extent n elements shorter than the
// buffer really is: accesses to the last n elements are then reported (LA_ERR_BOUNDS) and
// skipped, while every access made stays inside the real buffer. It exists to test the
// reporting path without touching memory outside an allocation.
static Extents make_extents(int B, int H, int64_t T, int d, int dv, const Strides& st, int64_t ws_floats) {
    Extents e;
    e.q = span(B, H, T, d, st.q_sb, st.q_sh, st.q_st);
    e.k = span(B, H, T, d, st.k_sb, st.k_sh, st.k_st);
    e.v = span(B, H, T, dv, st.v_sb, st.v_sh, st.v_st);
    e.o = span(B, H, T, dv, st.o_sb, st.o_sh, st.o_st);
    e.M_in = e.M_out = (int64_t)B * H * d * dv;
    e.z_in = e.z_out = (int64_t)B * H * d;
    e.ws = ws_floats;
#if LA_CHECKS
    const int64_t shrink = env_int("LA_CHECKS_SHRINK", 0);
    for (int64_t* x : {&e.q, &e.k, &e.v, &e.o, &e.M_in, &e.z_in, &e.M_out, &e.z_out, &e.ws}) *x -= shrink;
#endif
    return e;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------------ forward
// Schedules of the tensor-core forward (per head, the chunks are split into ranges
// that run on different SMs):
//   single  one range per head (B*H fills the GPU, or no scratch for an aliased state)
//   fused2  two ranges; range 1 forms the state of range 0's chunks itself
//   parts   P > 2 ranges; parts_tc writes the state sum of each range but the last
//           to the workspace, and range r starts from M_in plus those of ranges < r
struct FwdPlan {
    bool tc = false;
    int nranges = 1;
    int chunks_per_range = 0;
    int split = 0;
    int meet = -1;            // fused2 with a hand-off: range 0 publishes its state after this chunk
    size_t ws_bytes = 0;      // scratch that enables the plan (0: none needed)
};

// Scratch of the fused schedule's hand-off: one state record per head, then one word per head.
static size_t pub_bytes(int64_t BH, int d, int dv) {
    const size_t rec = sizeof(float) * ((size_t)d * dv + d) * (size_t)BH;
    return ((rec + 255) / 256) * 256 + ((sizeof(int) * (size_t)BH + 255) / 256) * 256;
}

static FwdPlan plan_fwd(int B, int H, int64_t T, int d, int dv, int chunk, la_dtype dtype, int sm_count,
                        bool aliased, size_t ws_avail) {
    FwdPlan pl;
    // The chunk length only sets the blocking: every chunk length gives the same outputs up
    // to rounding (the chunk equation of mode 3 is the token recurrence regrouped). The
    // tensor-core kernel works in 64-token chunks whatever length is asked for; the SIMT
    // kernel uses the length given.
    (void)chunk;
    const bool tc_shape = (d == 64 || d == 128) && (dv == 64 || dv == 128);
    pl.tc = dtype == LA_BF16 && tc_shape && env_int("LA_FORCE_SIMT", 0) == 0 && T < (int64_t(1) << 31);
    if (!pl.tc) return pl;
    const int64_t nch = ceil_div(T, 64);
    const int64_t BH = (int64_t)B * H;
    const size_t rec_bytes = sizeof(float) * ((size_t)d * dv + d) * (size_t)BH;
    int P = env_int("LA_FWD_RANGES", 0);
    if (P <= 0) P = (int)std::max<int64_t>(1, (sm_count > 0 ? sm_count : 148) / BH);
    P = (int)std::min<int64_t>(P, nch);
    pl.chunks_per_range = (int)nch;
    if (P <= 1) return pl;
    const size_t alias_bytes = aliased ? rec_bytes : 0;   // copy of M_in/z_in read by every range
    if (P > 2) {
        const int64_t cpr = ceil_div(nch, P);
        const int P2 = (int)ceil_div(nch, cpr);
        const size_t need = rec_bytes * (size_t)(P2 - 1) + alias_bytes;
        if (P2 > 2 && ws_avail >= need) {
            pl.nranges = P2;
            pl.chunks_per_range = (int)cpr;
            pl.ws_bytes = need;
            return pl;
        }
        P = 2;
    }
    if (ws_avail < alias_bytes) return pl;
    pl.nranges = 2;
    pl.ws_bytes = alias_bytes;
    // With scratch for the hand-off, range 0 publishes its state after chunk meet and range 1
    // sums only the chunks between meet and the split: range 0 takes a smaller share.
    const size_t pubb = pub_bytes(BH, d, dv);
    // (a cooperative grid cannot start its set-up under the previous kernel, and the hand-off
    // itself costs a few microseconds: it pays only on long sequences)
    const int64_t min_chunks = env_int("LA_FWD_PUB_MIN_CHUNKS", 256);
    if (env_int("LA_FWD_PUBLISH", 1) && nch >= min_chunks && ws_avail >= alias_bytes + pubb) {
        const int pct = env_int("LA_FWD_SPLIT_PCT", d >= 128 ? 60 : 60);
        const int meet_pct = env_int("LA_FWD_MEET_PCT", 33);  // of the split
        int64_t split = (nch * pct + 50) / 100;
        split = std::max<int64_t>(3, std::min<int64_t>(split, nch - 1));
        int64_t meet = (split * meet_pct + 50) / 100 - 1;
        meet = std::max<int64_t>(0, std::min<int64_t>(meet, split - 2));  // range 1 sums at least one chunk
        pl.split = (int)split;
        pl.meet = (int)meet;
        pl.ws_bytes = alias_bytes + pubb;
        return pl;
    }
    // range 0's share of the chunks: range 1 re-forms their state first (measured optimum:
    // 68% at d = 128, 66% at d = 64, where a chunk's fixed costs weigh more)
    const int pct = env_int("LA_FWD_SPLIT_PCT", d >= 128 ? 68 : 66);
    int64_t split = (nch * pct + 50) / 100;
    split = std::max<int64_t>(1, std::min<int64_t>(split, nch - 1));
    pl.split = (int)split;
    return pl;
}

// With M_seg / z_seg (tensor-core path only, the caller checks): the state after every
// segment of seg_chunks 64-token chunks is written too.
static int fwd_impl(const void* q, const void* k, const void* v, void* out, const float* M_in, const float* z_in,
                    float* M_out, float* z_out, int B, int H, int64_t T, int d, int dv, int chunk, float eps,
                    la_dtype dtype, const int64_t* strides, void* ws, size_t ws_bytes, bool use_registered,
                    cudaStream_t stream, bool phi_ident = false, float* M_seg = nullptr, float* z_seg = nullptr,
                    int seg_chunks = 0) {
    t_launches = 0;
    if (!q || !k || !v || !out) return LA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || T <= 0 || !(eps >= 0.f)) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_UNSUPPORTED;
    if (!shape_ok(d, dv)) return LA_ERR_UNSUPPORTED;
    if (chunk != 16 && chunk != 32 && chunk != 64 && chunk != 128) return LA_ERR_UNSUPPORTED;
    if (out == q || out == k || out == v) return LA_ERR_INVALID_ARG;
    if (ws && (reinterpret_cast<uintptr_t>(ws) & 255u)) return LA_ERR_WORKSPACE;
    const Strides st = strides ? from_array(strides) : contiguous(H, T, d, dv);
    if (!strides_valid(st, d, dv, true)) return LA_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    int rc = current_device(&ds);
    if (rc) return rc;
    if (use_registered) ws = ds->ws, ws_bytes = ds->ws_bytes;
    if (!ws) ws_bytes = 0;

    const bool aliased = (M_in && (const void*)M_in == (const void*)M_out) ||
                         (z_in && (const void*)z_in == (const void*)z_out);
    FwdPlan pl = plan_fwd(B, H, T, d, dv, chunk, dtype, ds->sm_count, aliased, ws_bytes);
    if (pl.tc && !(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out) && strides_tma(st, true)))
        pl.tc = false;
    if (pl.tc) {
        CUtensorMap mq, mk, mv, mo;
        if (!make_map(&mq, q, d, T, H, B, st.q_st, st.q_sh, st.q_sb) ||
            !make_map(&mk, k, d, T, H, B, st.k_st, st.k_sh, st.k_sb) ||
            !make_map(&mv, v, dv, T, H, B, st.v_st, st.v_sh, st.v_sb) ||
            !make_map(&mo, out, dv, T, H, B, st.o_st, st.o_sh, st.o_sb))
            return LA_ERR_CUDA;
        const int64_t BH = (int64_t)B * H;
        const int64_t rec = (int64_t)d * dv + d;
        float* wsf = static_cast<float*>(ws);
        const float* Mi = M_in;
        const float* zi = z_in;
        if (pl.nranges > 1 && aliased) {
            // every range reads the initial state while the last one writes the final
            // state in place: read the initial state from a copy
            float* base = wsf + (pl.nranges > 2 ? (size_t)BH * (pl.nranges - 1) * rec : 0);
            if (M_in && (const void*)M_in == (const void*)M_out) {
                if (cudaMemcpyAsync(base, M_in, sizeof(float) * BH * d * dv, cudaMemcpyDeviceToDevice, stream))
                    return LA_ERR_CUDA;
                Mi = base;
            }
            if (z_in && (const void*)z_in == (const void*)z_out) {
                if (cudaMemcpyAsync(base + BH * d * dv, z_in, sizeof(float) * BH * d, cudaMemcpyDeviceToDevice,
                                    stream))
                    return LA_ERR_CUDA;
                zi = base + BH * d * dv;
            }
        }
        if (pl.nranges > 2) {
            PartsParams pp{};
            pp.k = k, pp.v = v, pp.dst_M = wsf, pp.dst_z = wsf + (size_t)d * dv;
            pp.rec_M = rec, pp.rec_z = rec;
            pp.B = B, pp.H = H, pp.T = T, pp.d = d, pp.dv = dv;
            pp.part_len = (int64_t)pl.chunks_per_range * 64;
            pp.nparts = pl.nranges - 1;
            pp.eps = eps, pp.st = st, pp.status = ds->status, pp.phi_ident = phi_ident;
            rc = cuda_rc(launch_parts_tc(pp, mk, mv, stream));
            if (rc) return rc;
            ++t_launches;
        }
        FwdTcParams fp{};
        fp.phi_ident = phi_ident;
        fp.M_in = Mi, fp.z_in = zi, fp.M_out = M_out, fp.z_out = z_out;
        fp.ws = pl.nranges > 2 ? wsf : nullptr;
        fp.rec = rec, fp.nranges = pl.nranges, fp.chunks_per_range = pl.chunks_per_range, fp.split = pl.split;
        fp.H = H, fp.T = T, fp.eps = eps, fp.status = ds->status;
        fp.M_seg = M_seg, fp.z_seg = z_seg, fp.seg_chunks = seg_chunks;
        if (pl.meet >= 0) {  // the hand-off area follows the aliased-state copy, if any
            const size_t alias_floats = aliased ? (size_t)BH * rec : 0;
            fp.pub = wsf + alias_floats;
            fp.pub_flag = reinterpret_cast<int*>(reinterpret_cast<char*>(fp.pub) +
                                                 ((sizeof(float) * (size_t)BH * rec + 255) / 256) * 256);
            fp.meet = pl.meet;
        }
        // at d = dv = 64 the fused schedule's state-only chunks stream two at a time (128-token boxes)
        CUtensorMap mk2 = mk, mv2 = mv;
        if (pl.split > 0 && d == 64 && dv == 64 &&
            !(make_map(&mk2, k, d, T, H, B, st.k_st, st.k_sh, st.k_sb, 128) &&
                              make_map(&mv2, v, dv, T, H, B, st.v_st, st.v_sh, st.v_sb, 128)))
            return LA_ERR_CUDA;
        rc = cuda_rc(launch_fwd_tc(fp, d, dv, B, mq, mk, mv, mo, mk2, mv2, stream));
        if (!rc) ++t_launches;
        return rc;
    }
    if (M_seg || z_seg) return LA_ERR_UNSUPPORTED;  // (the caller runs such cases segment by segment)
    if (fwd_simt_smem(d, dv, chunk) > (size_t)kSmemLimit) return LA_ERR_UNSUPPORTED;
    FwdParams p{};
    p.q = q, p.k = k, p.v = v, p.out = out, p.M_in = M_in, p.z_in = z_in, p.M_out = M_out, p.z_out = z_out;
    p.B = B, p.H = H, p.T = T, p.d = d, p.dv = dv, p.chunk = chunk, p.eps = eps, p.st = st;
    p.ext = make_extents(B, H, T, d, dv, st, 0), p.status = ds->status, p.phi_ident = phi_ident;
    rc = cuda_rc(launch_fwd_simt(p, dtype == LA_BF16, stream));
    if (!rc) ++t_launches;
    return rc;
}

// ------------------------------------------------------------------ prefill
struct PrefillPlan {
    bool tc = false;
    int64_t part_len = 0;
    int nparts = 1;
    size_t parts_bytes = 0;   // per-part records
    size_t final_bytes = 0;   // final state when M_out / z_out are not given
};

static bool aligned16_or_null(const void* p) { return !p || aligned16(p); }

static PrefillPlan plan_prefill(int B, int H, int64_t T, int d, int dv, int segment, la_dtype dtype) {
    PrefillPlan pl;
    const int64_t BH = (int64_t)B * H;
    const size_t rec = (size_t)d * dv + d;
    int64_t seg = segment > 0 ? segment : 4096;
    pl.tc = dtype == LA_BF16 && (d == 64 || d == 128) && (dv == 64 || dv == 128) && seg % 64 == 0 &&
            env_int("LA_FORCE_SIMT", 0) == 0 && T < (int64_t(1) << 31);
    pl.part_len = std::min<int64_t>(seg, T);
    pl.nparts = (int)ceil_div(T, pl.part_len);
    pl.parts_bytes = pl.nparts > 1 ? sizeof(float) * rec * BH * pl.nparts : 0;
    pl.final_bytes = sizeof(float) * rec * BH;
    return pl;
}

size_t prefill_scratch_bytes(int B, int H, int64_t T, int d, int dv, int segment, la_dtype dtype,
                             const void* out_last, const float* M_out, const float* z_out) {
    if (!out_last && !M_out && !z_out) return 0;  // nothing requested: the call returns at once
    const PrefillPlan pl = plan_prefill(B, H, T, d, dv, segment, dtype);
    const bool need_final = out_last && (!M_out || !z_out);
    return pl.parts_bytes + (need_final ? pl.final_bytes : 0);
}

int prefill_impl(const void* q, const void* k, const void* v, void* out_last, const float* M_in,
                        const float* z_in, float* M_out, float* z_out, int B, int H, int64_t T, int d, int dv,
                        int segment, float eps, la_dtype dtype, const int64_t* strides, void* ws, size_t ws_bytes,
                        bool use_registered, cudaStream_t stream) {
    t_launches = 0;
    if (!q || !k || !v) return LA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || T <= 0 || segment < 0 || !(eps >= 0.f)) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_UNSUPPORTED;
    if (!shape_ok(d, dv)) return LA_ERR_UNSUPPORTED;
    // the ordered reduce of the parts moves the state in 16-byte vectors
    if (!aligned16_or_null(M_in) || !aligned16_or_null(z_in) || !aligned16_or_null(M_out) ||
        !aligned16_or_null(z_out))
        return LA_ERR_INVALID_ARG;
    if (ws && (reinterpret_cast<uintptr_t>(ws) & 255u)) return LA_ERR_WORKSPACE;
    Strides st = strides ? from_array(strides) : contiguous(H, T, d, dv);
    if (!strides_valid(st, d, dv, false)) return LA_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    int rc = current_device(&ds);
    if (rc) return rc;
    if (use_registered) ws = ds->ws, ws_bytes = ds->ws_bytes;
    if (!out_last && !M_out && !z_out) return LA_OK;  // nothing requested

    const int64_t BH = (int64_t)B * H;
    const int64_t rec = (int64_t)d * dv + d;
    PrefillPlan pl = plan_prefill(B, H, T, d, dv, segment, dtype);
    if (pl.tc && !(aligned16(k) && aligned16(v) && strides_tma(st, false))) pl.tc = false;
    const bool need_final = out_last && (!M_out || !z_out);
    const size_t need = prefill_scratch_bytes(B, H, T, d, dv, segment, dtype, out_last, M_out, z_out);
    if (ws_bytes < need || !ws) {
        // no (or too little) scratch: one part per head, state straight into M_out/z_out
        pl.nparts = 1;
        pl.part_len = T;
        pl.parts_bytes = 0;
    }
    float* wsf = static_cast<float*>(ws);
    const bool have_final_ws = need_final && ws && ws_bytes >= pl.parts_bytes + pl.final_bytes;
    // where the final state goes
    float* fM = M_out;
    float* fz = z_out;
    if (need_final && have_final_ws) {
        float* fin = wsf + pl.parts_bytes / sizeof(float);
        if (!fM) fM = fin;
        if (!fz) fz = fin + BH * d * dv;
    }
    const bool bf16 = dtype == LA_BF16;
    // extents for the checked build: out_last is [B, H, dv]; the part records (when T is
    // split) are BH * nparts records of rec floats from wsf
    Extents ext = make_extents(B, H, T, d, dv, st, pl.nparts > 1 ? BH * pl.nparts * rec : 0);
    ext.o = BH * dv;
#if LA_CHECKS
    ext.o -= env_int("LA_CHECKS_SHRINK", 0);
#endif

    if (need_final && (!fM || !fz)) {
        // no place for a final state: the SIMT kernel keeps it on chip and reads out itself
        if (parts_simt_smem(d, dv) > (size_t)kSmemLimit) return LA_ERR_UNSUPPORTED;
        PartsParams pp{};
        pp.q = q, pp.k = k, pp.v = v, pp.out_last = out_last, pp.base_M = M_in, pp.base_z = z_in;
        pp.dst_M = M_out, pp.dst_z = z_out, pp.rec_M = (int64_t)d * dv, pp.rec_z = d;
        pp.B = B, pp.H = H, pp.T = T, pp.d = d, pp.dv = dv, pp.part_len = T, pp.nparts = 1;
        pp.eps = eps, pp.st = st, pp.status = ds->status;
        pp.ext = ext;
        rc = cuda_rc(launch_parts_simt(pp, bf16, stream));
        if (!rc) ++t_launches;
        return rc;
    }

    CUtensorMap mk, mv;
    if (pl.tc && (!make_map(&mk, k, d, T, H, B, st.k_st, st.k_sh, st.k_sb) ||
                  !make_map(&mv, v, dv, T, H, B, st.v_st, st.v_sh, st.v_sb)))
        return LA_ERR_CUDA;

    PartsParams pp{};
    pp.q = q, pp.k = k, pp.v = v;
    pp.B = B, pp.H = H, pp.T = T, pp.d = d, pp.dv = dv, pp.part_len = pl.part_len, pp.nparts = pl.nparts;
    pp.eps = eps, pp.st = st, pp.status = ds->status;
    pp.ext = ext;
    if (pl.nparts == 1) {
        pp.base_M = M_in, pp.base_z = z_in;
        pp.dst_M = fM, pp.dst_z = fz, pp.rec_M = (int64_t)d * dv, pp.rec_z = d;
    } else {
        pp.dst_M = wsf, pp.dst_z = wsf + (size_t)d * dv, pp.rec_M = rec, pp.rec_z = rec;
        pp.ext.M_out = ext.ws, pp.ext.z_out = ext.ws - (int64_t)d * dv;  // the record array
    }
    if (pl.tc) {
        if (!pp.dst_M || !pp.dst_z) {
            // the tensor-core kernel writes both halves of the state; route a missing one to scratch
            if (!have_final_ws) {
                if (parts_simt_smem(d, dv) > (size_t)kSmemLimit) return LA_ERR_UNSUPPORTED;
                pl.tc = false;
            } else {
                float* fin = wsf + pl.parts_bytes / sizeof(float);
                if (!pp.dst_M) pp.dst_M = fin, fM = fin;
                if (!pp.dst_z) pp.dst_z = fin + BH * d * dv, fz = fin + BH * d * dv;
            }
        }
    }
    if (pl.tc) {
        rc = cuda_rc(launch_parts_tc(pp, mk, mv, stream));
    } else {
        if (parts_simt_smem(d, dv) > (size_t)kSmemLimit) return LA_ERR_UNSUPPORTED;
        rc = cuda_rc(launch_parts_simt(pp, bf16, stream));
    }
    if (rc) return rc;
    ++t_launches;
    if (pl.nparts > 1 && (fM || fz)) {
        ReduceParams rp{};
        rp.base_M = M_in, rp.base_z = z_in, rp.parts_M = wsf, rp.parts_z = wsf + (size_t)d * dv;
        rp.rec_M = rec, rp.rec_z = rec, rp.dst_M = fM, rp.dst_z = fz;
        rp.BH = (int)BH, rp.d = d, rp.dv = dv, rp.nparts = pl.nparts;
        rp.ext = ext, rp.status = ds->status;
        if (!fM || !fz) return LA_ERR_INVALID_ARG;  // unreachable: both set when parts > 1
        rc = cuda_rc(launch_reduce_parts(rp, stream));
        if (rc) return rc;
        ++t_launches;
    }
    if (out_last) {
        PrefillOutParams op{};
        op.q = q, op.out = out_last, op.M = fM, op.z = fz, op.B = B, op.H = H, op.T = T, op.d = d, op.dv = dv;
        op.eps = eps, op.st = st, op.ext = ext, op.status = ds->status;
        rc = cuda_rc(launch_prefill_out(op, bf16, stream));
        if (rc) return rc;
        ++t_launches;
    }
    return LA_OK;
}

// Training backward behind la_causal_bwd / la_causal_bwd_ex: six launches on `stream`
// (la_bwd.cu), scratch from the registered workspace (use_registered) or (ws, ws_bytes).
static int bwd_impl(const void* q, const void* k, const void* v, const void* dout, const float* M_in,
                    const float* z_in, const float* dM_out, const float* dz_out, void* dq, void* dk, void* dv,
                    float* dM_in, float* dz_in, int B, int H, int64_t T, int d, int dv_dim, float eps,
                    la_dtype dtype, void* ws, size_t ws_bytes, bool use_registered, cudaStream_t stream) {
    t_launches = 0;
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return LA_ERR_INVALID_ARG;
    if (B <= 0 || H <= 0 || T <= 0 || !(eps >= 0.f)) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_UNSUPPORTED;
    if (!shape_ok(d, dv_dim)) return LA_ERR_UNSUPPORTED;
    const int64_t BH = (int64_t)B * H;
    const int64_t nch = ceil_div(T, BWD_CH);
    if (BH > 65535 || nch > 0x7fffffff) return LA_ERR_UNSUPPORTED;
    const void* ins[4] = {q, k, v, dout};
    void* outs[3] = {dq, dk, dv};
    for (void* o : outs)
        for (const void* i : ins)
            if (o == i) return LA_ERR_INVALID_ARG;
    if (dq == dk || dq == dv || dk == dv) return LA_ERR_INVALID_ARG;
    for (const void* a : ins)  // read as 16-byte vectors
        if (!aligned16(a)) return LA_ERR_INVALID_ARG;
    if (ws && (reinterpret_cast<uintptr_t>(ws) & 255u)) return LA_ERR_WORKSPACE;
    DeviceState* ds = nullptr;
    int rc = current_device(&ds);
    if (rc) return rc;
    if (use_registered) ws = ds->ws, ws_bytes = ds->ws_bytes;
    size_t off_rev = 0, off_G = 0, off_E = 0;
    const size_t need = sizeof(float) * bwd_workspace_floats(BH, T, d, dv_dim, &off_rev, &off_G, &off_E);
    if (!ws || ws_bytes < need) return LA_ERR_WORKSPACE;
    float* wsf = static_cast<float*>(ws);
    const int64_t rec = (int64_t)d * dv_dim + d;
    const bool bf16 = dtype == LA_BF16;

    const bool tc = bf16 && (d == 64 || d == 128) && (dv_dim == 64 || dv_dim == 128) &&
                    env_int("LA_FORCE_SIMT", 0) == 0 && T < (int64_t(1) << 31) && aligned16(dq) &&
                    aligned16(dk) && aligned16(dv);  // the gradients are stored in 16-byte vectors
    if (tc) {
        // tensor-core sweeps over ranges of 64-token chunks: the key-value sum of each range
        // (parts_tc), the dq sweep (with D_t, e_t and each range's sums of the state
        // gradient), then the dk/dv sweep
        const Strides st = contiguous(H, T, d, dv_dim);
        CUtensorMap mq, mk, mv, mdo;
        if (!make_map(&mq, q, d, T, H, B, st.q_st, st.q_sh, st.q_sb) ||
            !make_map(&mk, k, d, T, H, B, st.k_st, st.k_sh, st.k_sb) ||
            !make_map(&mv, v, dv_dim, T, H, B, st.v_st, st.v_sh, st.v_sb) ||
            !make_map(&mdo, dout, dv_dim, T, H, B, st.v_st, st.v_sh, st.v_sb))
            return LA_ERR_CUDA;
        // ranges: the fewest waves of blocks x chunks per block (plus one chunk's worth of
        // setup per block), ties to longer ranges
        int dev = 0, sms = 148;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t slots = (int64_t)sms * bwd_sweep_occupancy(d, dv_dim);
        int64_t cpr = nch, best = -1;
        const int64_t forced = env_int("LA_BWD_CPR", 0);
        if (forced > 0) {
            cpr = forced < nch ? forced : nch;
        } else {
            // by number of ranges per head: beyond a few waves of blocks more ranges only add
            // waves, so the search stops at 4 x slots ranges
            const int64_t max_nr = std::min<int64_t>(nch, 4 * slots);
            for (int64_t nr_c = 1; nr_c <= max_nr; ++nr_c) {
                const int64_t c = ceil_div(nch, nr_c);
                const int64_t cost = ceil_div(BH * ceil_div(nch, c), slots) * (c + 1);
                if (best < 0 || cost < best || (cost == best && c > cpr)) best = cost, cpr = c;
            }
        }
        const int64_t nr = ceil_div(nch, cpr);
        // up to BWD_FOLD_RANGES ranges per head each block adds up the records before (after)
        // its range itself; beyond that ordered scans over the ranges do it once, in place
        const bool folded = nr <= BWD_FOLD_RANGES;
        const int64_t nparts = folded ? nr - 1 : nr;  // a folded plan never reads the last range's sum
        if (nparts > 0) {
            PartsParams pp{};
            pp.k = k, pp.v = v, pp.dst_M = wsf, pp.dst_z = wsf + (size_t)d * dv_dim, pp.rec_M = rec, pp.rec_z = rec;
            pp.B = B, pp.H = H, pp.T = T, pp.d = d, pp.dv = dv_dim, pp.part_len = cpr * BWD_CH,
            pp.nparts = (int)nparts;
            pp.eps = eps, pp.st = st, pp.status = ds->status;
            if ((rc = cuda_rc(launch_parts_tc(pp, mk, mv, stream)))) return rc;
            ++t_launches;
        }
        if (!folded) {
            ScanParams sp{};
            sp.rec = wsf, sp.base_M = M_in, sp.base_z = z_in, sp.BH = (int)BH, sp.nch = (int)nr;
            sp.d = d, sp.dv = dv_dim, sp.len = rec, sp.reverse = false;
            if ((rc = cuda_rc(launch_scan_states(sp, stream)))) return rc;
            ++t_launches;
        }
        BwdTcParams tp{};
        tp.dq = dq, tp.dk = dk, tp.dv = dv, tp.states = wsf, tp.rev = wsf + off_rev;
        if (folded)
            tp.M_in = M_in, tp.z_in = z_in, tp.dM_out = dM_out, tp.dz_out = dz_out, tp.dM_in = dM_in, tp.dz_in = dz_in;
        tp.Dn = wsf + off_G, tp.E = wsf + off_E;  // D_t in the (here unused) G region
        tp.B = B, tp.H = H, tp.T = T, tp.d = d, tp.dv_dim = dv_dim, tp.nch = (int)nch;
        tp.nr = (int)nr, tp.cpr = (int)cpr, tp.scanned = !folded, tp.rec = rec, tp.eps = eps, tp.status = ds->status;
        if ((rc = cuda_rc(launch_bwd_dq_tc(tp, mq, mk, mv, mdo, stream)))) return rc;
        ++t_launches;
        if (!folded) {
            ScanParams rp{};
            rp.rec = wsf + off_rev, rp.base_M = dM_out, rp.base_z = dz_out, rp.total_M = dM_in, rp.total_z = dz_in;
            rp.BH = (int)BH, rp.nch = (int)nr, rp.d = d, rp.dv = dv_dim, rp.len = rec, rp.reverse = true;
            if ((rc = cuda_rc(launch_scan_states(rp, stream)))) return rc;
            ++t_launches;
        }
        if ((rc = cuda_rc(launch_bwd_dkdv_tc(tp, mq, mk, mv, mdo, stream)))) return rc;
        ++t_launches;
        return LA_OK;
    }

    BwdParams bp{};
    bp.q = q, bp.k = k, bp.v = v, bp.dout = dout, bp.dq = dq, bp.dk = dk, bp.dv = dv;
    bp.states = wsf, bp.rev = wsf + off_rev, bp.G = wsf + off_G, bp.E = wsf + off_E;
    bp.B = B, bp.H = H, bp.T = T, bp.d = d, bp.dv_dim = dv_dim, bp.nch = (int)nch, bp.rec = rec, bp.eps = eps;
    if ((rc = cuda_rc(launch_bwd_sums(bp, bf16, stream)))) return rc;  // 64-token key-value sums
    ++t_launches;

    ScanParams sp{};  // states before each chunk
    sp.rec = wsf, sp.base_M = M_in, sp.base_z = z_in, sp.BH = (int)BH, sp.nch = (int)nch;
    sp.d = d, sp.dv = dv_dim, sp.len = rec, sp.reverse = false;
    if ((rc = cuda_rc(launch_scan_states(sp, stream)))) return rc;
    ++t_launches;

    if ((rc = cuda_rc(launch_bwd_dq(bp, bf16, stream)))) return rc;
    ++t_launches;

    ScanParams rp{};  // state gradient from every token after each chunk; totals = dM_in, dz_in
    rp.rec = wsf + off_rev, rp.base_M = dM_out, rp.base_z = dz_out, rp.total_M = dM_in, rp.total_z = dz_in;
    rp.BH = (int)BH, rp.nch = (int)nch, rp.d = d, rp.dv = dv_dim, rp.len = rec, rp.reverse = true;
    if ((rc = cuda_rc(launch_scan_states(rp, stream)))) return rc;
    ++t_launches;

    if ((rc = cuda_rc(launch_bwd_dk(bp, bf16, stream)))) return rc;
    ++t_launches;
    if ((rc = cuda_rc(launch_bwd_dv(bp, bf16, stream)))) return rc;
    ++t_launches;
    return LA_OK;
}

}  // namespace la

using namespace la;

extern "C" {

int la_causal_fwd(const void* q, const void* k, const void* v, void* out, const float* M_in, const float* z_in,
                  float* M_out, float* z_out, int B, int H, int64_t T, int d, int dv, int chunk, float eps,
                  la_dtype dtype, la_stream_t stream) {
    return fwd_impl(q, k, v, out, M_in, z_in, M_out, z_out, B, H, T, d, dv, chunk, eps, dtype, nullptr, nullptr, 0,
                    true, (cudaStream_t)stream);
}

int la_causal_fwd_ex(const void* q, const void* k, const void* v, void* out, const float* M_in, const float* z_in,
                     float* M_out, float* z_out, int B, int H, int64_t T, int d, int dv, int chunk, float eps,
                     la_dtype dtype, const int64_t* strides, void* workspace, size_t workspace_bytes,
                     la_stream_t stream) {
    return fwd_impl(q, k, v, out, M_in, z_in, M_out, z_out, B, H, T, d, dv, chunk, eps, dtype, strides, workspace,
                    workspace_bytes, false, (cudaStream_t)stream);
}

int la_causal_fwd_mapped(const void* q, const void* k, const void* v, void* out, const float* M_in,
                         const float* z_in, float* M_out, float* z_out, int B, int H, int64_t T, int d, int dv,
                         int chunk, float eps, la_dtype dtype, const int64_t* strides, void* workspace,
                         size_t workspace_bytes, la_stream_t stream) {
    return fwd_impl(q, k, v, out, M_in, z_in, M_out, z_out, B, H, T, d, dv, chunk, eps, dtype, strides, workspace,
                    workspace_bytes, false, (cudaStream_t)stream, true);
}

static bool overlap(const void* a, size_t an, const void* b, size_t bn) {
    if (!a || !b) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bn && y < x + an;
}

int la_causal_fwd_segments(const void* q, const void* k, const void* v, void* out, const float* M_in,
                           const float* z_in, float* M_seg, float* z_seg, int B, int H, int64_t T, int d, int dv,
                           int64_t seg_len, float eps, la_dtype dtype, void* workspace, size_t workspace_bytes,
                           la_stream_t stream) {
    t_launches = 0;
    if (!M_seg || !z_seg || B <= 0 || H <= 0 || T <= 0 || seg_len <= 0 || seg_len % 64 != 0)
        return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_UNSUPPORTED;
    if (!shape_ok(d, dv)) return LA_ERR_UNSUPPORTED;
    const int64_t BH = (int64_t)B * H, nseg = ceil_div(T, seg_len);
    const size_t m_bytes = sizeof(float) * (size_t)(BH * d * dv), z_bytes = sizeof(float) * (size_t)(BH * d);
    // the outputs may overlap neither each other nor the initial state, which every range reads
    if (overlap(M_seg, m_bytes * nseg, z_seg, z_bytes * nseg) || overlap(M_seg, m_bytes * nseg, M_in, m_bytes) ||
        overlap(M_seg, m_bytes * nseg, z_in, z_bytes) || overlap(z_seg, z_bytes * nseg, M_in, m_bytes) ||
        overlap(z_seg, z_bytes * nseg, z_in, z_bytes))
        return LA_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    const bool tc = dtype == LA_BF16 && (d == 64 || d == 128) && (dv == 64 || dv == 128) &&
                    env_int("LA_FORCE_SIMT", 0) == 0 && T < (int64_t(1) << 31) && aligned16(q) && aligned16(k) &&
                    aligned16(v) && aligned16(out);
    if (tc)  // one launch: the state stays on chip across segment boundaries and is written at each
        return fwd_impl(q, k, v, out, M_in, z_in, nullptr, nullptr, B, H, T, d, dv, 64, eps, dtype, nullptr,
                        workspace, workspace_bytes, false, s, false, M_seg, z_seg, (int)(seg_len / 64));
    // other shapes and float32: one call per segment, each starting from the state the previous
    // one wrote (strided views of the [B,H,T,*] tensors)
    const size_t es = dtype == LA_BF16 ? 2 : 4;
    const int64_t st[12] = {(int64_t)H * T * d, T * d, d, (int64_t)H * T * d, T * d, d,
                            (int64_t)H * T * dv, T * dv, dv, (int64_t)H * T * dv, T * dv, dv};
    int launches = 0;
    for (int64_t sg = 0; sg < nseg; ++sg) {
        const int64_t t0 = sg * seg_len, Ts = std::min<int64_t>(seg_len, T - t0);
        const float* Mi = sg == 0 ? M_in : M_seg + (sg - 1) * BH * d * dv;
        const float* zi = sg == 0 ? z_in : z_seg + (sg - 1) * BH * d;
        const int rc = fwd_impl(static_cast<const char*>(q) + t0 * d * es, static_cast<const char*>(k) + t0 * d * es,
                                static_cast<const char*>(v) + t0 * dv * es, static_cast<char*>(out) + t0 * dv * es,
                                Mi, zi, M_seg + sg * BH * d * dv, z_seg + sg * BH * d, B, H, Ts, d, dv, 64, eps,
                                dtype, st, workspace, workspace_bytes, false, s);
        launches += t_launches;
        if (rc) {
            t_launches = launches;
            return rc;
        }
    }
    t_launches = launches;
    return LA_OK;
}

int la_feature_map_prf(const void* x, const void* W, void* out, int64_t rows, int d, int m, la_dtype dtype,
                       la_stream_t stream) {
    t_launches = 0;
    if (!x || !W || !out || rows <= 0) return LA_ERR_INVALID_ARG;
    if (dtype != LA_BF16 || (d != 64 && d != 128) || (m != 64 && m != 128)) return LA_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(W) || !aligned16(out)) return LA_ERR_INVALID_ARG;
    if (out == x || out == W) return LA_ERR_INVALID_ARG;
    if (rows >= (int64_t(1) << 31)) return LA_ERR_UNSUPPORTED;
    DeviceState* ds = nullptr;
    int rc = current_device(&ds);
    if (rc) return rc;
    CUtensorMap mx, mw;
    if (!make_map(&mx, x, d, rows, 1, 1, d, rows * d, rows * d) || !make_map(&mw, W, d, m, 1, 1, d, (int64_t)m * d,
                                                                           (int64_t)m * d))
        return LA_ERR_CUDA;
    rc = cuda_rc(launch_fmap_prf(mx, mw, out, rows, d, m, ds->status, (cudaStream_t)stream));
    if (!rc) ++t_launches;
    return rc;
}

size_t la_causal_fwd_workspace_size(int B, int H, int64_t T, int d, int dv, int chunk, la_dtype dtype) {
    if (B <= 0 || H <= 0 || T <= 0 || !shape_ok(d, dv)) return 0;
    int sm = 148;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, dev);
    // the largest scratch any plan for this shape may use (an in-place state included); a
    // two-range plan counts the state hand-off of long sequences at every T, so that the
    // size does not depend on T
    const FwdPlan pl = plan_fwd(B, H, T, d, dv, chunk, dtype, sm, true, SIZE_MAX);
    if (pl.nranges == 2 && pl.meet < 0) return pl.ws_bytes + pub_bytes((int64_t)B * H, d, dv);
    return pl.ws_bytes;
}

int la_prefill_state(const void* q, const void* k, const void* v, void* out_last, const float* M_in,
                     const float* z_in, float* M_out, float* z_out, int B, int H, int64_t T, int d, int dv,
                     int segment, float eps, la_dtype dtype, la_stream_t stream) {
    return prefill_impl(q, k, v, out_last, M_in, z_in, M_out, z_out, B, H, T, d, dv, segment, eps, dtype, nullptr,
                        nullptr, 0, true, (cudaStream_t)stream);
}

int la_prefill_state_ex(const void* q, const void* k, const void* v, void* out_last, const float* M_in,
                        const float* z_in, float* M_out, float* z_out, int B, int H, int64_t T, int d, int dv,
                        int segment, float eps, la_dtype dtype, const int64_t* strides, void* workspace,
                        size_t workspace_bytes, la_stream_t stream) {
    return prefill_impl(q, k, v, out_last, M_in, z_in, M_out, z_out, B, H, T, d, dv, segment, eps, dtype, strides,
                        workspace, workspace_bytes, false, (cudaStream_t)stream);
}

size_t la_prefill_workspace_size(int B, int H, int64_t T, int d, int dv, int segment, la_dtype dtype) {
    if (B <= 0 || H <= 0 || T <= 0 || !shape_ok(d, dv) || segment < 0) return 0;
    PrefillPlan pl = plan_prefill(B, H, T, d, dv, segment, dtype);
    return pl.parts_bytes + pl.final_bytes;
}

int la_decode_step(const void* q, const void* k, const void* v, void* out, float* M, float* z, int N, int H, int d,
                   int dv, float eps, la_dtype dtype, la_stream_t stream) {
    t_launches = 0;
    if (!q || !k || !v || !out || !M || !z) return LA_ERR_INVALID_ARG;
    if (N <= 0 || H <= 0 || !(eps >= 0.f)) return LA_ERR_INVALID_ARG;
    if (dtype != LA_F32 && dtype != LA_BF16) return LA_ERR_UNSUPPORTED;
    if (!shape_ok(d, dv)) return LA_ERR_UNSUPPORTED;
    if (!aligned16(M)) return LA_ERR_INVALID_ARG;
    if (out == q || out == k || out == v) return LA_ERR_INVALID_ARG;
    DeviceState* ds = nullptr;
    int rc = current_device(&ds);
    if (rc) return rc;
    DecodeParams p{};
    p.q = q, p.k = k, p.v = v, p.out = out, p.M = M, p.z = z, p.N = N, p.H = H, p.d = d, p.dv = dv, p.eps = eps;
    // extents: one token per (stream, head); the state [N, H, d, dv] and [N, H, d]
    p.ext = make_extents(N, H, 1, d, dv, contiguous(H, 1, d, dv), 0), p.status = ds->status;
    rc = cuda_rc(launch_decode(p, dtype == LA_BF16, (cudaStream_t)stream));
    if (!rc) ++t_launches;
    return rc;
}

int la_causal_bwd(const void* q, const void* k, const void* v, const void* dout, const float* M_in, const float* z_in,
                  const float* dM_out, const float* dz_out, void* dq, void* dk, void* dv, float* dM_in, float* dz_in,
                  int B, int H, int64_t T, int d, int dv_dim, float eps, la_dtype dtype, la_stream_t stream) {
    return bwd_impl(q, k, v, dout, M_in, z_in, dM_out, dz_out, dq, dk, dv, dM_in, dz_in, B, H, T, d, dv_dim, eps,
                    dtype, nullptr, 0, true, (cudaStream_t)stream);
}

int la_causal_bwd_ex(const void* q, const void* k, const void* v, const void* dout, const float* M_in,
                     const float* z_in, const float* dM_out, const float* dz_out, void* dq, void* dk, void* dv,
                     float* dM_in, float* dz_in, int B, int H, int64_t T, int d, int dv_dim, float eps, la_dtype dtype,
                     void* workspace, size_t workspace_bytes, la_stream_t stream) {
    return bwd_impl(q, k, v, dout, M_in, z_in, dM_out, dz_out, dq, dk, dv, dM_in, dz_in, B, H, T, d, dv_dim, eps,
                    dtype, workspace, workspace_bytes, false, (cudaStream_t)stream);
}

size_t la_causal_bwd_workspace_size(int B, int H, int64_t T, int d, int dv) {
    if (B <= 0 || H <= 0 || T <= 0 || !shape_ok(d, dv)) return 0;
    size_t a = 0, b = 0, c = 0;
    return sizeof(float) * bwd_workspace_floats((int64_t)B * H, T, d, dv, &a, &b, &c);
}

int la_set_workspace(void* ptr, size_t bytes) {
    if (ptr && (reinterpret_cast<uintptr_t>(ptr) & 255u)) return LA_ERR_WORKSPACE;
    DeviceState* ds = nullptr;
    int rc = current_device(&ds);
    if (rc) return rc;
    std::lock_guard<std::mutex> lock(g_mu);
    ds->ws = ptr;
    ds->ws_bytes = ptr ? bytes : 0;
    return LA_OK;
}

int la_get_last_device_status(la_stream_t stream) {
    DeviceState* ds = nullptr;
    int rc = current_device(&ds);
    if (rc) return rc;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, ds->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return LA_ERR_CUDA;
    if (v) {
        const int zero = 0;
        if (cudaMemcpy(ds->status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return LA_ERR_CUDA;
    }
    if (v & STATUS_TIMEOUT) return LA_ERR_TIMEOUT;
    return (v & STATUS_BOUNDS) ? LA_ERR_BOUNDS : LA_OK;
}

const char* la_get_error_string(int code) {
    switch (code) {
        case LA_OK: return "ok";
        case LA_ERR_INVALID_ARG: return "invalid argument";
        case LA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case LA_ERR_CUDA: return "CUDA runtime or launch failure";
        case LA_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
        case LA_ERR_WORKSPACE: return "workspace pointer not 256-byte aligned, or too small for a call that needs one";
        case LA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the library's static buffer holds";
        case LA_ERR_BOUNDS: return "checked build: a kernel access fell outside a buffer's extent and was skipped";
        default: return "unknown error";
    }
}

int la_last_launch_count(void) { return t_launches; }

int la_checked_build(void) { return LA_CHECKS; }

}  // extern "C"
