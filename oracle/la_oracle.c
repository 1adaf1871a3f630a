/*
 * float64 reference for causal linear attention in the Katharopoulos form.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the oracle that the CUDA library is
 * checked against. Only the tests, the smoke check and the benchmark's CPU
 * baseline may load it; the library never does.
 *
 * What it computes (token by token, float64, no blocking or reordering):
 *   The recurrence of "Implementing Causality with Cumulative Sums" on the
 *   page "Attention_Kernel_Mask" (allenlu2009.github.io, 2024-11-17):
 *       S_t = S_{t-1} + k_t             (key sum; called z here)
 *       Z_t = Z_{t-1} + k_t v_t^T       (context sum; called M here, d x dv)
 *       D_t = q_t^T S_t + eps
 *       out_t = q_t^T Z_t / D_t
 *   applied to phi(q), phi(k) with phi(x) = elu(x) + 1 = (x > 0 ? x + 1 : exp(x)),
 *   the feature map of Katharopoulos et al. 2020 ("Transformers are RNNs"),
 *   whose update and retrieval rule the page "Segment-Wise Attention"
 *   (github.com/beomi/infinitransformer, issue 2) names for the compressive
 *   memory. The state (M, z) is one per (batch, head) and may be carried in
 *   from a previous segment (M_in, z_in) and out to the next (M_out, z_out),
 *   which is the segment-wise use described on that page.
 *
 * Inputs are the storage arrays the GPU also reads: bf16 bit patterns
 * (dtype 1), float32 (dtype 0) or float64 (dtype 2), contiguous [B, H, T, d]
 * for q and k and [B, H, T, dv] for v. They are widened exactly to float64
 * before use.
 *
 * The feature map: phi_kind 0 is elu(x) + 1 on q and k (the map above);
 * phi_kind 1 takes q and k as feature values already (phi applied by the
 * caller, for instance a random-feature map), so that other feature maps run
 * through the same recurrence.
 *
 * The `mutation` argument exists only so the pin tests can show that each
 * planted mistake is caught; 0 is the oracle proper:
 *   1 read the state before adding token t (output excludes its own token)
 *   2 drop eps from the denominator
 *   3 phi = elu (without the +1)
 *   4 use M transposed in the read-out (q^T Z read as Z q over the other index)
 *   5 drop the key sum from the denominator's update (z not accumulated for t > 0)
 *   6 apply phi to v as well
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static inline double widen(const void* base, int dtype, int64_t i) {
    if (dtype == 2) return ((const double*)base)[i];
    if (dtype == 1) {
        union { uint32_t u; float f; } c;
        c.u = (uint32_t)((const uint16_t*)base)[i] << 16;
        return (double)c.f;
    }
    return (double)((const float*)base)[i];
}

static inline double phi(double x, int mutation) {
    if (mutation == 3) return x > 0.0 ? x : exp(x) - 1.0;
    return x > 0.0 ? x + 1.0 : exp(x);
}

/* The feature map of q and k: elu + 1 (phi_kind 0), or the values as given (phi_kind 1). */
static inline double phi_qk(double x, int phi_kind, int mutation) {
    return phi_kind == 1 ? x : phi(x, mutation);
}

/* One (batch, head) stream: T tokens, state carried in M (d x dv) and z (d).
 * out (T x dv) may be NULL; if last_only, only row T-1 is written to out[0..dv). */
static void stream_fwd(const void* q, const void* k, const void* v, int dtype,
                       int64_t qoff, int64_t voff, int64_t T, int d, int dv,
                       double eps, double* M, double* z, double* out, int last_only,
                       int phi_kind, int mutation) {
    double* fq = (double*)malloc(sizeof(double) * (size_t)d);
    double* fk = (double*)malloc(sizeof(double) * (size_t)d);
    double* vv = (double*)malloc(sizeof(double) * (size_t)dv);
    for (int64_t t = 0; t < T; ++t) {
        for (int i = 0; i < d; ++i) {
            fq[i] = phi_qk(widen(q, dtype, qoff + t * d + i), phi_kind, mutation);
            fk[i] = phi_qk(widen(k, dtype, qoff + t * d + i), phi_kind, mutation);
        }
        for (int j = 0; j < dv; ++j) {
            double x = widen(v, dtype, voff + t * dv + j);
            vv[j] = (mutation == 6) ? phi(x, 0) : x;
        }
        int want = out && (!last_only || t == T - 1);
        double* o = out ? (last_only ? out : out + t * dv) : NULL;
        if (mutation == 1 && want) {          /* planted: read before update */
            double den = eps;
            for (int i = 0; i < d; ++i) den += fq[i] * z[i];
            for (int j = 0; j < dv; ++j) {
                double s = 0.0;
                for (int i = 0; i < d; ++i) s += fq[i] * M[(int64_t)i * dv + j];
                o[j] = s / den;
            }
        }
        /* S_t = S_{t-1} + phi(k_t);  Z_t = Z_{t-1} + phi(k_t) v_t^T */
        if (!(mutation == 5 && t > 0))
            for (int i = 0; i < d; ++i) z[i] += fk[i];
        for (int i = 0; i < d; ++i) {
            double* row = M + (int64_t)i * dv;
            const double a = fk[i];
            for (int j = 0; j < dv; ++j) row[j] += a * vv[j];
        }
        if (want && mutation != 1) {
            /* D_t = phi(q_t)^T S_t + eps;  out_t = phi(q_t)^T Z_t / D_t */
            double den = (mutation == 2) ? 0.0 : eps;
            for (int i = 0; i < d; ++i) den += fq[i] * z[i];
            for (int j = 0; j < dv; ++j) o[j] = 0.0;
            if (mutation == 4) {
                /* planted: transposed state read (only meaningful for d == dv) */
                for (int j = 0; j < dv; ++j) {
                    double s = 0.0;
                    for (int i = 0; i < d && i < dv; ++i) s += fq[i] * M[(int64_t)j * dv + i];
                    o[j] = s;
                }
            } else {
                for (int i = 0; i < d; ++i) {
                    const double a = fq[i];
                    const double* row = M + (int64_t)i * dv;
                    for (int j = 0; j < dv; ++j) o[j] += a * row[j];
                }
            }
            for (int j = 0; j < dv; ++j) o[j] /= den;
        }
    }
    free(fq);
    free(fk);
    free(vv);
}

static void load_state(const double* M_in, const double* z_in, int64_t bh, int d, int dv,
                       double* M, double* z) {
    const int64_t ms = (int64_t)d * dv;
    if (M_in) memcpy(M, M_in + bh * ms, sizeof(double) * (size_t)ms);
    else memset(M, 0, sizeof(double) * (size_t)ms);
    if (z_in) memcpy(z, z_in + bh * d, sizeof(double) * (size_t)d);
    else memset(z, 0, sizeof(double) * (size_t)d);
}

static void store_state(double* M_out, double* z_out, int64_t bh, int d, int dv,
                        const double* M, const double* z) {
    const int64_t ms = (int64_t)d * dv;
    if (M_out) memcpy(M_out + bh * ms, M, sizeof(double) * (size_t)ms);
    if (z_out) memcpy(z_out + bh * d, z, sizeof(double) * (size_t)d);
}

/* Training-mode forward: all T outputs per (b, h), plus the final state.
 * out: [B, H, T, dv] float64 (may be NULL); M_in/z_in/M_out/z_out: float64
 * [B, H, d, dv] / [B, H, d], each may be NULL (NULL input = zero state).
 * Parallel over (b, h) with OpenMP; each stream is a plain sequential loop. */
void oracle_causal_fwd(const void* q, const void* k, const void* v, int dtype,
                       const double* M_in, const double* z_in,
                       double* out, double* M_out, double* z_out,
                       int64_t B, int64_t H, int64_t T, int d, int dv, double eps,
                       int phi_kind, int mutation) {
    const int64_t BH = B * H;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double* M = (double*)malloc(sizeof(double) * (size_t)d * dv);
        double* z = (double*)malloc(sizeof(double) * (size_t)d);
        load_state(M_in, z_in, bh, d, dv, M, z);
        stream_fwd(q, k, v, dtype, bh * T * d, bh * T * dv, T, d, dv, eps, M, z,
                   out ? out + bh * T * dv : NULL, 0, phi_kind, mutation);
        store_state(M_out, z_out, bh, d, dv, M, z);
        free(M);
        free(z);
    }
}

/* Prefill ("prompt") mode: the final state and only the last token's output.
 * out_last: [B, H, dv] float64 (may be NULL). */
void oracle_prefill(const void* q, const void* k, const void* v, int dtype,
                    const double* M_in, const double* z_in,
                    double* out_last, double* M_out, double* z_out,
                    int64_t B, int64_t H, int64_t T, int d, int dv, double eps,
                    int phi_kind, int mutation) {
    const int64_t BH = B * H;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double* M = (double*)malloc(sizeof(double) * (size_t)d * dv);
        double* z = (double*)malloc(sizeof(double) * (size_t)d);
        load_state(M_in, z_in, bh, d, dv, M, z);
        stream_fwd(q, k, v, dtype, bh * T * d, bh * T * dv, T, d, dv, eps, M, z,
                   out_last ? out_last + bh * dv : NULL, 1, phi_kind, mutation);
        store_state(M_out, z_out, bh, d, dv, M, z);
        free(M);
        free(z);
    }
}

/* Generation mode: one recurrent step for N independent streams x H heads.
 * q, k: [N, H, d]; v: [N, H, dv] storage arrays; M, z: float64 [N, H, d, dv] /
 * [N, H, d], updated in place; out: [N, H, dv] float64. */
void oracle_decode_step(const void* q, const void* k, const void* v, int dtype,
                        double* M, double* z, double* out,
                        int64_t N, int64_t H, int d, int dv, double eps, int phi_kind,
                        int mutation) {
    const int64_t NH = N * H;
    #pragma omp parallel for schedule(static)
    for (int64_t nh = 0; nh < NH; ++nh) {
        stream_fwd(q, k, v, dtype, nh * d, nh * dv, 1, d, dv, eps,
                   M + nh * (int64_t)d * dv, z + nh * d, out + nh * dv, 0, phi_kind, mutation);
    }
}

/* ------------------------------------------------------------------------
 * Training backward (float64).
 *
 * Gradients of a scalar loss L whose gradients with respect to the forward's
 * outputs are given: dout_t for every output, dM_out and dz_out for the final
 * state. The pages name a training-backward mode (page "Attention_Kernel_Mask",
 * table "Causal Attention Training and Inferencing") but print no formula, so
 * this is the chain rule applied to the recurrence above, token by token:
 *   forward sweep, t = 0 .. T-1 (z_t and M_t include token t):
 *       g_t = dout_t / D_t               gradient of phi(q_t)^T M_t
 *       e_t = -(g_t . out_t)             gradient of D_t
 *       dphi(q_t) = M_t g_t + e_t z_t
 *   reverse sweep, i = T-1 .. 0, from R = dM_out and r = dz_out:
 *       R += phi(q_i) g_i^T,  r += e_i phi(q_i)   (every read at t >= i sees token i)
 *       dphi(k_i) = R v_i + r,  dv_i = R^T phi(k_i)
 *   after the sweep dM_in = R and dz_in = r; dx = dphi(x) phi'(x), where
 *   phi'(x) = 1 for x > 0 and exp(x) otherwise.
 *
 * mutation (pin tests only): 11 drop e_t z_t from dphi(q_t); 12 use the state
 * before token t in dphi(q_t); 13 ignore dM_out and dz_out; 14 use R and r before
 * adding token i's own term; 15 phi' = 1 everywhere; 16 dv_i = R phi(k_i) read
 * over the other index (d == dv only).
 */
static inline double dphi(double x, int mutation) {
    if (mutation == 15) return 1.0;
    return x > 0.0 ? 1.0 : exp(x);
}

static void stream_bwd(const void* q, const void* k, const void* v, int dtype, int64_t qoff, int64_t voff,
                       int64_t T, int d, int dv, double eps, double* M, double* z, const double* dout,
                       const double* dM_out, const double* dz_out, double* dq, double* dk, double* dvv,
                       double* dM_in, double* dz_in, int mutation) {
    double* fq_all = (double*)malloc(sizeof(double) * (size_t)(T * d));
    double* g_all = (double*)malloc(sizeof(double) * (size_t)(T * dv));
    double* e_all = (double*)malloc(sizeof(double) * (size_t)T);
    double* fk = (double*)malloc(sizeof(double) * (size_t)d);
    double* vv = (double*)malloc(sizeof(double) * (size_t)dv);
    double* o = (double*)malloc(sizeof(double) * (size_t)dv);
    double* R = (double*)malloc(sizeof(double) * (size_t)d * dv);
    double* r = (double*)malloc(sizeof(double) * (size_t)d);
    for (int64_t t = 0; t < T; ++t) {
        double* fq = fq_all + t * d;
        double* g = g_all + t * dv;
        for (int i = 0; i < d; ++i) {
            fq[i] = phi(widen(q, dtype, qoff + t * d + i), 0);
            fk[i] = phi(widen(k, dtype, qoff + t * d + i), 0);
        }
        for (int j = 0; j < dv; ++j) vv[j] = widen(v, dtype, voff + t * dv + j);
        for (int i = 0; i < d; ++i) {
            z[i] += fk[i];
            double* row = M + (int64_t)i * dv;
            for (int j = 0; j < dv; ++j) row[j] += fk[i] * vv[j];
        }
        double den = eps;
        for (int i = 0; i < d; ++i) den += fq[i] * z[i];
        for (int j = 0; j < dv; ++j) o[j] = 0.0;
        for (int i = 0; i < d; ++i) {
            const double* row = M + (int64_t)i * dv;
            for (int j = 0; j < dv; ++j) o[j] += fq[i] * row[j];
        }
        double e = 0.0;
        for (int j = 0; j < dv; ++j) {
            o[j] /= den;
            g[j] = dout[t * dv + j] / den;
            e -= g[j] * o[j];
        }
        e_all[t] = e;
        for (int i = 0; i < d; ++i) {
            const double* row = M + (int64_t)i * dv;
            double s = 0.0;
            for (int j = 0; j < dv; ++j) s += row[j] * g[j];
            double zi = z[i];
            if (mutation == 12) {   /* planted: state before token t */
                double vg = 0.0;
                for (int j = 0; j < dv; ++j) vg += vv[j] * g[j];
                s -= fk[i] * vg;
                zi -= fk[i];
            }
            if (mutation != 11) s += e * zi;
            dq[t * d + i] = s * dphi(widen(q, dtype, qoff + t * d + i), mutation);
        }
    }
    for (int64_t a = 0; a < (int64_t)d * dv; ++a) R[a] = (dM_out && mutation != 13) ? dM_out[a] : 0.0;
    for (int i = 0; i < d; ++i) r[i] = (dz_out && mutation != 13) ? dz_out[i] : 0.0;
    for (int64_t t = T - 1; t >= 0; --t) {
        const double* fq = fq_all + t * d;
        const double* g = g_all + t * dv;
        for (int i = 0; i < d; ++i) fk[i] = phi(widen(k, dtype, qoff + t * d + i), 0);
        for (int j = 0; j < dv; ++j) vv[j] = widen(v, dtype, voff + t * dv + j);
        if (mutation != 14) {
            for (int i = 0; i < d; ++i) {
                double* row = R + (int64_t)i * dv;
                for (int j = 0; j < dv; ++j) row[j] += fq[i] * g[j];
                r[i] += e_all[t] * fq[i];
            }
        }
        for (int i = 0; i < d; ++i) {
            const double* row = R + (int64_t)i * dv;
            double s = r[i];
            for (int j = 0; j < dv; ++j) s += row[j] * vv[j];
            dk[t * d + i] = s * dphi(widen(k, dtype, qoff + t * d + i), mutation);
        }
        for (int j = 0; j < dv; ++j) {
            double s = 0.0;
            if (mutation == 16) {
                for (int i = 0; i < d && i < dv; ++i) s += R[(int64_t)j * dv + i] * fk[i];
            } else {
                for (int i = 0; i < d; ++i) s += R[(int64_t)i * dv + j] * fk[i];
            }
            dvv[t * dv + j] = s;
        }
        if (mutation == 14) {
            for (int i = 0; i < d; ++i) {
                double* row = R + (int64_t)i * dv;
                for (int j = 0; j < dv; ++j) row[j] += fq[i] * g[j];
                r[i] += e_all[t] * fq[i];
            }
        }
    }
    if (dM_in) memcpy(dM_in, R, sizeof(double) * (size_t)d * dv);
    if (dz_in) memcpy(dz_in, r, sizeof(double) * (size_t)d);
    free(fq_all);
    free(g_all);
    free(e_all);
    free(fk);
    free(vv);
    free(o);
    free(R);
    free(r);
}

/* q, k: [B, H, T, d], v: [B, H, T, dv] storage arrays (dtype as above); dout
 * [B, H, T, dv], dM_out [B, H, d, dv], dz_out [B, H, d] float64 (the two state
 * gradients may be NULL = zero); M_in, z_in float64 (NULL = zero state).
 * Outputs float64: dq, dk [B, H, T, d], dv [B, H, T, dv], dM_in, dz_in (may be NULL). */
void oracle_causal_bwd(const void* q, const void* k, const void* v, int dtype,
                       const double* M_in, const double* z_in, const double* dout,
                       const double* dM_out, const double* dz_out,
                       double* dq, double* dk, double* dvv, double* dM_in, double* dz_in,
                       int64_t B, int64_t H, int64_t T, int d, int dv, double eps, int mutation) {
    const int64_t BH = B * H;
    const int64_t ms = (int64_t)d * dv;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double* M = (double*)malloc(sizeof(double) * (size_t)ms);
        double* z = (double*)malloc(sizeof(double) * (size_t)d);
        load_state(M_in, z_in, bh, d, dv, M, z);
        stream_bwd(q, k, v, dtype, bh * T * d, bh * T * dv, T, d, dv, eps, M, z, dout + bh * T * dv,
                   dM_out ? dM_out + bh * ms : NULL, dz_out ? dz_out + bh * d : NULL,
                   dq + bh * T * d, dk + bh * T * d, dvv + bh * T * dv,
                   dM_in ? dM_in + bh * ms : NULL, dz_in ? dz_in + bh * d : NULL, mutation);
        free(M);
        free(z);
    }
}

/* phi on its own, for the pin tests. */
void oracle_phi(const double* x, double* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = phi(x[i], 0);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
