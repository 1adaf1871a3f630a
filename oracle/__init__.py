"""float64 CPU oracle for causal linear attention (Katharopoulos form, phi = elu + 1).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg use it. The library under compressive_memory_attention_02_b300
never imports it and shares no code with it.

Contents
  causal_fwd / prefill / decode_step   the token recurrence in plain C (la_oracle.c),
                                       page "Attention_Kernel_Mask", section
                                       "Implementing Causality with Cumulative Sums"
  causal_bwd                           its training backward: the chain rule on that
                                       recurrence, a forward sweep for dq and a reverse
                                       sweep carrying the state gradient (la_oracle.c);
                                       the page's mode table names the training-backward
                                       mode but prints no formula
  brute_force                          the same outputs from the lower-triangular
                                       (masked O(T^2)) form of that page's question
                                       about multiplying by an all-ones lower-
                                       triangular matrix; numpy matmul as the step
  chunked_form                         the page's "chunk sequential mode" (mode 3)
                                       equation: inter-chunk Q S_prev plus intra-chunk
                                       ((Q K^T) masked) V, with the normaliser split the
                                       same way (the page prints no normaliser; the
                                       split of D_t is our reading)
  noncausal                            all-token (non-causal) linear attention
  phi                                  elu(x) + 1
  phi_prf / orf_matrix                 positive (and orthogonal) random features, used
                                       with phi="identity": the recurrence on feature
                                       values given by the caller
  rel_err_rows / rel_err_state         the tolerance metrics

Readings taken where the pages are silent or garbled:
  phi = elu + 1 on q and k only; eps is added to the denominator; out_t includes
  token t (update then read); the chunk equation's inter term uses the state of
  all tokens before the chunk; no 1/sqrt(d) scaling; state is one (M, z) per head.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile la_oracle.c into _build/liboracle.so (gcc -O2, OpenMP; no fast-math,
    no FMA contraction, so every step rounds as written)."""
    src = os.path.join(_HERE, "la_oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        os.makedirs(os.path.dirname(_SO), exist_ok=True)
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-fopenmp",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, c_int, vp, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
        lib.oracle_causal_fwd.argtypes = [vp, vp, vp, c_int, vp, vp, vp, vp, vp,
                                          i64, i64, i64, c_int, c_int, dbl, c_int, c_int]
        lib.oracle_prefill.argtypes = lib.oracle_causal_fwd.argtypes
        lib.oracle_decode_step.argtypes = [vp, vp, vp, c_int, vp, vp, vp,
                                           i64, i64, c_int, c_int, dbl, c_int, c_int]
        lib.oracle_phi.argtypes = [vp, vp, i64]
        lib.oracle_causal_bwd.argtypes = [vp, vp, vp, c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                          i64, i64, i64, c_int, c_int, dbl, c_int]
        lib.oracle_max_threads.restype = c_int
        for f in (lib.oracle_causal_fwd, lib.oracle_prefill, lib.oracle_decode_step, lib.oracle_phi,
                  lib.oracle_causal_bwd):
            f.restype = None
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.float64:
        return 2
    raise TypeError("storage arrays are uint16 (bf16 bits), float32 or float64")


_PHI = {"elu1": 0, "identity": 1}


def _phi_kind(phi):
    """'elu1': phi = elu + 1 applied to q and k; 'identity': q and k are feature values
    already (another feature map applied by the caller)."""
    return _PHI[phi]


def _c(a):
    return np.ascontiguousarray(a)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _state_or_none(a, shape):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float64)
    assert a.shape == tuple(shape), (a.shape, shape)
    return a


def causal_fwd(q, k, v, M_in=None, z_in=None, eps=1e-6, want_out=True, mutation=0, phi="elu1"):
    """All outputs and the final state. q, k: [B,H,T,d]; v: [B,H,T,dv] storage arrays
    (the same dtype). Returns (out [B,H,T,dv] float64 or None, M [B,H,d,dv], z [B,H,d])."""
    q, k, v = _c(q), _c(k), _c(v)
    assert q.dtype == k.dtype == v.dtype
    B, H, T, d = q.shape
    dv = v.shape[3]
    assert k.shape == q.shape and v.shape[:3] == (B, H, T)
    M_in = _state_or_none(M_in, (B, H, d, dv))
    z_in = _state_or_none(z_in, (B, H, d))
    out = np.empty((B, H, T, dv)) if want_out else None
    M = np.empty((B, H, d, dv))
    z = np.empty((B, H, d))
    _load().oracle_causal_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, _dtype_code(q),
                              _ptr(M_in), _ptr(z_in), _ptr(out), M.ctypes.data, z.ctypes.data,
                              B, H, T, d, dv, float(eps), _phi_kind(phi), int(mutation))
    return out, M, z


def prefill(q, k, v, M_in=None, z_in=None, eps=1e-6, mutation=0, phi="elu1"):
    """Final state and last-token output. Returns (out_last [B,H,dv], M, z)."""
    q, k, v = _c(q), _c(k), _c(v)
    B, H, T, d = q.shape
    dv = v.shape[3]
    M_in = _state_or_none(M_in, (B, H, d, dv))
    z_in = _state_or_none(z_in, (B, H, d))
    out = np.empty((B, H, dv))
    M = np.empty((B, H, d, dv))
    z = np.empty((B, H, d))
    _load().oracle_prefill(q.ctypes.data, k.ctypes.data, v.ctypes.data, _dtype_code(q),
                           _ptr(M_in), _ptr(z_in), out.ctypes.data, M.ctypes.data, z.ctypes.data,
                           B, H, T, d, dv, float(eps), _phi_kind(phi), int(mutation))
    return out, M, z


def decode_step(q, k, v, M, z, eps=1e-6, mutation=0, phi="elu1"):
    """One recurrent step. q, k: [N,H,d]; v: [N,H,dv]; M [N,H,d,dv], z [N,H,d]
    float64 (not modified). Returns (out [N,H,dv], M_new, z_new)."""
    q, k, v = _c(q), _c(k), _c(v)
    N, H, d = q.shape
    dv = v.shape[2]
    M2 = np.array(M, dtype=np.float64, copy=True, order="C")
    z2 = np.array(z, dtype=np.float64, copy=True, order="C")
    assert M2.shape == (N, H, d, dv) and z2.shape == (N, H, d)
    out = np.empty((N, H, dv))
    _load().oracle_decode_step(q.ctypes.data, k.ctypes.data, v.ctypes.data, _dtype_code(q),
                               M2.ctypes.data, z2.ctypes.data, out.ctypes.data,
                               N, H, d, dv, float(eps), _phi_kind(phi), int(mutation))
    return out, M2, z2


def causal_bwd(q, k, v, dout, M_in=None, z_in=None, dM_out=None, dz_out=None, eps=1e-6, mutation=0):
    """Training backward: the gradients of L = sum(dout * out) + sum(dM_out * M_T) +
    sum(dz_out * z_T) with respect to the float64 values of q, k, v (storage arrays,
    as for causal_fwd) and of the initial state. dout [B,H,T,dv], dM_out [B,H,d,dv],
    dz_out [B,H,d] are float64 (the state gradients may be None = zero).
    Returns (dq, dk, dv, dM_in, dz_in), all float64."""
    q, k, v = _c(q), _c(k), _c(v)
    assert q.dtype == k.dtype == v.dtype
    B, H, T, d = q.shape
    dv = v.shape[3]
    M_in = _state_or_none(M_in, (B, H, d, dv))
    z_in = _state_or_none(z_in, (B, H, d))
    dM_out = _state_or_none(dM_out, (B, H, d, dv))
    dz_out = _state_or_none(dz_out, (B, H, d))
    dout = np.ascontiguousarray(dout, dtype=np.float64)
    assert dout.shape == (B, H, T, dv)
    dq = np.empty((B, H, T, d))
    dk = np.empty((B, H, T, d))
    dvv = np.empty((B, H, T, dv))
    dM_in = np.empty((B, H, d, dv))
    dz_in = np.empty((B, H, d))
    _load().oracle_causal_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, _dtype_code(q),
                              _ptr(M_in), _ptr(z_in), dout.ctypes.data, _ptr(dM_out), _ptr(dz_out),
                              dq.ctypes.data, dk.ctypes.data, dvv.ctypes.data, dM_in.ctypes.data,
                              dz_in.ctypes.data, B, H, T, d, dv, float(eps), int(mutation))
    return dq, dk, dvv, dM_in, dz_in


def phi(x) -> np.ndarray:
    """elu(x) + 1 evaluated by the C oracle (float64)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_phi(x.ctypes.data, y.ctypes.data, x.size)
    return y


# ---------------------------------------------------------------------------
# numpy forms (float64). These are separate formulations of the same function,
# used to pin the token recurrence above; they are not faster paths.

def _f64(a):
    """Storage array -> float64 values (bf16 bits are the high half of a float32)."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _phi_np(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def brute_force(q, k, v, M_in=None, z_in=None, eps=1e-6):
    """out_t = (sum_{i<=t} (phi q_t . phi k_i) v_i + phi q_t^T M0) /
               (sum_{i<=t} phi q_t . phi k_i + phi q_t . z0 + eps)
    for every (b, h): the masked all-pairs form, O(T^2) per head."""
    Q, K, V = _phi_np(_f64(q)), _phi_np(_f64(k)), _f64(v)
    B, H, T, d = Q.shape
    A = np.einsum("bhtd,bhsd->bhts", Q, K)
    A = A * np.tril(np.ones((T, T)))[None, None]
    num = np.einsum("bhts,bhsv->bhtv", A, V)
    den = A.sum(-1) + eps
    if M_in is not None:
        num = num + np.einsum("bhtd,bhdv->bhtv", Q, np.asarray(M_in, dtype=np.float64))
    if z_in is not None:
        den = den + np.einsum("bhtd,bhd->bht", Q, np.asarray(z_in, dtype=np.float64))
    return num / den[..., None]


def chunked_form(q, k, v, chunk, M_in=None, z_in=None, eps=1e-6):
    """The page's chunk-sequential mode for chunks of `chunk` tokens:
         O_c = phi(Q_c) M_{c-1} + ((phi(Q_c) phi(K_c)^T) * mask) V_c
         D_c = phi(Q_c) z_{c-1} + rowsum((phi(Q_c) phi(K_c)^T) * mask) + eps
         M_c = M_{c-1} + phi(K_c)^T V_c,   z_c = z_{c-1} + colsum(phi(K_c))
       mask = lower triangle including the diagonal. Returns (out, M, z)."""
    Q, K, V = _phi_np(_f64(q)), _phi_np(_f64(k)), _f64(v)
    B, H, T, d = Q.shape
    dv = V.shape[3]
    M = np.zeros((B, H, d, dv)) if M_in is None else np.array(M_in, dtype=np.float64)
    z = np.zeros((B, H, d)) if z_in is None else np.array(z_in, dtype=np.float64)
    out = np.empty((B, H, T, dv))
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        Qc, Kc, Vc = Q[:, :, c0:c1], K[:, :, c0:c1], V[:, :, c0:c1]
        S = np.einsum("bhtd,bhsd->bhts", Qc, Kc) * np.tril(np.ones((c1 - c0, c1 - c0)))
        num = np.einsum("bhtd,bhdv->bhtv", Qc, M) + np.einsum("bhts,bhsv->bhtv", S, Vc)
        den = np.einsum("bhtd,bhd->bht", Qc, z) + S.sum(-1) + eps
        out[:, :, c0:c1] = num / den[..., None]
        M = M + np.einsum("bhsd,bhsv->bhdv", Kc, Vc)
        z = z + Kc.sum(2)
    return out, M, z


def noncausal(q, k, v, eps=1e-6):
    """Every query attends to all T keys: out_t = phi q_t^T (sum_i phi k_i v_i^T) /
    (phi q_t . sum_i phi k_i + eps)."""
    Q, K, V = _phi_np(_f64(q)), _phi_np(_f64(k)), _f64(v)
    M = np.einsum("bhsd,bhsv->bhdv", K, V)
    z = K.sum(2)
    return np.einsum("bhtd,bhdv->bhtv", Q, M) / (np.einsum("bhtd,bhd->bht", Q, z) + eps)[..., None]


# ---------------------------------------------------------------------------
# other feature maps (inputs of the identity path)

def phi_prf(x, W):
    """Positive random features: phi(x) = exp(W x - |x|^2 / 2) / sqrt(m) for x [..., d] and
    W [m, d] (storage arrays; float64 arithmetic). The page "Attention_Kernel_Mask" lists
    positive random features (PRF) and orthogonal random features (ORF) among the feature
    maps of its non-causal kernel discussion without printing them; this is the positive
    random-feature map of that family, whose expectation over Gaussian rows w ~ N(0, I_d)
    gives E[phi(q) . phi(k)] = exp(q . k). The result is a feature vector per token, to be
    used with phi='identity'."""
    X = _f64(x)
    Wf = _f64(W)
    m = Wf.shape[0]
    return np.exp(X @ Wf.T - 0.5 * (X * X).sum(-1, keepdims=True)) / np.sqrt(m)


def orf_matrix(G, N):
    """Orthogonal random features from Gaussian draws G and N, both [m, d] with m a multiple
    of d: every block of d rows of G is orthogonalised (Q of its QR factorisation, a library
    step), and row i is then scaled to the norm of row i of N, so that each row has the
    length distribution of a Gaussian row while the rows of a block are exactly
    orthogonal. Returns W [m, d] float64."""
    G = np.asarray(G, dtype=np.float64)
    N = np.asarray(N, dtype=np.float64)
    m, d = G.shape
    assert m % d == 0 and N.shape == G.shape
    W = np.empty((m, d))
    for b0 in range(0, m, d):
        Q, _ = np.linalg.qr(G[b0:b0 + d].T)   # columns of Q: orthonormal basis
        W[b0:b0 + d] = Q.T
    return W * np.linalg.norm(N, axis=1, keepdims=True)


# ---------------------------------------------------------------------------
# tolerance metrics

def rel_err_rows(got, ref) -> float:
    """max over rows of ||got_row - ref_row||_inf / ||ref_row||_inf (last axis = row)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.abs(got - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max()) if num.size else 0.0


def rel_err_state(got, ref, axes) -> float:
    """max over the leading (b, h) index of max|got-ref| / max|ref| over `axes`."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.abs(got - ref).max(axis=axes)
    den = np.abs(ref).max(axis=axes)
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max()) if num.size else 0.0
