"""GPU parity of the other feature maps against the float64 oracle: the positive
random-feature map on the tensor cores (la_feature_map_prf, per element against
oracle.phi_prf on the same bf16 x and W), and causal linear attention on mapped features
(la_causal_fwd_mapped: the chunked kernels with the map applied by the caller) against
the oracle's recurrence on the oracle's own features, with Gaussian (PRF) and orthogonal
(ORF) projections, on the tensor-core and the SIMT paths."""
import numpy as np
import pytest
import torch

import compressive_memory_attention_02_b300 as la
import oracle
import synthetic
from gpu_helpers import TOL_BF16, TOL_F32, check_status, to_dev, to_host

pytestmark = pytest.mark.gpu


def _W(kind, seed, m, d):
    G = synthetic.normal(seed, 10, (m, d), 1.0, "f32")
    if kind == "prf":
        return synthetic.to_bf16_bits(G)
    return synthetic.to_bf16_bits(oracle.orf_matrix(G, synthetic.normal(seed, 11, (m, d), 1.0, "f32")))


def _map(x, W):
    rows = int(np.prod(x.shape[:-1]))
    d, m = x.shape[-1], W.shape[0]
    out = torch.empty(*x.shape[:-1], m, dtype=torch.bfloat16, device="cuda")
    la.la_feature_map_prf(to_dev(x), to_dev(W), out, rows, d, m)
    return out


@pytest.mark.parametrize("d,m", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_prf_map_matches_oracle(d, m):
    x = synthetic.normal(800 + d + m, 0, (1000, d), 0.3, "bf16")     # 1000 rows: a ragged last tile
    W = _W("prf", 801, m, d)
    got = _map(x, W)
    check_status()
    ref = oracle.phi_prf(x, W)
    e = oracle.rel_err_rows(to_host(got), ref)
    print(f"PARITY prf_map_d{d}_m{m} rows={e:.3e}")
    assert e <= TOL_BF16


@pytest.mark.parametrize("kind", ["prf", "orf"])
@pytest.mark.parametrize("d,T", [(64, 700), (128, 300)])
def test_random_feature_attention_on_tensor_cores(kind, d, T):
    B, H, m = 2, 2, d
    q = synthetic.normal(820 + d, 0, (B, H, T, d), 0.25, "bf16")
    k = synthetic.normal(820 + d, 1, (B, H, T, d), 0.25, "bf16")
    v = synthetic.normal(820 + d, 2, (B, H, T, d), 0.5, "bf16")
    W = _W(kind, 821, m, d)
    fq, fk = _map(q, W), _map(k, W)
    out = torch.empty(B, H, T, d, dtype=torch.bfloat16, device="cuda")
    M = torch.empty(B, H, m, d, device="cuda")
    z = torch.empty(B, H, m, device="cuda")
    nws = la.la_causal_fwd_workspace_size(B, H, T, m, d, 64, la.LA_BF16)
    ws = torch.empty(max(nws, 256), dtype=torch.uint8, device="cuda")
    la.la_causal_fwd_mapped(fq, fk, to_dev(v), out, None, None, M, z, B, H, T, m, d, 64, 1e-6, la.LA_BF16,
                            None, ws, nws)
    check_status()
    r_out, r_M, r_z = oracle.causal_fwd(oracle.phi_prf(q, W), oracle.phi_prf(k, W), synthetic.to_f64(v),
                                        phi="identity")
    e = (oracle.rel_err_rows(to_host(out), r_out), oracle.rel_err_state(to_host(M), r_M, (2, 3)),
         oracle.rel_err_state(to_host(z), r_z, (2,)))
    print(f"PARITY {kind}_attention_d{d}_T{T} out={e[0]:.3e} M={e[1]:.3e} z={e[2]:.3e}")
    assert max(e) <= TOL_BF16


def test_mapped_features_on_the_float32_path():
    """Float32 feature values (the oracle's PRF features rounded to f32) through the SIMT path."""
    B, H, T, d, m = 1, 2, 200, 16, 32
    q, k, v = (synthetic.normal(840, i, (B, H, T, d), 0.5, "f32") for i in range(3))
    W = synthetic.normal(841, 10, (m, d), 1.0, "f32")
    fq, fk = oracle.phi_prf(q, W), oracle.phi_prf(k, W)
    fq32, fk32 = fq.astype(np.float32), fk.astype(np.float32)
    out = torch.empty(B, H, T, d, device="cuda")
    M = torch.empty(B, H, m, d, device="cuda")
    z = torch.empty(B, H, m, device="cuda")
    la.la_causal_fwd_mapped(to_dev(fq32), to_dev(fk32), to_dev(v), out, None, None, M, z, B, H, T, m, d, 32, 1e-6,
                            la.LA_F32, None, None, 0)
    check_status()
    r_out, r_M, _ = oracle.causal_fwd(fq32, fk32, v, phi="identity")
    assert oracle.rel_err_rows(to_host(out), r_out) <= TOL_F32
    assert oracle.rel_err_state(to_host(M), r_M, (2, 3)) <= TOL_F32


def test_mapped_path_with_elu1_features_equals_the_elu1_path():
    """The identity path on features the elu + 1 map produced equals la_causal_fwd itself
    (float32 SIMT path: both compute phi in f32 from the same values)."""
    B, H, T, d = 1, 2, 150, 32
    q, k, v = (synthetic.normal(850, i, (B, H, T, d), 1.0, "f32") for i in range(3))
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    a = torch.empty(B, H, T, d, device="cuda")
    la.la_causal_fwd_ex(tq, tk, tv, a, None, None, None, None, B, H, T, d, d, 64, 1e-6, la.LA_F32, None, None, 0)
    fq = torch.where(tq > 0, tq + 1, torch.exp(tq))
    fk = torch.where(tk > 0, tk + 1, torch.exp(tk))
    b = torch.empty_like(a)
    la.la_causal_fwd_mapped(fq, fk, tv, b, None, None, None, None, B, H, T, d, d, 64, 1e-6, la.LA_F32, None, None, 0)
    check_status()
    assert oracle.rel_err_rows(to_host(b), to_host(a)) <= 1e-5
