"""GPU parity of the training backward (la_causal_bwd / la_causal_bwd_ex) against the
float64 oracle backward on the same seeded storage arrays. Every gradient is compared
per head as max|diff| / max|ref| over that head's tensor; rows are not normalised one
by one because some cancel to nearly zero by construction (the first token's output
depends on q only through eps). Tolerances: <= 1e-4 on the float32 path, <= 2e-2 for
bf16 inputs and gradients (float32 arithmetic inside)."""
import os

import numpy as np
import pytest
import torch

import compressive_memory_attention_02_b300 as la
import oracle
import synthetic
from gpu_helpers import TOL_BF16, TOL_F32, check_status, dtype_code, fwd, rand_state, to_dev, to_host

pytestmark = pytest.mark.gpu


def _inputs(seed, B, H, T, d, dv, dtype, scale):
    q = synthetic.normal(seed, 0, (B, H, T, d), scale, dtype)
    k = synthetic.normal(seed, 1, (B, H, T, d), scale, dtype)
    v = synthetic.normal(seed, 2, (B, H, T, dv), scale, dtype)
    dout = synthetic.normal(seed, 7, (B, H, T, dv), 1.0, dtype)
    return q, k, v, dout


def _values(a):
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _state_grads(seed, B, H, d, dv):
    rng = np.random.default_rng(seed)
    return rng.normal(size=(B, H, d, dv)).astype(np.float32), rng.normal(size=(B, H, d)).astype(np.float32)


def bwd(q, k, v, dout, M_in=None, z_in=None, dM_out=None, dz_out=None, eps=1e-6, want_state=True, dM_in=None,
        dz_in=None, launches=None):
    B, H, T, d = q.shape
    dv = v.shape[3]
    dq, dk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if want_state and dM_in is None:
        dM_in = torch.empty(B, H, d, dv, dtype=torch.float32, device=q.device)
    if want_state and dz_in is None:
        dz_in = torch.empty(B, H, d, dtype=torch.float32, device=q.device)
    nws = la.la_causal_bwd_workspace_size(B, H, T, d, dv)
    ws = torch.empty(nws, dtype=torch.uint8, device=q.device)
    la.la_causal_bwd_ex(q, k, v, dout, M_in, z_in, dM_out, dz_out, dq, dk, dvv, dM_in, dz_in, B, H, T, d, dv, eps,
                        dtype_code(q), ws, nws)
    # bf16 with d, dv in {64, 128}: the tensor-core sweeps, 2 launches (one range per head), 3
    # (range key-value sums, dq sweep, dk/dv sweep) or 5 (plus the two scans over more than
    # eight ranges per head); otherwise the float32 SIMT kernels, 6 launches
    tc = q.dtype == torch.bfloat16 and d in (64, 128) and dv in (64, 128) and not os.environ.get("LA_FORCE_SIMT")
    n = la.la_last_launch_count()
    if launches is not None:
        assert n == launches
    assert n in ((2, 3, 5) if tc else (6,))
    check_status()
    return dq, dk, dvv, dM_in, dz_in


def _compare(got, ref, tol, name=None):
    errs = {}
    for key, g, r in zip(("dq", "dk", "dv", "dM_in", "dz_in"), got, ref):
        if g is None:
            continue
        errs[key] = oracle.rel_err_state(to_host(g), r, tuple(range(2, r.ndim)))
    if name:
        print(f"PARITY bwd_{name} " + " ".join(f"{k}={v:.3e}" for k, v in errs.items()))
    assert max(errs.values()) <= tol, errs
    return errs


def _case(seed, B, H, T, d, dv, dtype, scale, with_state=True, launches=None):
    q, k, v, dout = _inputs(seed, B, H, T, d, dv, dtype, scale)
    M0 = z0 = dM = dz = None
    if with_state:
        M0, z0 = rand_state(seed + 1, B, H, d, dv)
        dM, dz = _state_grads(seed + 2, B, H, d, dv)
    ref = oracle.causal_bwd(q, k, v, _values(dout), M0, z0, dM, dz)
    dev = lambda a: None if a is None else to_dev(a)
    got = bwd(to_dev(q), to_dev(k), to_dev(v), to_dev(dout), dev(M0), dev(z0), dev(dM), dev(dz), launches=launches)
    return got, ref


# ------------------------------------------------------------------ float32 inputs

@pytest.mark.parametrize("d,dv,T", [(32, 32, 200), (64, 32, 257), (128, 128, 130), (16, 48, 64), (8, 8, 1),
                                    (8, 128, 65), (128, 8, 127)])
def test_fp32_shapes_with_state(d, dv, T):
    got, ref = _case(400 + d + dv + T, 2, 3, T, d, dv, "f32", 1.0)
    _compare(got, ref, TOL_F32)


def test_fp32_zero_state_and_no_state_gradients():
    got, ref = _case(450, 1, 2, 300, 64, 64, "f32", 1.0, with_state=False)
    _compare(got, ref, TOL_F32)


# ------------------------------------------------------------------ bf16 inputs

@pytest.mark.parametrize("d,dv,T", [(64, 64, 200), (128, 128, 130), (64, 128, 100), (128, 64, 64), (32, 16, 333)])
def test_bf16_shapes_with_state(d, dv, T):
    got, ref = _case(500 + d + dv + T, 2, 3, T, d, dv, "bf16", 0.5)
    _compare(got, ref, TOL_BF16, f"shapes_d{d}_dv{dv}_T{T}")


@pytest.mark.parametrize("T", [1, 63, 65, 129])
@pytest.mark.parametrize("d", [64, 128])
def test_bf16_tensor_core_short_and_ragged(d, T):
    got, ref = _case(540 + d + T, 1, 3, T, d, d, "bf16", 0.5)
    _compare(got, ref, TOL_BF16, f"ragged_d{d}_T{T}")


@pytest.mark.parametrize("case", ["eps", "large"])
@pytest.mark.parametrize("d", [64, 128])
def test_bf16_tensor_core_edges(case, d):
    """eps-dominated denominators (q, k ~ -9 + 0.5 N(0,1)) and inputs at scale 4."""
    B, H, T = 1, 2, 300
    if case == "eps":
        q = synthetic.normal(560 + d, 0, (B, H, T, d), 0.5, "bf16", shift=-9.0)
        k = synthetic.normal(560 + d, 1, (B, H, T, d), 0.5, "bf16", shift=-9.0)
        v = synthetic.normal(560 + d, 2, (B, H, T, d), 0.5, "bf16")
    else:
        q, k, v = (synthetic.normal(560 + d, i, (B, H, T, d), 4.0, "bf16") for i in range(3))
    dout = synthetic.normal(560 + d, 7, (B, H, T, d), 1.0, "bf16")
    ref = oracle.causal_bwd(q, k, v, _values(dout))
    got = bwd(to_dev(q), to_dev(k), to_dev(v), to_dev(dout))
    _compare(got, ref, TOL_BF16, f"{case}_d{d}")


@pytest.mark.parametrize("cpr", [1, 2, 3, 5])
@pytest.mark.parametrize("d,dv,T", [(64, 64, 333), (128, 128, 449), (64, 128, 257), (64, 64, 600), (128, 128, 1100)])
def test_bf16_sweeps_over_forced_range_lengths(monkeypatch, cpr, d, dv, T):
    """The sweeps' ranges of cpr chunks (the default plan puts a whole short sequence in one range):
    every range boundary hands the state and the state gradient over through the per-range records,
    and the last range is ragged. Up to eight ranges per head the blocks add the records up
    themselves and range 0 writes the initial state's gradient (T = 600 and 1100 at cpr = 1, and
    1100 at cpr = 2, take the scans instead)."""
    monkeypatch.setenv("LA_BWD_CPR", str(cpr))
    nr = -(-(-(-T // 64)) // cpr)
    launches = (3 if nr > 1 else 2) if nr <= 8 else 5
    got, ref = _case(590 + cpr + d + T, 1, 3, T, d, dv, "bf16", 0.5, launches=launches)
    _compare(got, ref, TOL_BF16, f"ranges_cpr{cpr}_d{d}_dv{dv}_T{T}")


@pytest.mark.parametrize("cpr", [1, 3])
@pytest.mark.parametrize("grads", ["none", "dM_only", "dz_only"])
def test_bf16_sweeps_partial_state_arguments(monkeypatch, cpr, grads):
    """Initial state given, final-state gradients partly absent, and only one of dM_in / dz_in
    asked for: the folded prologue sums and range 0's write take each pointer on its own."""
    monkeypatch.setenv("LA_BWD_CPR", str(cpr))
    B, H, T, d, dv = 1, 2, 400, 64, 64
    q, k, v, dout = _inputs(640 + cpr, B, H, T, d, dv, "bf16", 0.5)
    M0, z0 = rand_state(641, B, H, d, dv)
    dM, dz = _state_grads(642, B, H, d, dv)
    if grads in ("none", "dz_only"):
        dM = None
    if grads in ("none", "dM_only"):
        dz = None
    ref = oracle.causal_bwd(q, k, v, _values(dout), M0, z0, dM, dz)
    dev = lambda a: None if a is None else to_dev(a)
    want_dM = grads != "dz_only"
    dM_in = torch.empty(B, H, d, dv, dtype=torch.float32, device="cuda") if want_dM else None
    dz_in = torch.empty(B, H, d, dtype=torch.float32, device="cuda") if not want_dM else None
    got = bwd(to_dev(q), to_dev(k), to_dev(v), to_dev(dout), dev(M0), dev(z0), dev(dM), dev(dz), want_state=False,
              dM_in=dM_in, dz_in=dz_in)
    ref = list(ref)
    if not want_dM:
        ref[3] = None
    else:
        ref[4] = None
    _compare(got, tuple(ref), TOL_BF16, f"partial_{grads}_cpr{cpr}")


def test_bf16_training_workload_full_sampled_heads():
    """The training backward at the size the bench times (B=4, H=16, T=4096, d=dv=64, dout ~
    N(0,1)), one call over every head, checked on sampled heads against the oracle backward
    (each head's gradients depend on that head's inputs alone)."""
    w = synthetic.WORKLOADS["train"]
    B, H, T, d, dv = w.B, w.H, w.T, w.d, w.dv
    q, k, v = synthetic.qkv(w)
    dout = synthetic.normal(w.seed, 7, (B, H, T, dv), 1.0, "bf16")
    got = bwd(to_dev(q), to_dev(k), to_dev(v), to_dev(dout))
    heads = [(0, 0), (1, 9), (3, 15)]
    sel = lambda a: np.stack([a[b, h] for b, h in heads])[None]
    ref = oracle.causal_bwd(sel(q), sel(k), sel(v), _values(sel(dout)))
    got_sel = tuple(np.stack([to_host(g[b, h]) for b, h in heads])[None] for g in got)
    errs = {}
    for key, g, r in zip(("dq", "dk", "dv", "dM_in", "dz_in"), got_sel, ref):
        errs[key] = oracle.rel_err_state(g, r, tuple(range(2, r.ndim)))
    print("PARITY bwd_training_workload " + " ".join(f"{k}={v:.3e}" for k, v in errs.items()))
    assert max(errs.values()) <= TOL_BF16, errs
