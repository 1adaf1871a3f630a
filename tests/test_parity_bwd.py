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
        dz_in=None):
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
    # bf16 with d, dv in {64, 128}: the tensor-core sweeps (range key-value sums, scan, dq sweep,
    # reverse scan, dk/dv sweep); otherwise the float32 SIMT kernels (one more launch)
    tc = q.dtype == torch.bfloat16 and d in (64, 128) and dv in (64, 128) and not os.environ.get("LA_FORCE_SIMT")
    assert la.la_last_launch_count() == (5 if tc else 6)
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


def _case(seed, B, H, T, d, dv, dtype, scale, with_state=True):
    q, k, v, dout = _inputs(seed, B, H, T, d, dv, dtype, scale)
    M0 = z0 = dM = dz = None
    if with_state:
        M0, z0 = rand_state(seed + 1, B, H, d, dv)
        dM, dz = _state_grads(seed + 2, B, H, d, dv)
    ref = oracle.causal_bwd(q, k, v, _values(dout), M0, z0, dM, dz)
    dev = lambda a: None if a is None else to_dev(a)
    got = bwd(to_dev(q), to_dev(k), to_dev(v), to_dev(dout), dev(M0), dev(z0), dev(dM), dev(dz))
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
@pytest.mark.parametrize("d,dv,T", [(64, 64, 333), (128, 128, 449), (64, 128, 257)])
def test_bf16_sweeps_over_forced_range_lengths(monkeypatch, cpr, d, dv, T):
    """The sweeps' ranges of cpr chunks (the default plan puts a whole short sequence in one range):
    every range boundary hands the state (prefix scan) and the state gradient (reverse scan) over
    through the per-range records, and the last range is ragged."""
    monkeypatch.setenv("LA_BWD_CPR", str(cpr))
    got, ref = _case(590 + cpr + d + T, 1, 3, T, d, dv, "bf16", 0.5)
    _compare(got, ref, TOL_BF16, f"ranges_cpr{cpr}_d{d}_dv{dv}_T{T}")


def test_bf16_tensor_core_and_simt_paths_agree(monkeypatch):
    got_tc, ref = _case(580, 1, 2, 400, 128, 128, "bf16", 0.5)
    monkeypatch.setenv("LA_FORCE_SIMT", "1")
    got_simt, _ = _case(580, 1, 2, 400, 128, 128, "bf16", 0.5)
    for a, b in zip(got_tc, got_simt):
        r = to_host(b)
        assert np.abs(to_host(a) - r).max() <= TOL_BF16 * np.abs(r).max()


def test_bf16_training_workload_sampled_heads():
    """The training-style workload (B=4, H=16, T=4096, d=dv=64) in one call; two heads
    checked against the oracle (each head's gradients depend on that head only)."""
    w = synthetic.WORKLOADS["train"]
    q, k, v = synthetic.qkv(w)
    dout = synthetic.normal(w.seed, 7, (w.B, w.H, w.T, w.dv), 1.0, w.dtype)
    got = bwd(to_dev(q), to_dev(k), to_dev(v), to_dev(dout))
    for b, h in ((0, 0), (3, 15)):
        sl = lambda a: np.ascontiguousarray(a[b:b + 1, h:h + 1])
        ref = oracle.causal_bwd(sl(q), sl(k), sl(v), _values(sl(dout)))
        head = [g[b:b + 1, h:h + 1] for g in got]
        _compare(head, ref, TOL_BF16, f"workload_train_b{b}h{h}")


def test_bf16_segment_call_shape_sampled_heads():
    """One segment call of the segmented workload's shape (B=2, H=32, T=2048, d=dv=128) with a
    carried-in state and state gradients; three heads checked against the oracle."""
    B, H, T, d, dv = 2, 32, 2048, 128, 128
    q, k, v, dout = _inputs(700, B, H, T, d, dv, "bf16", 0.5)
    M0, z0 = rand_state(701, B, H, d, dv)
    dM, dz = _state_grads(702, B, H, d, dv)
    got = bwd(to_dev(q), to_dev(k), to_dev(v), to_dev(dout), to_dev(M0), to_dev(z0), to_dev(dM), to_dev(dz))
    for b, h in ((0, 0), (1, 17), (1, 31)):
        sl = lambda a: np.ascontiguousarray(a[b:b + 1, h:h + 1])
        ref = oracle.causal_bwd(sl(q), sl(k), sl(v), _values(sl(dout)), sl(M0), sl(z0), sl(dM), sl(dz))
        _compare([g[b:b + 1, h:h + 1] for g in got], ref, TOL_BF16, f"segment_shape_b{b}h{h}")


# ------------------------------------------------------------------ properties and the ABI

def test_segment_backwards_chain_through_state_gradients():
    """Backward of [0, T) == backward of [cut, T) from the first part's final state, then
    backward of [0, cut) fed with that call's dM_in, dz_in (float32 inputs)."""
    B, H, T, d, dv, cut = 1, 2, 320, 32, 32, 192
    q, k, v, dout = (to_dev(a) for a in _inputs(610, B, H, T, d, dv, "f32", 1.0))
    M0, z0 = (to_dev(a) for a in rand_state(611, B, H, d, dv))
    dM, dz = (to_dev(a) for a in _state_grads(612, B, H, d, dv))
    full = bwd(q, k, v, dout, M0, z0, dM, dz)
    part = lambda a, s: a[:, :, s].contiguous()
    s1, s2 = slice(0, cut), slice(cut, T)
    _, M1, z1 = fwd(part(q, s1), part(k, s1), part(v, s1), M0, z0)
    g2 = bwd(part(q, s2), part(k, s2), part(v, s2), part(dout, s2), M1, z1, dM, dz)
    g1 = bwd(part(q, s1), part(k, s1), part(v, s1), part(dout, s1), M0, z0, g2[3], g2[4])
    joined = [torch.cat([a, b], 2) for a, b in zip(g1[:3], g2[:3])] + [g1[3], g1[4]]
    for a, b in zip(joined, full):
        ref = to_host(b)
        assert np.abs(to_host(a) - ref).max() <= 1e-4 * np.abs(ref).max()


def test_state_gradient_in_place():
    B, H, T, d, dv = 1, 2, 100, 32, 16
    q, k, v, dout = (to_dev(a) for a in _inputs(620, B, H, T, d, dv, "f32", 1.0))
    dM, dz = (to_dev(a) for a in _state_grads(621, B, H, d, dv))
    ref = bwd(q, k, v, dout, None, None, dM.clone(), dz.clone())
    got = bwd(q, k, v, dout, None, None, dM, dz, dM_in=dM, dz_in=dz)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)


def test_registered_workspace_and_errors():
    B, H, T, d, dv = 1, 1, 70, 16, 16
    q, k, v, dout = (to_dev(a) for a in _inputs(630, B, H, T, d, dv, "f32", 1.0))
    dq, dk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nws = la.la_causal_bwd_workspace_size(B, H, T, d, dv)
    args = (q, k, v, dout, None, None, None, None, dq, dk, dvv, None, None, B, H, T, d, dv, 1e-6, la.LA_F32)
    la.la_set_workspace(None, 0)
    with pytest.raises(la.LinAttnError) as e:  # no workspace registered
        la.la_causal_bwd(*args)
    assert e.value.code == la.LA_ERR_WORKSPACE
    small = torch.empty(nws - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(la.LinAttnError) as e:
        la.la_causal_bwd_ex(*args, small, small.numel())
    assert e.value.code == la.LA_ERR_WORKSPACE
    with pytest.raises(la.LinAttnError) as e:  # an output aliasing an input
        la.la_causal_bwd_ex(q, k, v, dout, None, None, None, None, q, dk, dvv, None, None, B, H, T, d, dv, 1e-6,
                            la.LA_F32, small, small.numel())
    assert e.value.code == la.LA_ERR_INVALID_ARG
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    la.la_set_workspace(ws, nws)
    try:
        la.la_causal_bwd(*args)
        check_status()
    finally:  # put back a buffer registered earlier in this process, if any
        cur = la._workspaces.get(torch.cuda.current_device())
        la.la_set_workspace(cur if cur is not None else None, cur.numel() if cur is not None else 0)
    ref = oracle.causal_bwd(*(a.cpu().numpy() for a in (q, k, v)), dout.double().cpu().numpy())
    _compare((dq, dk, dvv, None, None), ref, TOL_F32)
