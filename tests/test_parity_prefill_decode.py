"""GPU parity of the prompt (prefill) and generation (decode) modes against the
float64 oracle, plus the cross-mode identities: prefill state == forward final
state, and a decode step == the last row of a forward over the appended token."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_helpers import TOL_BF16, TOL_F32, check_status, decode, fwd, prefill, rand_state, to_dev, to_host

pytestmark = pytest.mark.gpu


def _inputs(seed, B, H, T, d, dv, dtype, scale):
    return (synthetic.normal(seed, 0, (B, H, T, d), scale, dtype),
            synthetic.normal(seed, 1, (B, H, T, d), scale, dtype),
            synthetic.normal(seed, 2, (B, H, T, dv), scale, dtype))


def _cmp_prefill(got, ref, tol):
    out, M, z = got
    r_out, r_M, r_z = ref
    if out is not None:
        assert oracle.rel_err_rows(to_host(out), r_out) <= tol
    if M is not None:
        assert oracle.rel_err_state(to_host(M), r_M, (2, 3)) <= tol
    if z is not None:
        assert oracle.rel_err_state(to_host(z), r_z, (2,)) <= tol


# ------------------------------------------------------------------ prefill

@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (128, 64)])
@pytest.mark.parametrize("T,segment", [(64, 64), (1000, 256), (4133, 4096), (3000, 0)])
def test_prefill_bf16(d, dv, T, segment):
    q, k, v = _inputs(500 + T + d, 2, 3, T, d, dv, "bf16", 0.5)
    M0, z0 = rand_state(9, 2, 3, d, dv, scale=2.0)
    got = prefill(to_dev(q), to_dev(k), to_dev(v), to_dev(M0), to_dev(z0), segment=segment)
    _cmp_prefill(got, oracle.prefill(q, k, v, M_in=M0, z_in=z0), TOL_BF16)


@pytest.mark.parametrize("workspace", [True, False])
@pytest.mark.parametrize("want_M", [True, False])
def test_prefill_output_only(workspace, want_M):
    q, k, v = _inputs(51, 1, 4, 2000, 128, 128, "bf16", 0.5)
    got = prefill(to_dev(q), to_dev(k), to_dev(v), segment=512, workspace=workspace, want_M=want_M, want_z=want_M)
    _cmp_prefill(got, oracle.prefill(q, k, v), TOL_BF16)


def test_prefill_fp32():
    q, k, v = _inputs(52, 2, 2, 700, 32, 48, "f32", 1.0)
    M0, z0 = rand_state(10, 2, 2, 32, 48)
    got = prefill(to_dev(q), to_dev(k), to_dev(v), to_dev(M0), to_dev(z0), segment=128)
    _cmp_prefill(got, oracle.prefill(q, k, v, M_in=M0, z_in=z0), TOL_F32)


def test_prefill_state_equals_forward_state():
    q, k, v = _inputs(53, 2, 4, 3000, 128, 128, "bf16", 0.5)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    o_f, M_f, z_f = fwd(tq, tk, tv)
    o_p, M_p, z_p = prefill(tq, tk, tv, segment=512)
    assert oracle.rel_err_state(to_host(M_p), to_host(M_f), (2, 3)) <= 1e-3
    assert oracle.rel_err_state(to_host(z_p), to_host(z_f), (2,)) <= 1e-4
    assert oracle.rel_err_rows(to_host(o_p), to_host(o_f[:, :, -1])) <= TOL_BF16


def test_prefill_workload_full_sampled_heads():
    w = synthetic.WORKLOADS["prefill"]
    q, k, v = synthetic.qkv(w)
    got = prefill(to_dev(q), to_dev(k), to_dev(v), segment=w.segment, eps=w.eps)
    heads = [1, 6]
    r_out, r_M, r_z = oracle.prefill(q[:, heads], k[:, heads], v[:, heads], eps=w.eps)
    out, M, z = got
    e_out = oracle.rel_err_rows(to_host(out[:, heads]), r_out)
    e_M = oracle.rel_err_state(to_host(M[:, heads]), r_M, (2, 3))
    e_z = oracle.rel_err_state(to_host(z[:, heads]), r_z, (2,))
    print(f"PARITY workload_prefill out={e_out:.3e} M={e_M:.3e} z={e_z:.3e} (2 sampled heads)")
    assert e_out <= TOL_BF16 and e_M <= TOL_BF16 and e_z <= TOL_BF16


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("d,dv,dtype", [(128, 128, "bf16"), (64, 64, "bf16"), (32, 48, "f32"), (128, 128, "f32")])
def test_decode_steps(d, dv, dtype):
    N, H, steps = 5, 3, 12
    M0, z0 = rand_state(11, N, H, d, dv, scale=2.0)
    Md, zd = to_dev(M0), to_dev(z0)
    M_ref, z_ref = M0.astype(np.float64), z0.astype(np.float64)
    tol = TOL_BF16 if dtype == "bf16" else TOL_F32
    for s in range(steps):
        q = synthetic.normal(60 + s, 0, (N, H, d), 0.5, dtype)
        k = synthetic.normal(60 + s, 1, (N, H, d), 0.5, dtype)
        v = synthetic.normal(60 + s, 2, (N, H, dv), 0.5, dtype)
        out = decode(to_dev(q), to_dev(k), to_dev(v), Md, zd)
        r_out, M_ref, z_ref = oracle.decode_step(q, k, v, M_ref, z_ref)
        assert oracle.rel_err_rows(to_host(out), r_out) <= tol
    check_status()
    assert oracle.rel_err_state(to_host(Md), M_ref, (2, 3)) <= (1e-5 if dtype == "f32" else 1e-5)
    assert oracle.rel_err_state(to_host(zd), z_ref, (2,)) <= 1e-5


def test_decode_equals_appended_forward():
    q, k, v = _inputs(54, 2, 3, 501, 128, 128, "bf16", 0.5)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    o_all, _, _ = fwd(tq, tk, tv)
    _, M, z = prefill(tq[:, :, :500].contiguous(), tk[:, :, :500].contiguous(), tv[:, :, :500].contiguous(),
                      segment=128, want_out=False)
    o = decode(tq[:, :, 500].contiguous(), tk[:, :, 500].contiguous(), tv[:, :, 500].contiguous(), M, z)
    check_status()
    assert oracle.rel_err_rows(to_host(o), to_host(o_all[:, :, 500])) <= TOL_BF16


def test_generation_workload_full_sampled_heads():
    """256 streams x 32 heads: state from a 2048-token prefill (run in blocks of
    heads), then 1024 decode steps; sampled (stream, head) pairs are checked against
    the oracle at every step, and the state at the end."""
    w = synthetic.WORKLOADS["generation"]
    N, H, d, dv, T0, steps = w.B, w.H, w.d, w.dv, w.T, w.decode_steps
    NH = N * H
    M = torch.empty(NH, d, dv, device="cuda")
    z = torch.empty(NH, d, device="cuda")
    blk = 1024
    for a in range(0, NH, blk):
        # heads [a, a+blk) of the [N*H, T0, d] prompt tensors: a contiguous flat index range
        kk = synthetic.normal(w.seed, synthetic.TID_K, (1, blk, T0, d), w.scale, "bf16", first=a * T0 * d)
        vv = synthetic.normal(w.seed, synthetic.TID_V, (1, blk, T0, dv), w.scale, "bf16", first=a * T0 * dv)
        tk, tv = to_dev(kk), to_dev(vv)
        _, Mb, zb = prefill(tk, tk, tv, segment=512, want_out=False)   # prompt queries do not enter the state
        M[a:a + blk] = Mb[0]
        z[a:a + blk] = zb[0]
        del tk, tv
    sample = [0 * H + 0, 17 * H + 5, 128 * H + 31, 255 * H + 12]
    ks = np.concatenate([synthetic.normal(w.seed, synthetic.TID_K, (1, 1, T0, d), w.scale, "bf16", first=i * T0 * d)
                         for i in sample], axis=1)
    vs = np.concatenate([synthetic.normal(w.seed, synthetic.TID_V, (1, 1, T0, dv), w.scale, "bf16",
                                          first=i * T0 * dv) for i in sample], axis=1)
    _, M_ref, z_ref = oracle.prefill(ks, ks, vs, eps=w.eps)
    M_ref, z_ref = M_ref[0], z_ref[0]
    e_pre = oracle.rel_err_state(to_host(M[sample]), M_ref, (1, 2))
    print(f"PARITY workload_generation_prompt M={e_pre:.3e}")
    assert e_pre <= TOL_BF16
    M4, z4 = M.view(N, H, d, dv), z.view(N, H, d)
    out = torch.empty(N, H, dv, dtype=torch.bfloat16, device="cuda")
    worst = 0.0
    for s in range(steps):
        q, k, v = synthetic.decode_tokens(w, s)
        decode(to_dev(q), to_dev(k), to_dev(v), M4, z4, eps=w.eps, out=out)
        sel = lambda a: a.reshape(NH, -1)[sample][:, None]
        r_out, M_ref, z_ref = oracle.decode_step(sel(q), sel(k), sel(v), M_ref[:, None], z_ref[:, None], eps=w.eps)
        M_ref, z_ref = M_ref[:, 0], z_ref[:, 0]
        worst = max(worst, oracle.rel_err_rows(to_host(out.view(NH, dv)[sample]), r_out[:, 0]))
    check_status()
    e_M = oracle.rel_err_state(to_host(M[sample]), M_ref, (1, 2))
    e_z = oracle.rel_err_state(to_host(z[sample]), z_ref, (1,))
    print(f"PARITY workload_generation out={worst:.3e} M={e_M:.3e} z={e_z:.3e} (4 sampled streams, 1024 steps)")
    assert worst <= TOL_BF16, worst
    assert e_M <= TOL_BF16 and e_z <= TOL_BF16
