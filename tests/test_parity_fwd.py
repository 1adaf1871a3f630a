"""GPU parity of the training forward (la_causal_fwd / la_causal_fwd_ex) against the
float64 oracle on the same seeded storage arrays. Tolerances: max row-normwise
relative error <= 1e-4 on the float32 path, <= 2e-2 for bf16 inputs (float32
state); states compared per head as max|diff| / max|ref|."""
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
    return q, k, v


def _compare(got, ref, tol):
    out, M, z = got
    r_out, r_M, r_z = ref
    e_out = oracle.rel_err_rows(to_host(out), r_out)
    e_M = oracle.rel_err_state(to_host(M), r_M, (2, 3))
    e_z = oracle.rel_err_state(to_host(z), r_z, (2,))
    assert e_out <= tol and e_M <= tol and e_z <= tol, (e_out, e_M, e_z)
    return e_out, e_M, e_z


# ------------------------------------------------------------------ float32 (SIMT) path

def test_fp32_tiny_workload():
    w = synthetic.WORKLOADS["tiny"]
    q, k, v = synthetic.qkv(w)
    got = fwd(to_dev(q), to_dev(k), to_dev(v), chunk=w.chunk, eps=w.eps)
    e_out, e_M, e_z = _compare(got, oracle.causal_fwd(q, k, v, eps=w.eps), TOL_F32)
    print(f"PARITY workload_tiny out={e_out:.3e} M={e_M:.3e} z={e_z:.3e}")


@pytest.mark.parametrize("d,dv,chunk,T", [(32, 32, 16, 100), (64, 32, 32, 257), (128, 128, 64, 130),
                                          (16, 48, 128, 300), (8, 8, 16, 1)])
def test_fp32_shapes_with_initial_state(d, dv, chunk, T):
    q, k, v = _inputs(200 + d + T, 2, 3, T, d, dv, "f32", 1.0)
    M0, z0 = rand_state(5, 2, 3, d, dv)
    got = fwd(to_dev(q), to_dev(k), to_dev(v), to_dev(M0), to_dev(z0), chunk=chunk)
    _compare(got, oracle.causal_fwd(q, k, v, M_in=M0, z_in=z0), TOL_F32)


# ------------------------------------------------------------------ bf16 tensor-core path

@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("T", [64, 200, 1000])
@pytest.mark.parametrize("workspace", [True, False])
def test_bf16_tensor_core_shapes(d, dv, T, workspace):
    q, k, v = _inputs(300 + d + dv + T, 2, 3, T, d, dv, "bf16", 0.5)
    got = fwd(to_dev(q), to_dev(k), to_dev(v), workspace=workspace)
    _compare(got, oracle.causal_fwd(q, k, v), TOL_BF16)


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128)])
def test_bf16_initial_state_and_ranges(d, dv):
    q, k, v = _inputs(41, 1, 4, 777, d, dv, "bf16", 0.5)
    M0, z0 = rand_state(6, 1, 4, d, dv, scale=3.0)
    got = fwd(to_dev(q), to_dev(k), to_dev(v), to_dev(M0), to_dev(z0))
    _compare(got, oracle.causal_fwd(q, k, v, M_in=M0, z_in=z0), TOL_BF16)


def test_bf16_in_place_state_update():
    q, k, v = _inputs(42, 2, 2, 900, 128, 128, "bf16", 0.5)
    M0, z0 = rand_state(7, 2, 2, 128, 128)
    Md, zd = to_dev(M0), to_dev(z0)
    got = fwd(to_dev(q), to_dev(k), to_dev(v), Md, zd, M_out=Md, z_out=zd)
    _compare(got, oracle.causal_fwd(q, k, v, M_in=M0, z_in=z0), TOL_BF16)


@pytest.mark.parametrize("d", [32, 128])
def test_bf16_simt_path(d, monkeypatch):
    # d = 32 is not a tensor-core shape; d = 128 is forced onto the SIMT path
    if d == 128:
        monkeypatch.setenv("LA_FORCE_SIMT", "1")
    q, k, v = _inputs(43, 1, 2, 300, d, d, "bf16", 0.5)
    got = fwd(to_dev(q), to_dev(k), to_dev(v))
    _compare(got, oracle.causal_fwd(q, k, v), TOL_BF16)


def test_bf16_tensor_core_matches_simt_path(monkeypatch):
    q, k, v = _inputs(44, 2, 2, 512, 128, 128, "bf16", 0.5)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    a = fwd(tq, tk, tv)
    monkeypatch.setenv("LA_FORCE_SIMT", "1")
    b = fwd(tq, tk, tv)
    assert oracle.rel_err_rows(to_host(a[0]), to_host(b[0])) < TOL_BF16


def test_bf16_causality_is_exact():
    q, k, v = _inputs(45, 1, 2, 640, 128, 128, "bf16", 0.5)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    a = fwd(tq, tk, tv)[0].clone()
    cut = 300                                  # inside a chunk (300 = 4*64 + 44)
    tq2, tk2, tv2 = tq.clone(), tk.clone(), tv.clone()
    tk2[:, :, cut:] = -tk2[:, :, cut:]
    tv2[:, :, cut:] += 3.0
    tq2[:, :, cut:] *= 2.0
    b = fwd(tq2, tk2, tv2)[0]
    assert torch.equal(a[:, :, :cut], b[:, :, :cut])
    assert not torch.equal(a[:, :, cut:], b[:, :, cut:])


def test_bf16_deterministic():
    q, k, v = _inputs(46, 2, 4, 1000, 128, 128, "bf16", 0.5)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    a = fwd(tq, tk, tv)
    b = fwd(tq, tk, tv)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bf16_strided_segment_equals_contiguous_copy():
    B, H, T, d = 2, 2, 1024, 128
    q, k, v = _inputs(47, B, H, T, d, d, "bf16", 0.5)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    s0, s1 = 256, 640
    out = torch.zeros(B, H, T, d, dtype=torch.bfloat16, device="cuda")
    st = [H * T * d, T * d, d] * 4
    M0, z0 = rand_state(8, B, H, d, d)
    Md, zd = to_dev(M0), to_dev(z0)
    sl = lambda t: t[:, :, s0:s1]
    a = fwd(sl(tq), sl(tk), sl(tv), Md, zd, out=sl(out), strides=st, T=s1 - s0)
    b = fwd(sl(tq).contiguous(), sl(tk).contiguous(), sl(tv).contiguous(), Md, zd)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert torch.count_nonzero(out[:, :, :s0]) == 0 and torch.count_nonzero(out[:, :, s1:]) == 0


@pytest.mark.parametrize("T", [1, 63, 65, 129])
def test_bf16_short_and_ragged(T):
    q, k, v = _inputs(48 + T, 3, 5, T, 64, 64, "bf16", 0.5)
    got = fwd(to_dev(q), to_dev(k), to_dev(v))
    _compare(got, oracle.causal_fwd(q, k, v), TOL_BF16)


def test_bf16_many_heads_single_range():
    # B*H above the SM count: one range per head
    q, k, v = _inputs(49, 4, 50, 130, 64, 64, "bf16", 0.5)
    got = fwd(to_dev(q), to_dev(k), to_dev(v))
    _compare(got, oracle.causal_fwd(q, k, v), TOL_BF16)


# ------------------------------------------------------------------ workloads at full size

def test_train_workload_full():
    w = synthetic.WORKLOADS["train"]
    q, k, v = synthetic.qkv(w)
    got = fwd(to_dev(q), to_dev(k), to_dev(v), chunk=w.chunk, eps=w.eps)
    e_out, e_M, e_z = _compare(got, oracle.causal_fwd(q, k, v, eps=w.eps), TOL_BF16)
    print(f"PARITY workload_train out={e_out:.3e} M={e_M:.3e} z={e_z:.3e}")


def test_segmented_workload_full_sampled_heads():
    """16 segments of 2048 chained through M, z (strided calls on one [B,H,T,d]
    tensor, ping-pong state buffers), checked on sampled heads against the oracle
    over all 32768 tokens, and against one unsegmented call on the GPU."""
    w = synthetic.WORKLOADS["segmented"]
    q, k, v = synthetic.qkv(w)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    B, H, T, d, dv, S = w.B, w.H, w.T, w.d, w.dv, w.segment
    out = torch.empty(B, H, T, dv, dtype=torch.bfloat16, device="cuda")
    st = [H * T * d, T * d, d] * 3 + [H * T * dv, T * dv, dv]
    Ms = [torch.empty(B, H, d, dv, device="cuda") for _ in range(2)]
    zs = [torch.empty(B, H, d, device="cuda") for _ in range(2)]
    for s in range(T // S):
        sl = lambda t: t[:, :, s * S:(s + 1) * S]
        Mi, zi = (None, None) if s == 0 else (Ms[(s - 1) % 2], zs[(s - 1) % 2])
        fwd(sl(tq), sl(tk), sl(tv), Mi, zi, chunk=w.chunk, eps=w.eps, out=sl(out),
            M_out=Ms[s % 2], z_out=zs[s % 2], strides=st, T=S)
    M_fin, z_fin = Ms[(T // S - 1) % 2], zs[(T // S - 1) % 2]
    heads = [(0, 0), (0, 31), (1, 7), (1, 20)]
    sel = lambda a: np.stack([a[b, h] for b, h in heads])[None]
    r_out, r_M, r_z = oracle.causal_fwd(sel(q), sel(k), sel(v), eps=w.eps)
    g_out = np.stack([to_host(out[b, h]) for b, h in heads])[None]
    g_M = np.stack([to_host(M_fin[b, h]) for b, h in heads])[None]
    g_z = np.stack([to_host(z_fin[b, h]) for b, h in heads])[None]
    e_out = oracle.rel_err_rows(g_out, r_out)
    e_M = oracle.rel_err_state(g_M, r_M, (2, 3))
    e_z = oracle.rel_err_state(g_z, r_z, (2,))
    print(f"PARITY workload_segmented out={e_out:.3e} M={e_M:.3e} z={e_z:.3e} (4 sampled heads, 32768 tokens)")
    assert e_out <= TOL_BF16 and e_M <= TOL_BF16 and e_z <= TOL_BF16
    # segment invariance on the GPU: one call over all T
    one = fwd(tq, tk, tv, chunk=w.chunk, eps=w.eps)
    e_one = oracle.rel_err_rows(to_host(one[0]), to_host(out))
    print(f"PARITY workload_segmented_vs_one_call out={e_one:.3e}")
    assert e_one <= TOL_BF16
    # properties over every head: outputs inside the hull of the values seen so far
    vmax = torch.cummax(tv.float().abs(), dim=2).values
    assert bool((out.float().abs() <= vmax * 1.02 + 1e-6).all())


def test_segments_call_full_workload_sampled_heads():
    """The segmented workload as the bench runs it: one la_causal_fwd_segments call over
    B=2, H=32, T=32768 (16 segments of 2048, the bench's workspace), checked on sampled heads
    against the oracle run segment by segment: all 32768 outputs and the state after every
    segment."""
    w = synthetic.WORKLOADS["segmented"]
    q, k, v = synthetic.qkv(w)
    B, H, T, d, dv, S = w.B, w.H, w.T, w.d, w.dv, w.segment
    nseg = T // S
    out = torch.empty(B, H, T, dv, dtype=torch.bfloat16, device="cuda")
    M_seg = torch.full((nseg, B, H, d, dv), float("nan"), device="cuda")
    z_seg = torch.full((nseg, B, H, d), float("nan"), device="cuda")
    nws = la.la_causal_fwd_workspace_size(B, H, T, d, dv, w.chunk, la.LA_BF16)
    ws = torch.empty(max(nws, 256), dtype=torch.uint8, device="cuda")
    la.la_causal_fwd_segments(to_dev(q), to_dev(k), to_dev(v), out, None, None, M_seg, z_seg, B, H, T, d, dv, S,
                              w.eps, la.LA_BF16, ws, nws)
    assert la.la_last_launch_count() == 1
    check_status()
    heads = [(0, 0), (0, 31), (1, 7), (1, 20)]
    sel = lambda a: np.stack([a[b, h] for b, h in heads])[None]
    r_out, r_M, r_z = _segment_refs(sel(q), sel(k), sel(v), None, None, S)
    errs = {"out": oracle.rel_err_rows(np.stack([to_host(out[b, h]) for b, h in heads])[None], r_out)}
    for s in range(nseg):
        g_M = np.stack([to_host(M_seg[s, b, h]) for b, h in heads])[None]
        g_z = np.stack([to_host(z_seg[s, b, h]) for b, h in heads])[None]
        errs[f"M{s}"] = oracle.rel_err_state(g_M, r_M[s], (2, 3))
        errs[f"z{s}"] = oracle.rel_err_state(g_z, r_z[s], (2,))
    worst = max(errs, key=lambda key: errs[key])
    print(f"PARITY workload_segments_call out={errs['out']:.3e} worst={worst}:{errs[worst]:.3e} "
          f"(4 sampled heads, 32768 tokens, 16 segment states)")
    assert all(e <= TOL_BF16 for e in errs.values()), errs
    # every head and segment state was written (no NaN left), and the last segment's is finite
    assert not bool(torch.isnan(M_seg).any()) and not bool(torch.isnan(z_seg).any())


def test_bf16_calls_captured_in_a_cuda_graph_match_eager_calls():
    """Segment calls chained through M, z, captured in one CUDA graph and replayed, give the
    eager calls' results bit for bit (the calls make no synchronising CUDA call)."""
    import compressive_memory_attention_02_b300 as la
    B, H, S, Tseg, d = 2, 4, 3, 256, 128
    q, k, v = _inputs(50, B, H, S * Tseg, d, d, "bf16", 0.5)
    seg = lambda a, s: to_dev(np.ascontiguousarray(a[:, :, s * Tseg:(s + 1) * Tseg]))
    qs, ks, vs = [seg(q, s) for s in range(S)], [seg(k, s) for s in range(S)], [seg(v, s) for s in range(S)]
    nws = la.la_causal_fwd_workspace_size(B, H, Tseg, d, d, 64, la.LA_BF16)
    ws = torch.empty(max(nws, 256), dtype=torch.uint8, device="cuda")

    def run(outs, Ms, zs):
        for s in range(S):
            Mi, zi = (None, None) if s == 0 else (Ms[s - 1], zs[s - 1])
            la.la_causal_fwd_ex(qs[s], ks[s], vs[s], outs[s], Mi, zi, Ms[s], zs[s], B, H, Tseg, d, d, 64, 1e-6,
                                la.LA_BF16, None, ws, nws)

    mk = lambda: ([torch.empty(B, H, Tseg, d, dtype=torch.bfloat16, device="cuda") for _ in range(S)],
                  [torch.empty(B, H, d, d, device="cuda") for _ in range(S)],
                  [torch.empty(B, H, d, device="cuda") for _ in range(S)])
    eager = mk()
    run(*eager)
    torch.cuda.synchronize()
    graphed = mk()
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        run(*graphed)
    g.replay()
    torch.cuda.synchronize()
    assert la.la_get_last_device_status() == la.LA_OK
    for a, b in zip(eager, graphed):
        for x, y in zip(a, b):
            assert torch.equal(x, y)


@pytest.mark.parametrize("chunk", [16, 32, 128])
def test_bf16_any_chunk_length_runs_on_the_tensor_core_path(chunk):
    """The chunk length is a blocking choice: the bf16 tensor-core shapes run the same
    64-token tensor-core kernel for every chunk length (identical results), and match the
    oracle."""
    import compressive_memory_attention_02_b300 as la
    q, k, v = _inputs(51, 1, 3, 700, 128, 128, "bf16", 0.5)
    tq, tk, tv = to_dev(q), to_dev(k), to_dev(v)
    a = fwd(tq, tk, tv, chunk=chunk)
    b = fwd(tq, tk, tv, chunk=64)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    _compare(a, oracle.causal_fwd(q, k, v), TOL_BF16)


# ------------------------------------------------------------------ segment-wise call

def _segments(q, k, v, M0, z0, seg_len, workspace):
    B, H, T, d = q.shape
    dv = v.shape[3]
    nseg = -(-T // seg_len)
    out = torch.empty(B, H, T, dv, dtype=q.dtype, device="cuda")
    M_seg = torch.full((nseg, B, H, d, dv), float("nan"), device="cuda")
    z_seg = torch.full((nseg, B, H, d), float("nan"), device="cuda")
    nws = la.la_causal_fwd_workspace_size(B, H, T, d, dv, 64, dtype_code(q)) if workspace else 0
    ws = torch.empty(max(nws, 256), dtype=torch.uint8, device="cuda") if workspace else None
    la.la_causal_fwd_segments(q, k, v, out, M0, z0, M_seg, z_seg, B, H, T, d, dv, seg_len, 1e-6, dtype_code(q),
                              ws, nws)
    n = la.la_last_launch_count()
    check_status()
    return out, M_seg, z_seg, n


def _segment_refs(q, k, v, M0, z0, seg_len):
    """The oracle run segment by segment, each segment starting from the state the previous
    one ended with: every output and the state after each segment."""
    T = q.shape[2]
    outs, Ms, zs = [], [], []
    M, z = M0, z0
    for t0 in range(0, T, seg_len):
        sl = slice(t0, min(T, t0 + seg_len))
        o, M, z = oracle.causal_fwd(q[:, :, sl], k[:, :, sl], v[:, :, sl], M_in=M, z_in=z)
        outs.append(o), Ms.append(M), zs.append(z)
    return np.concatenate(outs, axis=2), Ms, zs


@pytest.mark.parametrize("d,dv,T,seg_len", [(64, 64, 1000, 192), (128, 128, 700, 256), (64, 128, 640, 64),
                                            (128, 64, 333, 512)])
@pytest.mark.parametrize("workspace", [False, True])
def test_bf16_segments_one_launch(d, dv, T, seg_len, workspace):
    """One launch over all segments (the sequence-split schedules included), the state after
    every segment written, the last segment ragged."""
    B, H = 1, 3
    q, k, v = _inputs(700 + d + dv + T, B, H, T, d, dv, "bf16", 0.5)
    M0, z0 = rand_state(701, B, H, d, dv)
    out, M_seg, z_seg, n = _segments(to_dev(q), to_dev(k), to_dev(v), to_dev(M0), to_dev(z0), seg_len, workspace)
    assert n == (2 if workspace else 1)  # with scratch: the range pre-pass, then the chunked kernel
    r_out, r_M, r_z = _segment_refs(q, k, v, M0, z0, seg_len)
    errs = [oracle.rel_err_rows(to_host(out), r_out)]
    for s in range(len(r_M)):
        errs.append(oracle.rel_err_state(to_host(M_seg[s]), r_M[s], (2, 3)))
        errs.append(oracle.rel_err_state(to_host(z_seg[s]), r_z[s], (2,)))
    print(f"PARITY segments_d{d}_dv{dv}_T{T}_seg{seg_len} max={max(errs):.3e}")
    assert all(e <= TOL_BF16 for e in errs), errs  # (an entry never written stays NaN and fails)


def test_fp32_segments_one_call_per_segment():
    """float32 (and shapes outside the tensor-core set): one la_causal_fwd_ex per segment."""
    B, H, T, d, dv, seg_len = 2, 2, 300, 32, 16, 128
    q, k, v = _inputs(710, B, H, T, d, dv, "f32", 1.0)
    M0, z0 = rand_state(711, B, H, d, dv)
    out, M_seg, z_seg, n = _segments(to_dev(q), to_dev(k), to_dev(v), to_dev(M0), to_dev(z0), seg_len, False)
    assert n == 3
    r_out, r_M, r_z = _segment_refs(q, k, v, M0, z0, seg_len)
    assert oracle.rel_err_rows(to_host(out), r_out) <= TOL_F32
    for s in range(3):
        assert oracle.rel_err_state(to_host(M_seg[s]), r_M[s], (2, 3)) <= TOL_F32
        assert oracle.rel_err_state(to_host(z_seg[s]), r_z[s], (2,)) <= TOL_F32


def test_bf16_segments_outside_the_tensor_core_shapes():
    """bf16 with d, dv outside {64, 128}: one la_causal_fwd_ex per segment (SIMT kernel)."""
    B, H, T, d, dv, seg_len = 1, 2, 200, 32, 16, 64
    q, k, v = _inputs(720, B, H, T, d, dv, "bf16", 0.5)
    M0, z0 = rand_state(721, B, H, d, dv)
    out, M_seg, z_seg, n = _segments(to_dev(q), to_dev(k), to_dev(v), to_dev(M0), to_dev(z0), seg_len, False)
    assert n == 4
    r_out, r_M, r_z = _segment_refs(q, k, v, M0, z0, seg_len)
    errs = [oracle.rel_err_rows(to_host(out), r_out)]
    for s in range(4):
        errs.append(oracle.rel_err_state(to_host(M_seg[s]), r_M[s], (2, 3)))
        errs.append(oracle.rel_err_state(to_host(z_seg[s]), r_z[s], (2,)))
    assert all(e <= TOL_BF16 for e in errs), errs


def test_bf16_segments_in_a_cuda_graph_equal_eager_calls():
    """The one-launch segments call captured in a CUDA graph gives the eager call's bits."""
    B, H, T, d, seg_len = 2, 4, 1024, 128, 256
    q, k, v = (to_dev(a) for a in _inputs(730, B, H, T, d, d, "bf16", 0.5))
    outs = []
    for graph in (False, True):
        out = torch.empty(B, H, T, d, dtype=torch.bfloat16, device="cuda")
        M_seg = torch.empty(T // seg_len, B, H, d, d, device="cuda")
        z_seg = torch.empty(T // seg_len, B, H, d, device="cuda")
        call = lambda: la.la_causal_fwd_segments(q, k, v, out, None, None, M_seg, z_seg, B, H, T, d, d, seg_len,
                                                 1e-6, la.LA_BF16)
        if graph:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                call()  # attributes set and modules loaded outside the capture
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                call()
            out.zero_(), M_seg.zero_(), z_seg.zero_()
            g.replay()
        else:
            call()
        torch.cuda.synchronize()
        check_status()
        outs.append((out.clone(), M_seg.clone(), z_seg.clone()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
@pytest.mark.parametrize("T", [200, 1000])
def test_bf16_fused_state_hand_off(monkeypatch, d, dv, T):
    """The fused two-range schedule with range 0 handing its state after chunk `meet` to range
    1 (forced on short sequences): outputs and final state with an initial state, twice in a row
    (the second call re-arms the hand-off word the first cleared), and through the segments call."""
    monkeypatch.setenv("LA_FWD_PUB_MIN_CHUNKS", "1")
    monkeypatch.setenv("LA_FWD_RANGES", "2")  # the two-range schedule (few heads would take the parts one)
    B, H = 1, 3
    q, k, v = _inputs(740 + d + dv + T, B, H, T, d, dv, "bf16", 0.5)
    M0, z0 = rand_state(741, B, H, d, dv)
    ref = oracle.causal_fwd(q, k, v, M_in=M0, z_in=z0)
    for _ in range(2):
        got = fwd(to_dev(q), to_dev(k), to_dev(v), to_dev(M0), to_dev(z0))
        check_status()
        _compare(got, ref, TOL_BF16)
    out, M_seg, z_seg, n = _segments(to_dev(q), to_dev(k), to_dev(v), to_dev(M0), to_dev(z0), 128, True)
    assert n == 1
    r_out, r_M, r_z = _segment_refs(q, k, v, M0, z0, 128)
    errs = [oracle.rel_err_rows(to_host(out), r_out)]
    for s in range(len(r_M)):
        errs.append(oracle.rel_err_state(to_host(M_seg[s]), r_M[s], (2, 3)))
        errs.append(oracle.rel_err_state(to_host(z_seg[s]), r_z[s], (2,)))
    print(f"PARITY hand_off_d{d}_dv{dv}_T{T} max={max(errs):.3e}")
    assert all(e <= TOL_BF16 for e in errs), errs


def test_bf16_hand_off_long_ragged_segments(monkeypatch):
    """The hand-off at its default threshold (313 chunks): a 20000-token sequence in segments of
    2048 (the last one 1568 tokens) with an initial state, two ranges per head."""
    monkeypatch.setenv("LA_FWD_RANGES", "2")
    B, H, T, d, seg_len = 1, 2, 20000, 128, 2048
    q, k, v = _inputs(760, B, H, T, d, d, "bf16", 0.5)
    M0, z0 = rand_state(761, B, H, d, d)
    out, M_seg, z_seg, n = _segments(to_dev(q), to_dev(k), to_dev(v), to_dev(M0), to_dev(z0), seg_len, True)
    assert n == 1
    r_out, r_M, r_z = _segment_refs(q, k, v, M0, z0, seg_len)
    errs = [oracle.rel_err_rows(to_host(out), r_out)]
    for s in range(len(r_M)):
        errs.append(oracle.rel_err_state(to_host(M_seg[s]), r_M[s], (2, 3)))
        errs.append(oracle.rel_err_state(to_host(z_seg[s]), r_z[s], (2,)))
    print(f"PARITY hand_off_long_ragged max={max(errs):.3e} ({len(r_M)} segments)")
    assert all(e <= TOL_BF16 for e in errs), errs
