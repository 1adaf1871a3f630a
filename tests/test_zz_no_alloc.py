"""la_prefill_state_noalloc: the prefill entry point for callers that cannot allocate
device memory (a host that hands the operator only its input and output buffers, or
code that must not call cudaMalloc because it can synchronise the device). Its
multi-part scratch is a fixed-size device array inside the library.

This file is collected last on purpose: if it fails, a run that stops at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import compressive_memory_attention_02_b300 as la
import synthetic


def test_rejects_problems_beyond_the_static_scratch_without_touching_the_device():
    # 256 parts x 8 heads of d = dv = 128 need about 136 MB of scratch: more than the array holds
    need = la.la_prefill_workspace_size(1, 8, 1 << 20, 128, 128, 4096, la.LA_BF16)
    assert need > la.LA_NOALLOC_SCRATCH_BYTES
    rc = la.lib.la_prefill_state_noalloc(16, 32, 48, 64, None, None, None, None, 1, 8, 1 << 20, 128, 128, 4096,
                                         1e-6, la.LA_BF16, None)
    assert rc == la.LA_ERR_SCRATCH_LIMIT
    assert "static buffer" in la.error_string(rc)
    assert la.lib.la_last_launch_count() == 0


def test_limit_counts_only_the_scratch_the_call_uses():
    # host-side decisions only (fake device addresses): nothing here reaches a device
    rec = 4 * (128 * 128 + 128)            # bytes of one part's state sum for one head
    H, seg = 4, 64
    # 126 parts + a final state per head: 4 * 127 records, just under the limit
    T = 126 * seg
    need = la.la_prefill_workspace_size(1, H, T, 128, 128, seg, la.LA_BF16)
    assert need == H * 127 * rec <= la.LA_NOALLOC_SCRATCH_BYTES
    # 127 parts + a final state: 4 * 128 records, just over
    T2 = 127 * seg
    assert la.la_prefill_workspace_size(1, H, T2, 128, 128, seg, la.LA_BF16) > la.LA_NOALLOC_SCRATCH_BYTES
    rc = la.lib.la_prefill_state_noalloc(16, 32, 48, 64, None, None, None, None, 1, H, T2, 128, 128, seg, 1e-6,
                                         la.LA_BF16, None)
    assert rc == la.LA_ERR_SCRATCH_LIMIT and la.lib.la_last_launch_count() == 0
    # nothing requested: returns at once, without a launch
    rc = la.lib.la_prefill_state_noalloc(16, 32, 48, None, None, None, None, None, 1, H, T2, 128, 128, seg, 1e-6,
                                         la.LA_BF16, None)
    assert rc == la.LA_OK and la.lib.la_last_launch_count() == 0


def test_misaligned_state_is_an_argument_error_before_any_launch():
    # the parts are summed in 16-byte vectors: a state pointer off a 16-byte boundary is
    # refused on the host (fake device addresses: the check comes before any CUDA call)
    for M_in, z_in, M_out, z_out in ((4100, None, None, None), (None, 8196, None, None),
                                     (None, None, 12292, 16384), (None, None, 16384, 20484)):
        for fn in (la.lib.la_prefill_state, la.lib.la_prefill_state_noalloc):
            rc = fn(256, 512, 768, 1024, M_in, z_in, M_out, z_out, 1, 2, 3000, 128, 128, 512, 1e-6,
                    la.LA_BF16, None)
            assert rc == la.LA_ERR_INVALID_ARG, (fn, M_in, z_in, M_out, z_out)
            assert la.lib.la_last_launch_count() == 0


def _inputs(seed, B, H, T, d, dv):
    q = synthetic.normal(seed, 0, (B, H, T, d), 0.5, "bf16")
    k = synthetic.normal(seed, 1, (B, H, T, d), 0.5, "bf16")
    v = synthetic.normal(seed, 2, (B, H, T, dv), 0.5, "bf16")
    dev = lambda a: torch.from_numpy(a).view(torch.bfloat16).cuda()
    return dev(q), dev(k), dev(v)


def _rel_rows(a, b):
    a, b = a.double().cpu(), b.double().cpu()
    den = b.abs().amax(dim=-1).clamp_min(1e-30)
    return float(((a - b).abs().amax(dim=-1) / den).max())


@pytest.mark.gpu
def test_noalloc_prefill_matches_workspace_prefill_on_two_calls_in_a_row():
    from gpu_helpers import TOL_BF16
    B, H, T, d, dv, seg = 2, 4, 3000, 128, 128, 512      # 6 parts per head
    assert la.la_prefill_workspace_size(B, H, T, d, dv, seg, la.LA_BF16) <= la.LA_NOALLOC_SCRATCH_BYTES
    rng = np.random.default_rng(3)
    M0 = torch.from_numpy(rng.normal(size=(B, H, d, dv)).astype(np.float32)).cuda()
    z0 = torch.from_numpy(rng.uniform(5, 20, size=(B, H, d)).astype(np.float32)).cuda()

    def reference(q, k, v, M_in, z_in, want_state):
        out = torch.empty(B, H, dv, dtype=torch.bfloat16, device="cuda")
        M = torch.empty(B, H, d, dv, device="cuda") if want_state else None
        z = torch.empty(B, H, d, device="cuda") if want_state else None
        nws = la.la_prefill_workspace_size(B, H, T, d, dv, seg, la.LA_BF16)
        ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
        la.la_prefill_state_ex(q, k, v, out, M_in, z_in, M, z, B, H, T, d, dv, seg, 1e-6, la.LA_BF16, None, ws, nws)
        return out, M, z

    # call 1: initial state in, last output and final state out
    q, k, v = _inputs(61, B, H, T, d, dv)
    out1 = torch.empty(B, H, dv, dtype=torch.bfloat16, device="cuda")
    M1 = torch.empty(B, H, d, dv, device="cuda")
    z1 = torch.empty(B, H, d, device="cuda")
    la.la_prefill_state_noalloc(q, k, v, out1, M0, z0, M1, z1, B, H, T, d, dv, seg, 1e-6, la.LA_BF16)
    torch.cuda.synchronize()
    assert la.la_get_last_device_status() == la.LA_OK
    r_out, r_M, r_z = reference(q, k, v, M0, z0, True)
    torch.cuda.synchronize()
    assert _rel_rows(out1, r_out) <= TOL_BF16
    assert _rel_rows(M1.flatten(2), r_M.flatten(2)) <= TOL_BF16
    assert _rel_rows(z1, r_z) <= TOL_BF16

    # call 2, right after: other inputs, no initial state, last output only (the final
    # state then also lives in the static scratch); no device memory may be taken
    q2, k2, v2 = _inputs(62, B, H, T, d, dv)
    out2 = torch.empty(B, H, dv, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    la.la_prefill_state_noalloc(q2, k2, v2, out2, None, None, None, None, B, H, T, d, dv, seg, 1e-6, la.LA_BF16)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free_before
    assert la.la_get_last_device_status() == la.LA_OK
    r_out2, _, _ = reference(q2, k2, v2, None, None, False)
    torch.cuda.synchronize()
    assert _rel_rows(out2, r_out2) <= TOL_BF16
    # the second call did not reuse anything from the first
    assert _rel_rows(out2, r_out) > TOL_BF16


def _workspace_prefill(q, k, v, M_in, z_in, want_state, seg):
    B, H, T, d = q.shape
    dv = v.shape[3]
    out = torch.empty(B, H, dv, dtype=torch.bfloat16, device="cuda")
    M = torch.empty(B, H, d, dv, device="cuda") if want_state else None
    z = torch.empty(B, H, d, device="cuda") if want_state else None
    nws = la.la_prefill_workspace_size(B, H, T, d, dv, seg, la.LA_BF16)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    la.la_prefill_state_ex(q, k, v, out, M_in, z_in, M, z, B, H, T, d, dv, seg, 1e-6, la.LA_BF16, None, ws, nws)
    torch.cuda.synchronize()
    return out, M, z


@pytest.mark.gpu
def test_noalloc_prefill_in_place_state_and_scratch_at_the_limit():
    from gpu_helpers import TOL_BF16
    # 4 heads x 126 parts of 64 tokens, last output only: parts plus final state fill the
    # static array to within 2 KB of its end
    B, H, d, dv, seg = 1, 4, 128, 128, 64
    T = 126 * seg
    assert la.la_prefill_workspace_size(B, H, T, d, dv, seg, la.LA_BF16) > la.LA_NOALLOC_SCRATCH_BYTES - 4096
    q, k, v = _inputs(63, B, H, T, d, dv)
    out = torch.empty(B, H, dv, dtype=torch.bfloat16, device="cuda")
    la.la_prefill_state_noalloc(q, k, v, out, None, None, None, None, B, H, T, d, dv, seg, 1e-6, la.LA_BF16)
    torch.cuda.synchronize()
    assert la.la_get_last_device_status() == la.LA_OK
    r_out, _, _ = _workspace_prefill(q, k, v, None, None, False, seg)
    assert _rel_rows(out, r_out) <= TOL_BF16

    # the state updated in place (M_out is M_in, z_out is z_in), 6 parts per head
    B, H, T, seg = 2, 4, 3000, 512
    rng = np.random.default_rng(4)
    M0 = torch.from_numpy(rng.normal(size=(B, H, d, dv)).astype(np.float32)).cuda()
    z0 = torch.from_numpy(rng.uniform(5, 20, size=(B, H, d)).astype(np.float32)).cuda()
    q, k, v = _inputs(64, B, H, T, d, dv)
    r_out, r_M, r_z = _workspace_prefill(q, k, v, M0, z0, True, seg)
    Mi, zi = M0.clone(), z0.clone()
    out = torch.empty(B, H, dv, dtype=torch.bfloat16, device="cuda")
    la.la_prefill_state_noalloc(q, k, v, out, Mi, zi, Mi, zi, B, H, T, d, dv, seg, 1e-6, la.LA_BF16)
    torch.cuda.synchronize()
    assert la.la_get_last_device_status() == la.LA_OK
    assert _rel_rows(out, r_out) <= TOL_BF16
    assert torch.equal(Mi, r_M) and torch.equal(zi, r_z)   # same kernels, same order: bit for bit


@pytest.mark.gpu
def test_noalloc_prefill_that_needs_no_scratch_runs_beyond_the_array_size():
    from gpu_helpers import TOL_BF16
    # one part per head and the final state into M_out, z_out: no scratch at all, though
    # the workspace size (which also counts a final state) is four times the array
    B, H, T, d, dv, seg = 64, 32, 2048, 128, 128, 4096
    assert la.la_prefill_workspace_size(B, H, T, d, dv, seg, la.LA_BF16) > 4 * la.LA_NOALLOC_SCRATCH_BYTES
    q, k, v = _inputs(65, B, H, T, d, dv)
    out = torch.empty(B, H, dv, dtype=torch.bfloat16, device="cuda")
    M = torch.empty(B, H, d, dv, device="cuda")
    z = torch.empty(B, H, d, device="cuda")
    rc = la.lib.la_prefill_state_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), None, None,
                                         M.data_ptr(), z.data_ptr(), B, H, T, d, dv, seg, 1e-6, la.LA_BF16, None)
    assert rc == la.LA_OK
    torch.cuda.synchronize()
    assert la.la_get_last_device_status() == la.LA_OK
    r_out, r_M, r_z = _workspace_prefill(q, k, v, None, None, True, seg)
    assert _rel_rows(out, r_out) <= TOL_BF16
    assert torch.equal(M, r_M) and torch.equal(z, r_z)
