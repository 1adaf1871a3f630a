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
