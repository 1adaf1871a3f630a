"""The state is the checkpoint: (M, z) after any call resumes the stream exactly, also
after a round trip through host memory (the segment carry of the "Segment-Wise
Attention" page). And the cost is linear in the sequence: the forward's time grows in
proportion to T (the linear compute and storage bounds of the page
"Attention_Kernel_Mask", comparison table), while its workspace does not grow with T."""
import time

import numpy as np
import pytest

import compressive_memory_attention_02_b300 as la
import synthetic


def test_forward_workspace_does_not_grow_with_T():
    sizes = [la.la_causal_fwd_workspace_size(2, 32, T, 128, 128, 64, la.LA_BF16) for T in (4096, 32768, 262144)]
    assert sizes[0] == sizes[1] == sizes[2]


@pytest.mark.gpu
def test_state_round_trip_through_host_resumes_exactly():
    import torch
    from gpu_helpers import fwd, to_dev
    B, H, S, d = 2, 4, 512, 128
    q = synthetic.normal(91, 0, (B, H, 4 * S, d), 0.5, "bf16")
    k = synthetic.normal(91, 1, (B, H, 4 * S, d), 0.5, "bf16")
    v = synthetic.normal(91, 2, (B, H, 4 * S, d), 0.5, "bf16")
    seg = lambda a, s: to_dev(np.ascontiguousarray(a[:, :, s * S:(s + 1) * S]))
    outs_dev, outs_host = [], []
    M = z = None
    Mh = zh = None
    for s in range(4):
        o, M, z = fwd(seg(q, s), seg(k, s), seg(v, s), M, z)
        outs_dev.append(o)
        # the same chain, with the state checkpointed to host memory and restored between segments
        Md = None if Mh is None else torch.from_numpy(Mh).cuda()
        zd = None if zh is None else torch.from_numpy(zh).cuda()
        o2, M2, z2 = fwd(seg(q, s), seg(k, s), seg(v, s), Md, zd)
        outs_host.append(o2)
        Mh, zh = M2.cpu().numpy().copy(), z2.cpu().numpy().copy()
    for a, b in zip(outs_dev, outs_host):
        assert torch.equal(a, b)
    assert np.array_equal(M.cpu().numpy(), Mh) and np.array_equal(z.cpu().numpy(), zh)


@pytest.mark.gpu
def test_forward_time_is_linear_in_T():
    import torch
    B, H, d = 2, 32, 128
    ws = la.ensure_workspace(la.la_causal_fwd_workspace_size(B, H, 32768, d, d, 64, la.LA_BF16))
    times = {}
    for T in (4096, 32768):
        g = torch.Generator(device="cuda").manual_seed(T)
        q, k, v = ((torch.randn(B, H, T, d, device="cuda", generator=g) * 0.5).bfloat16() for _ in range(3))
        out = torch.empty_like(q)
        M = torch.empty(B, H, d, d, device="cuda")
        z = torch.empty(B, H, d, device="cuda")
        call = lambda: la.la_causal_fwd(q, k, v, out, None, None, M, z, B, H, T, d, d, 64, 1e-6, la.LA_BF16)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(5):
            call()
        e1.record()
        torch.cuda.synchronize()
        times[T] = e0.elapsed_time(e1) / 5
    assert la.la_get_last_device_status() == la.LA_OK
    ratio = times[32768] / times[4096]
    assert 5.0 <= ratio <= 10.0, (times, ratio)   # 8x the tokens: linear, with a fixed cost per call
    del ws
