"""Run one mode of the library a few times on seeded inputs, for profilers.

  python -m compressive_memory_attention_02_b300.profile_case --mode fwd --B 2 --H 32 --T 2048 --repeat 3

Modes: fwd (la_causal_fwd, training forward), segments (la_causal_fwd_segments:
the sequence as segments of --segment tokens, the state written after each), bwd
(la_causal_bwd, training backward with dout ~ N(0,1)), prefill (la_prefill_state),
decode (la_decode_step on a [B, H] batch of one-token streams with a random state). Inputs are the seeded synthetic N(0,1)*0.5 bf16 values; the call's
workspace is registered before the first launch.
"""
from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--mode", default="fwd", choices=["fwd", "segments", "bwd", "prefill", "decode"])
    ap.add_argument("--B", type=int, default=2)
    ap.add_argument("--H", type=int, default=32)
    ap.add_argument("--T", type=int, default=2048)
    ap.add_argument("--d", type=int, default=128)
    ap.add_argument("--dv", type=int, default=128)
    ap.add_argument("--segment", type=int, default=4096)
    ap.add_argument("--repeat", type=int, default=3)
    a = ap.parse_args()

    import torch

    import compressive_memory_attention_02_b300 as la
    import synthetic

    dev = torch.device("cuda", 0)
    bf = lambda x: torch.from_numpy(x).view(torch.bfloat16).to(dev)
    if a.mode == "decode":
        q = bf(synthetic.normal(1, 3, (a.B, a.H, a.d), 0.5, "bf16"))
        k = bf(synthetic.normal(1, 4, (a.B, a.H, a.d), 0.5, "bf16"))
        v = bf(synthetic.normal(1, 5, (a.B, a.H, a.dv), 0.5, "bf16"))
        M = torch.randn(a.B, a.H, a.d, a.dv, device=dev)
        z = torch.rand(a.B, a.H, a.d, device=dev) * 100 + 1
        out = torch.empty(a.B, a.H, a.dv, dtype=torch.bfloat16, device=dev)
        for _ in range(a.repeat):
            la.la_decode_step(q, k, v, out, M, z, a.B, a.H, a.d, a.dv, 1e-6, la.LA_BF16)
    else:
        q = bf(synthetic.normal(1, 0, (a.B, a.H, a.T, a.d), 0.5, "bf16"))
        k = bf(synthetic.normal(1, 1, (a.B, a.H, a.T, a.d), 0.5, "bf16"))
        v = bf(synthetic.normal(1, 2, (a.B, a.H, a.T, a.dv), 0.5, "bf16"))
        M = torch.empty(a.B, a.H, a.d, a.dv, device=dev)
        z = torch.empty(a.B, a.H, a.d, device=dev)
        if a.mode == "bwd":
            dout = bf(synthetic.normal(1, 7, (a.B, a.H, a.T, a.dv), 1.0, "bf16"))
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            la.ensure_workspace(la.la_causal_bwd_workspace_size(a.B, a.H, a.T, a.d, a.dv))
            for _ in range(a.repeat):
                la.la_causal_bwd(q, k, v, dout, None, None, None, None, dq, dk, dv, M, z, a.B, a.H, a.T, a.d, a.dv,
                                 1e-6, la.LA_BF16)
        elif a.mode == "fwd":
            out = torch.empty(a.B, a.H, a.T, a.dv, dtype=torch.bfloat16, device=dev)
            la.ensure_workspace(la.la_causal_fwd_workspace_size(a.B, a.H, a.T, a.d, a.dv, 64, la.LA_BF16))
            for _ in range(a.repeat):
                la.la_causal_fwd(q, k, v, out, None, None, M, z, a.B, a.H, a.T, a.d, a.dv, 64, 1e-6, la.LA_BF16)
        elif a.mode == "segments":
            out = torch.empty(a.B, a.H, a.T, a.dv, dtype=torch.bfloat16, device=dev)
            nseg = -(-a.T // a.segment)
            M_seg = torch.empty(nseg, a.B, a.H, a.d, a.dv, device=dev)
            z_seg = torch.empty(nseg, a.B, a.H, a.d, device=dev)
            nws = la.la_causal_fwd_workspace_size(a.B, a.H, a.T, a.d, a.dv, 64, la.LA_BF16)
            ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=dev)
            for _ in range(a.repeat):
                la.la_causal_fwd_segments(q, k, v, out, None, None, M_seg, z_seg, a.B, a.H, a.T, a.d, a.dv,
                                          a.segment, 1e-6, la.LA_BF16, ws, nws)
        else:
            out = torch.empty(a.B, a.H, a.dv, dtype=torch.bfloat16, device=dev)
            la.ensure_workspace(la.la_prefill_workspace_size(a.B, a.H, a.T, a.d, a.dv, a.segment, la.LA_BF16))
            for _ in range(a.repeat):
                la.la_prefill_state(q, k, v, out, None, None, M, z, a.B, a.H, a.T, a.d, a.dv, a.segment, 1e-6,
                                    la.LA_BF16)
    torch.cuda.synchronize()
    rc = la.la_get_last_device_status()
    print(f"{a.mode} done, device status {rc}")
    return 0 if rc == 0 else 1


if __name__ == "__main__":
    sys.exit(main())
