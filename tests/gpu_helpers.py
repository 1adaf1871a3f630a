"""Shared plumbing of the GPU parity tests: storage arrays <-> device tensors and
thin wrappers that call the library through its C ABI (via the binding)."""
from __future__ import annotations

import numpy as np
import torch

import compressive_memory_attention_02_b300 as la

TOL_F32 = 1e-4   # max row-normwise relative error, float32 path
TOL_BF16 = 2e-2  # bf16 inputs, float32 state


def to_dev(a: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def dtype_code(t: torch.Tensor) -> int:
    return la.LA_BF16 if t.dtype == torch.bfloat16 else la.LA_F32


def check_status():
    torch.cuda.synchronize()
    assert la.la_get_last_device_status() == la.LA_OK


def fwd(q, k, v, M_in=None, z_in=None, chunk=64, eps=1e-6, workspace=True, out=None, M_out=None, z_out=None,
        strides=None, T=None):
    """la_causal_fwd_ex on device tensors [B,H,T,d]; returns (out, M_out, z_out)."""
    B, H = q.shape[0], q.shape[1]
    T = q.shape[2] if T is None else T
    d, dv = q.shape[3], v.shape[3]
    dt = dtype_code(q)
    if out is None:
        out = torch.empty(B, H, T, dv, dtype=q.dtype, device=q.device)
    if M_out is None:
        M_out = torch.empty(B, H, d, dv, dtype=torch.float32, device=q.device)
    if z_out is None:
        z_out = torch.empty(B, H, d, dtype=torch.float32, device=q.device)
    ws, nws = None, 0
    if workspace:
        nws = la.la_causal_fwd_workspace_size(B, H, T, d, dv, chunk, dt)
        ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=q.device)
    la.la_causal_fwd_ex(q, k, v, out, M_in, z_in, M_out, z_out, B, H, T, d, dv, chunk, eps, dt, strides, ws, nws)
    check_status()
    return out, M_out, z_out


def prefill(q, k, v, M_in=None, z_in=None, segment=0, eps=1e-6, workspace=True, want_out=True,
            want_M=True, want_z=True):
    B, H, T, d = q.shape
    dv = v.shape[3]
    dt = dtype_code(q)
    out = torch.empty(B, H, dv, dtype=q.dtype, device=q.device) if want_out else None
    M_out = torch.empty(B, H, d, dv, dtype=torch.float32, device=q.device) if want_M else None
    z_out = torch.empty(B, H, d, dtype=torch.float32, device=q.device) if want_z else None
    ws, nws = None, 0
    if workspace:
        nws = la.la_prefill_workspace_size(B, H, T, d, dv, segment, dt)
        ws = torch.empty(max(nws, 256), dtype=torch.uint8, device=q.device)
    la.la_prefill_state_ex(q, k, v, out, M_in, z_in, M_out, z_out, B, H, T, d, dv, segment, eps, dt, None, ws, nws)
    check_status()
    return out, M_out, z_out


def decode(q, k, v, M, z, eps=1e-6, out=None):
    N, H, d = q.shape
    dv = v.shape[2]
    if out is None:
        out = torch.empty(N, H, dv, dtype=q.dtype, device=q.device)
    la.la_decode_step(q, k, v, out, M, z, N, H, d, dv, eps, dtype_code(q))
    return out


def rand_state(seed, B, H, d, dv, scale=1.0):
    rng = np.random.default_rng(seed)
    M = rng.normal(size=(B, H, d, dv)) * scale
    z = rng.uniform(0.5, 2.0, size=(B, H, d)) * scale * 10
    return M.astype(np.float32), z.astype(np.float32)
