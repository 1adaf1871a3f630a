"""Python binding of liblinattn.so: causal linear attention (phi = elu + 1) on B300.

Argument marshalling only. Every function has the name and argument order of
the C entry point it wraps (include/linattn.h); tensors are passed as torch
tensors (their device pointers are taken) or as raw integer addresses, None is
NULL, and `stream` defaults to torch's current stream on the tensors' device.
Every step of the computation runs in the library's CUDA kernels; there is no
other implementation here, and importing fails loudly if the library is missing.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
# LA_CHECKED=1 loads the checked library (device-side bounds checks, see la_checked_build)
LIB_PATH = os.path.join(_HERE, "liblinattn_checked.so" if os.environ.get("LA_CHECKED") == "1" else "liblinattn.so")

LA_F32, LA_BF16 = 0, 1
LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_TIMEOUT, LA_ERR_WORKSPACE = range(6)
LA_ERR_SCRATCH_LIMIT = 6
LA_ERR_BOUNDS = 7
LA_NOALLOC_SCRATCH_BYTES = 32 << 20  # size of the library's static prefill scratch

EXPORTS = (
    "la_causal_fwd", "la_causal_fwd_ex", "la_causal_fwd_workspace_size",
    "la_prefill_state", "la_prefill_state_ex", "la_prefill_workspace_size", "la_prefill_state_noalloc",
    "la_decode_step", "la_causal_bwd", "la_causal_bwd_ex", "la_causal_bwd_workspace_size",
    "la_set_workspace", "la_get_last_device_status",
    "la_get_error_string", "la_last_launch_count", "la_selftest_wait_timeout", "la_checked_build",
    "la_feature_map_prf", "la_causal_fwd_mapped", "la_causal_fwd_segments",
)


class LinAttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({error_string(code)})")
        self.code = code


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python -m compressive_memory_attention_02_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    i64p = ctypes.POINTER(ctypes.c_int64)
    fwd = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i64, i32, i32, i32, f32, i32]
    lib.la_causal_fwd.argtypes = fwd + [vp]
    lib.la_causal_fwd_ex.argtypes = fwd + [i64p, vp, sz, vp]
    lib.la_causal_fwd_mapped.argtypes = fwd + [i64p, vp, sz, vp]
    lib.la_feature_map_prf.argtypes = [vp, vp, vp, i64, i32, i32, i32, vp]
    lib.la_causal_fwd_segments.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i64, i32, i32, i64, f32, i32,
                                           vp, sz, vp]
    lib.la_causal_fwd_workspace_size.argtypes = [i32, i32, i64, i32, i32, i32, i32]
    lib.la_causal_fwd_workspace_size.restype = sz
    lib.la_prefill_state.argtypes = fwd + [vp]
    lib.la_prefill_state_ex.argtypes = fwd + [i64p, vp, sz, vp]
    lib.la_prefill_state_noalloc.argtypes = fwd + [vp]
    lib.la_prefill_workspace_size.argtypes = [i32, i32, i64, i32, i32, i32, i32]
    lib.la_prefill_workspace_size.restype = sz
    lib.la_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, i32, vp]
    bwd = [vp] * 13 + [i32, i32, i64, i32, i32, f32, i32]
    lib.la_causal_bwd.argtypes = bwd + [vp]
    lib.la_causal_bwd_ex.argtypes = bwd + [vp, sz, vp]
    lib.la_causal_bwd_workspace_size.argtypes = [i32, i32, i64, i32, i32]
    lib.la_causal_bwd_workspace_size.restype = sz
    lib.la_set_workspace.argtypes = [vp, sz]
    lib.la_get_last_device_status.argtypes = [vp]
    lib.la_get_error_string.argtypes = [i32]
    lib.la_get_error_string.restype = ctypes.c_char_p
    lib.la_last_launch_count.argtypes = []
    lib.la_checked_build.argtypes = []
    lib.la_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, vp]
    for name in EXPORTS:
        f = getattr(lib, name)
        if f.restype is ctypes.c_int or f.restype is None:
            f.restype = i32
    lib.la_causal_fwd_workspace_size.restype = sz
    lib.la_prefill_workspace_size.restype = sz
    lib.la_causal_bwd_workspace_size.restype = sz
    lib.la_get_error_string.restype = ctypes.c_char_p
    return lib


lib = _load()


def error_string(code: int) -> str:
    return lib.la_get_error_string(int(code)).decode()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream, *tensors):
    if stream is None:
        import torch
        dev = next((t.device for t in tensors if hasattr(t, "device") and t.device.type == "cuda"), None)
        return torch.cuda.current_stream(dev).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype(dtype, *tensors):
    if dtype is not None:
        return int(dtype)
    import torch
    t = next(t for t in tensors if hasattr(t, "dtype"))
    return LA_BF16 if t.dtype == torch.bfloat16 else LA_F32


def _check(fn, rc):
    if rc != LA_OK:
        raise LinAttnError(fn, rc)
    return rc


def _strides(strides):
    if strides is None:
        return None
    arr = (ctypes.c_int64 * 12)(*[int(s) for s in strides])
    return arr


def la_causal_fwd(q, k, v, out, M_in, z_in, M_out, z_out, B, H, T, d, dv, chunk, eps,
                  dtype=None, stream=None):
    rc = lib.la_causal_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(M_in), _ptr(z_in), _ptr(M_out),
                           _ptr(z_out), B, H, T, d, dv, chunk, eps, _dtype(dtype, q), _stream(stream, q))
    return _check("la_causal_fwd", rc)


def la_causal_fwd_ex(q, k, v, out, M_in, z_in, M_out, z_out, B, H, T, d, dv, chunk, eps,
                     dtype=None, strides=None, workspace=None, workspace_bytes=0, stream=None):
    rc = lib.la_causal_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(M_in), _ptr(z_in), _ptr(M_out),
                              _ptr(z_out), B, H, T, d, dv, chunk, eps, _dtype(dtype, q), _strides(strides),
                              _ptr(workspace), int(workspace_bytes), _stream(stream, q))
    return _check("la_causal_fwd_ex", rc)


def la_causal_fwd_mapped(q, k, v, out, M_in, z_in, M_out, z_out, B, H, T, d, dv, chunk, eps,
                         dtype=None, strides=None, workspace=None, workspace_bytes=0, stream=None):
    rc = lib.la_causal_fwd_mapped(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(M_in), _ptr(z_in), _ptr(M_out),
                                  _ptr(z_out), B, H, T, d, dv, chunk, eps, _dtype(dtype, q), _strides(strides),
                                  _ptr(workspace), int(workspace_bytes), _stream(stream, q))
    return _check("la_causal_fwd_mapped", rc)


def la_causal_fwd_segments(q, k, v, out, M_in, z_in, M_seg, z_seg, B, H, T, d, dv, seg_len, eps,
                           dtype=None, workspace=None, workspace_bytes=0, stream=None):
    rc = lib.la_causal_fwd_segments(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(M_in), _ptr(z_in), _ptr(M_seg),
                                    _ptr(z_seg), B, H, T, d, dv, seg_len, eps, _dtype(dtype, q),
                                    _ptr(workspace), int(workspace_bytes), _stream(stream, q))
    return _check("la_causal_fwd_segments", rc)


def la_feature_map_prf(x, W, out, rows, d, m, dtype=None, stream=None):
    rc = lib.la_feature_map_prf(_ptr(x), _ptr(W), _ptr(out), rows, d, m, _dtype(dtype, x), _stream(stream, x))
    return _check("la_feature_map_prf", rc)


def la_causal_fwd_workspace_size(B, H, T, d, dv, chunk, dtype) -> int:
    return int(lib.la_causal_fwd_workspace_size(B, H, T, d, dv, chunk, int(dtype)))


def la_prefill_state(q, k, v, out_last, M_in, z_in, M_out, z_out, B, H, T, d, dv, segment, eps,
                     dtype=None, stream=None):
    rc = lib.la_prefill_state(_ptr(q), _ptr(k), _ptr(v), _ptr(out_last), _ptr(M_in), _ptr(z_in), _ptr(M_out),
                              _ptr(z_out), B, H, T, d, dv, segment, eps, _dtype(dtype, q), _stream(stream, q))
    return _check("la_prefill_state", rc)


def la_prefill_state_ex(q, k, v, out_last, M_in, z_in, M_out, z_out, B, H, T, d, dv, segment, eps,
                        dtype=None, strides=None, workspace=None, workspace_bytes=0, stream=None):
    rc = lib.la_prefill_state_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out_last), _ptr(M_in), _ptr(z_in),
                                 _ptr(M_out), _ptr(z_out), B, H, T, d, dv, segment, eps, _dtype(dtype, q),
                                 _strides(strides), _ptr(workspace), int(workspace_bytes), _stream(stream, q))
    return _check("la_prefill_state_ex", rc)


def la_prefill_state_noalloc(q, k, v, out_last, M_in, z_in, M_out, z_out, B, H, T, d, dv, segment, eps,
                             dtype=None, stream=None):
    """Prefill whose multi-part scratch is the library's own static device buffer
    (LA_NOALLOC_SCRATCH_BYTES): nothing is allocated, by the library or here."""
    rc = lib.la_prefill_state_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out_last), _ptr(M_in), _ptr(z_in),
                                      _ptr(M_out), _ptr(z_out), B, H, T, d, dv, segment, eps, _dtype(dtype, q),
                                      _stream(stream, q))
    return _check("la_prefill_state_noalloc", rc)


def la_prefill_workspace_size(B, H, T, d, dv, segment, dtype) -> int:
    return int(lib.la_prefill_workspace_size(B, H, T, d, dv, segment, int(dtype)))


def la_decode_step(q, k, v, out, M, z, N, H, d, dv, eps, dtype=None, stream=None):
    rc = lib.la_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(M), _ptr(z), N, H, d, dv, eps,
                            _dtype(dtype, q), _stream(stream, q))
    return _check("la_decode_step", rc)


def la_causal_bwd(q, k, v, dout, M_in, z_in, dM_out, dz_out, dq, dk, dv, dM_in, dz_in, B, H, T, d, dv_dim, eps,
                  dtype=None, stream=None):
    rc = lib.la_causal_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(M_in), _ptr(z_in), _ptr(dM_out),
                           _ptr(dz_out), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dM_in), _ptr(dz_in), B, H, T, d, dv_dim,
                           eps, _dtype(dtype, q), _stream(stream, q))
    return _check("la_causal_bwd", rc)


def la_causal_bwd_ex(q, k, v, dout, M_in, z_in, dM_out, dz_out, dq, dk, dv, dM_in, dz_in, B, H, T, d, dv_dim, eps,
                     dtype=None, workspace=None, workspace_bytes=0, stream=None):
    rc = lib.la_causal_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(M_in), _ptr(z_in), _ptr(dM_out),
                              _ptr(dz_out), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dM_in), _ptr(dz_in), B, H, T, d,
                              dv_dim, eps, _dtype(dtype, q), _ptr(workspace), int(workspace_bytes),
                              _stream(stream, q))
    return _check("la_causal_bwd_ex", rc)


def la_causal_bwd_workspace_size(B, H, T, d, dv) -> int:
    return int(lib.la_causal_bwd_workspace_size(B, H, T, d, dv))


def la_set_workspace(ptr, nbytes):
    return _check("la_set_workspace", lib.la_set_workspace(_ptr(ptr), int(nbytes)))


def la_get_last_device_status(stream=None) -> int:
    return int(lib.la_get_last_device_status(_stream(stream) if stream is not None else None))


def la_get_error_string(code: int) -> str:
    return error_string(code)


def la_selftest_wait_timeout(limit_cycles, stream=None):
    return _check("la_selftest_wait_timeout",
                  lib.la_selftest_wait_timeout(int(limit_cycles), _stream(stream) if stream is not None else None))


def la_last_launch_count() -> int:
    return int(lib.la_last_launch_count())


def la_checked_build() -> int:
    return int(lib.la_checked_build())


_workspaces = {}


def ensure_workspace(nbytes: int, device=None):
    """Register a torch-allocated scratch buffer of at least nbytes with the library for
    `device` (current device by default); kept alive here and grown when needed.
    Call outside CUDA-graph capture."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else torch.device(device).index)
    cur = _workspaces.get(dev.index)
    if cur is not None and cur.numel() >= nbytes:
        return cur
    buf = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        la_set_workspace(buf.data_ptr(), buf.numel())
    _workspaces[dev.index] = buf
    return buf
