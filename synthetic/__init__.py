"""Seeded synthetic inputs shared by the oracle and the CUDA path.

Holds none of the attention method's arithmetic: it only draws counter-based
normal values (see gen.c for the generator's definition) and stores them in
the workload's storage dtype. bf16 arrays are returned as numpy uint16 bit
patterns; fp32 arrays as float32.

The five workloads are the shapes the method is exercised on:
  tiny          fp32 B=1 H=2 T=256 d=dv=32 chunk=64, N(0,1)
  train         bf16 B=4 H=16 T=4096 d=dv=64 chunk=64, 0.5 N(0,1)
  segmented     bf16 B=2 H=32 T=32768 d=dv=128, 16 segments of 2048, chunk=64
  prefill       bf16 B=1 H=8 T=1048576 d=dv=128, partial-sum unit 4096
  generation    bf16 256 sequences x H=32, d=dv=128: 2048 prompt tokens,
                then 1024 one-token decode steps
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None

# tensor ids inside one workload's seed
TID_Q, TID_K, TID_V = 0, 1, 2
TID_DEC_Q, TID_DEC_K, TID_DEC_V = 3, 4, 5


def build(force: bool = False) -> str:
    """Compile gen.c into _build/libsynth.so (gcc, OpenMP)."""
    src = os.path.join(_HERE, "gen.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        os.makedirs(os.path.dirname(_SO), exist_ok=True)
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.synth_normal.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                     ctypes.c_double, ctypes.c_int, ctypes.c_void_p]
        lib.synth_normal.restype = None
        lib.synth_normal_affine.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                            ctypes.c_double, ctypes.c_double, ctypes.c_int, ctypes.c_void_p]
        lib.synth_normal_affine.restype = None
        lib.synth_bf16_to_f32.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
        lib.synth_bf16_to_f32.restype = None
        _lib = lib
    return _lib


def normal(seed: int, tensor_id: int, shape, scale: float = 1.0, dtype: str = "bf16",
           first: int = 0, out: np.ndarray | None = None, shift: float = 0.0) -> np.ndarray:
    """shift + scale * N(0,1) for flat indices [first, first + prod(shape)) of tensor
    (seed, tensor_id).

    dtype "bf16" -> uint16 bit patterns, "f32" -> float32. `out` may be a
    preallocated C-contiguous array (e.g. a pinned host buffer viewed as numpy).
    """
    n = int(np.prod(shape)) if len(shape) else 1
    npdt = np.uint16 if dtype == "bf16" else np.float32
    if out is None:
        out = np.empty(shape, dtype=npdt)
    assert out.dtype == npdt and out.flags.c_contiguous and out.size == n
    dt = 1 if dtype == "bf16" else 0
    if shift == 0.0:
        _load().synth_normal(seed, tensor_id, first, n, scale, dt, out.ctypes.data)
    else:
        _load().synth_normal_affine(seed, tensor_id, first, n, scale, float(shift), dt, out.ctypes.data)
    return out


def to_bf16_bits(x) -> np.ndarray:
    """Round values to float32 and then to bf16 (round to nearest even), as uint16 bit
    patterns: a storage conversion (finite values only)."""
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def negate(arr: np.ndarray) -> np.ndarray:
    """-x of a storage array, exactly (bf16: the sign bit flipped)."""
    if arr.dtype == np.uint16:
        return arr ^ np.uint16(0x8000)
    return -arr


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 values."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float32)
    _load().synth_bf16_to_f32(bits.ctypes.data, out.ctypes.data, bits.size)
    return out


def to_f64(arr: np.ndarray) -> np.ndarray:
    """Storage array (uint16 bf16 bits or float32) -> float64 values."""
    if arr.dtype == np.uint16:
        return bf16_bits_to_f32(arr).astype(np.float64)
    return arr.astype(np.float64)


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str            # "f32" or "bf16"
    B: int
    H: int
    T: int
    d: int
    dv: int
    chunk: int
    scale: float
    seed: int
    segment: int = 0      # forward: segment length carried through M,z; prefill: partial-sum unit
    eps: float = 1e-6
    decode_steps: int = 0  # generation: one-token steps after a T-token prompt
    note: str = field(default="", compare=False)


WORKLOADS = {
    "tiny": Workload("tiny", "f32", 1, 2, 256, 32, 32, 64, 1.0, 1001,
                     note="fp32 oracle case, all outputs plus final M,z"),
    "train": Workload("train", "bf16", 4, 16, 4096, 64, 64, 64, 0.5, 1002,
                      note="training-style forward, all outputs"),
    "segmented": Workload("segmented", "bf16", 2, 32, 32768, 128, 128, 64, 0.5, 1003, segment=2048,
                          note="Infini-style: fp32 M,z carried across 16 segments of 2048"),
    "prefill": Workload("prefill", "bf16", 1, 8, 1048576, 128, 128, 64, 0.5, 1004, segment=4096,
                        note="streaming prefill: final M,z and last-token output"),
    "generation": Workload("generation", "bf16", 256, 32, 2048, 128, 128, 64, 0.5, 1005,
                           decode_steps=1024,
                           note="2048-token prefill then 1024 recurrent decode steps"),
}


def qkv(w: Workload, T: int | None = None, B: int | None = None, H: int | None = None):
    """Q, K, V storage arrays [B, H, T, d|dv] for workload w (optionally a smaller
    B/H/T cut of the same recipe: the same seed, a smaller flat index space)."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    T = w.T if T is None else T
    q = normal(w.seed, TID_Q, (B, H, T, w.d), w.scale, w.dtype)
    k = normal(w.seed, TID_K, (B, H, T, w.d), w.scale, w.dtype)
    v = normal(w.seed, TID_V, (B, H, T, w.dv), w.scale, w.dtype)
    return q, k, v


def decode_tokens(w: Workload, step: int, N: int | None = None, H: int | None = None):
    """One decode step's q, k, v storage arrays [N, H, d|dv] (step-major flat index)."""
    N = w.B if N is None else N
    H = w.H if H is None else H
    nq = N * H * w.d
    nv = N * H * w.dv
    q = normal(w.seed, TID_DEC_Q, (N, H, w.d), w.scale, w.dtype, first=step * nq)
    k = normal(w.seed, TID_DEC_K, (N, H, w.d), w.scale, w.dtype, first=step * nq)
    v = normal(w.seed, TID_DEC_V, (N, H, w.dv), w.scale, w.dtype, first=step * nv)
    return q, k, v
