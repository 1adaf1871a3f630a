"""The checked library (liblinattn_checked.so, LA_CHECKS=1): every global-memory access of
the SIMT, reduce, read-out and decode kernels is tested against the extent of the
caller's buffer first; an access outside it is skipped and reported as LA_ERR_BOUNDS
through the device status word, never trapped.

On CPU: the checked library loads and exports every declared entry point. On a GPU, in
child processes that load it (LA_CHECKED=1): the SIMT parity cases pass with no report,
and with every extent declared 64 elements short (LA_CHECKS_SHRINK, honoured by the
checked build only) the calls report LA_ERR_BOUNDS. The real buffers are full size, so
every access the kernels do make stays inside an allocation."""
import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CHECKED = os.path.join(ROOT, "compressive_memory_attention_02_b300", "liblinattn_checked.so")


def _build_checked():
    sys.path.insert(0, ROOT)
    from compressive_memory_attention_02_b300 import build
    return build.build(checked=True)


def test_checked_library_exports_every_declared_symbol():
    from test_abi import _declared
    so = ctypes.CDLL(_build_checked())
    for name in _declared():
        assert hasattr(so, name), name
    so.la_checked_build.restype = ctypes.c_int
    assert so.la_checked_build() == 1
    import compressive_memory_attention_02_b300 as la
    assert la.la_checked_build() == (1 if os.environ.get("LA_CHECKED") == "1" else 0)
    assert "checked build" in la.error_string(la.LA_ERR_BOUNDS)


def _child(code, **env):
    e = dict(os.environ, LA_CHECKED="1", **env)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=e, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    return r.stdout


@pytest.mark.gpu
def test_simt_parity_cases_pass_in_the_checked_build():
    _build_checked()
    out = _child("import sys, pytest; sys.exit(pytest.main(['-q', '-m', 'gpu', '-p', 'no:cacheprovider', "
                 "'tests/test_parity_fwd.py', 'tests/test_parity_prefill_decode.py', '-k', "
                 "'fp32 or simt or decode_steps or prefill_output_only or prefill_bf16']))")
    assert "passed" in out and "failed" not in out


_SHRUNK = r"""
import numpy as np, torch
import compressive_memory_attention_02_b300 as la
import synthetic
assert la.la_checked_build() == 1
dev = lambda a: torch.from_numpy(a).cuda()
B, H, T, d = 1, 2, 300, 32
q, k, v = (dev(synthetic.normal(5, i, (B, H, T, d), 1.0, "f32")) for i in range(3))
out = torch.empty_like(v); M = torch.empty(B, H, d, d, device="cuda"); z = torch.empty(B, H, d, device="cuda")
la.la_causal_fwd_ex(q, k, v, out, None, None, M, z, B, H, T, d, d, 64, 1e-6, la.LA_F32, None, None, 0)
assert la.la_get_last_device_status() == la.LA_ERR_BOUNDS
o1 = torch.empty(B, H, d, device="cuda")
la.la_decode_step(q[:, :, 0].contiguous(), k[:, :, 0].contiguous(), v[:, :, 0].contiguous(), o1, M, z,
                  B, H, d, d, 1e-6, la.LA_F32)
assert la.la_get_last_device_status() == la.LA_ERR_BOUNDS
assert la.la_get_last_device_status() == la.LA_OK   # read and cleared
print("bounds reported")
"""


@pytest.mark.gpu
def test_accesses_past_a_declared_extent_are_reported_not_made():
    _build_checked()
    assert "bounds reported" in _child(_SHRUNK, LA_CHECKS_SHRINK="64")
