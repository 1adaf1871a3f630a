"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
entry point include/linattn.h declares, sizes workspaces, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "linattn.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_modes():
    names = _declared()
    for n in ("la_causal_fwd", "la_prefill_state", "la_decode_step"):
        assert n in names


def test_library_exports_every_declared_symbol():
    import compressive_memory_attention_02_b300 as la
    so = ctypes.CDLL(la.LIB_PATH)
    for name in _declared():
        assert hasattr(so, name), name
    assert set(_declared()) <= set(la.EXPORTS) | {"la_stream_t"}


def test_error_strings():
    import compressive_memory_attention_02_b300 as la
    assert la.error_string(la.LA_OK) == "ok"
    assert "unsupported" in la.error_string(la.LA_ERR_UNSUPPORTED)
    assert la.error_string(99) == "unknown error"


def test_workspace_sizes():
    import compressive_memory_attention_02_b300 as la
    rec = 128 * 128 + 128
    # prefill: one record per part and head, plus a final state per head
    assert la.la_prefill_workspace_size(1, 8, 1 << 20, 128, 128, 4096, la.LA_BF16) == 4 * rec * 8 * (256 + 1)
    # a single part needs only the final-state area
    assert la.la_prefill_workspace_size(1, 8, 4096, 128, 128, 4096, la.LA_BF16) == 4 * rec * 8
    assert la.la_causal_fwd_workspace_size(1, 1, 64, 7, 64, 64, la.LA_BF16) == 0
    # float32 forward runs on the SIMT path, which needs no scratch
    assert la.la_causal_fwd_workspace_size(2, 32, 2048, 128, 128, 64, la.LA_F32) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(B=0), 1), (dict(T=0), 1), (dict(eps=-1.0), 1),
    (dict(d=7), 2), (dict(dv=136), 2), (dict(chunk=48), 2), (dict(dtype=5), 2),
])
def test_forward_rejects_bad_arguments_on_host(kw, code):
    import compressive_memory_attention_02_b300 as la
    a = dict(q=16, k=32, v=48, out=64, B=1, H=1, T=64, d=64, dv=64, chunk=64, eps=1e-6, dtype=la.LA_BF16)
    a.update(kw)
    rc = la.lib.la_causal_fwd(a["q"], a["k"], a["v"], a["out"], None, None, None, None, a["B"], a["H"], a["T"],
                              a["d"], a["dv"], a["chunk"], a["eps"], a["dtype"], None)
    assert rc == code


def test_decode_and_prefill_reject_bad_arguments_on_host():
    import compressive_memory_attention_02_b300 as la
    assert la.lib.la_decode_step(16, 32, 48, 64, None, 96, 1, 1, 64, 64, 1e-6, 1, None) == la.LA_ERR_INVALID_ARG
    assert la.lib.la_decode_step(16, 32, 48, 64, 84, 96, 1, 1, 64, 64, 1e-6, 1, None) == la.LA_ERR_INVALID_ARG  # M misaligned
    assert la.lib.la_decode_step(16, 32, 48, 64, 128, 96, 1, 1, 60, 64, 1e-6, 1, None) == la.LA_ERR_UNSUPPORTED
    assert la.lib.la_prefill_state(16, 32, 48, 64, None, None, None, None, 1, 1, 64, 64, 64, -1, 1e-6, 1,
                                   None) == la.LA_ERR_INVALID_ARG
    assert la.lib.la_set_workspace(8, 1024) == la.LA_ERR_WORKSPACE


def test_backward_workspace_size_and_host_checks():
    """Size of the backward's scratch: two float32 state records per 64-token chunk and
    head, plus T*(dv+1) floats per head, each region rounded up to 256 bytes; argument
    errors are found on the host before anything is launched."""
    import compressive_memory_attention_02_b300 as la
    up = lambda n: (n + 63) // 64 * 64
    for B, H, T, d, dv in [(1, 1, 1, 8, 8), (2, 3, 130, 64, 32), (4, 16, 4096, 64, 64), (2, 32, 2048, 128, 128)]:
        BH, nch, rec = B * H, (T + 63) // 64, d * dv + d
        want = 4 * (2 * up(BH * nch * rec) + up(BH * T * dv) + up(BH * T))
        assert la.la_causal_bwd_workspace_size(B, H, T, d, dv) == want
    assert la.la_causal_bwd_workspace_size(1, 1, 64, 12, 64) == 0   # d not a multiple of 8
    assert la.la_causal_bwd_workspace_size(1, 1, 0, 64, 64) == 0
    args = [16, 32, 48, 64, None, None, None, None, 80, 96, 112, None, None]
    assert la.lib.la_causal_bwd(*args, 1, 1, 64, 64, 64, 1e-6, 1, None) in (la.LA_ERR_WORKSPACE, la.LA_ERR_CUDA)
    assert la.lib.la_causal_bwd(*args, 1, 1, 64, 60, 64, 1e-6, 1, None) == la.LA_ERR_UNSUPPORTED
    assert la.lib.la_causal_bwd(*args, 1, 1, 0, 64, 64, 1e-6, 1, None) == la.LA_ERR_INVALID_ARG
    bad = list(args)
    bad[8] = 16  # dq aliases q
    assert la.lib.la_causal_bwd(*bad, 1, 1, 64, 64, 64, 1e-6, 1, None) == la.LA_ERR_INVALID_ARG
    assert la.lib.la_causal_bwd(*args, 1, 1, 64, 64, 64, 1e-6, 3, None) == la.LA_ERR_UNSUPPORTED


def test_backward_rejects_unaligned_inputs_on_host():
    import compressive_memory_attention_02_b300 as la
    args = [16, 32, 48, 72, None, None, None, None, 80, 96, 112, None, None]  # dout 8 bytes off
    assert la.lib.la_causal_bwd(*args, 1, 1, 64, 64, 64, 1e-6, 1, None) == la.LA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,code", [
    (dict(M_seg=None), 1), (dict(z_seg=None), 1), (dict(seg_len=100), 1), (dict(seg_len=0), 1), (dict(T=0), 1),
    (dict(z_seg=0x10000 + 4096), 1),     # z_seg inside M_seg (2 segments x 64 x 64 floats = 32 KB)
    (dict(M_in=0x10000 + 8192), 1),      # the initial state inside M_seg
    (dict(d=7), 2), (dict(dtype=5), 2),
])
def test_segments_call_rejects_bad_arguments_on_host(kw, code):
    """la_causal_fwd_segments checks its arguments before touching the device."""
    import compressive_memory_attention_02_b300 as la
    a = dict(q=16, k=32, v=48, out=64, M_in=None, M_seg=0x10000, z_seg=0x40000, B=1, H=1, T=128, d=64, dv=64,
             seg_len=64, dtype=la.LA_BF16)
    a.update(kw)
    rc = la.lib.la_causal_fwd_segments(a["q"], a["k"], a["v"], a["out"], a["M_in"], None, a["M_seg"], a["z_seg"],
                                       a["B"], a["H"], a["T"], a["d"], a["dv"], a["seg_len"], 1e-6, a["dtype"],
                                       None, 0, None)
    assert rc == code
