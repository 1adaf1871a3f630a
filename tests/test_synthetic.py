"""The seeded input generator: deterministic, counter based (any slice can be
regenerated alone), N(0, scale^2) distributed, and bf16 storage rounds to
nearest-even exactly as torch's float32 -> bfloat16 conversion does."""
import numpy as np
import torch

import synthetic


def test_deterministic_and_sliceable():
    a = synthetic.normal(5, 1, (4, 1000), 0.5, "f32")
    b = synthetic.normal(5, 1, (4, 1000), 0.5, "f32")
    np.testing.assert_array_equal(a, b)
    part = synthetic.normal(5, 1, (1000,), 0.5, "f32", first=2000)
    np.testing.assert_array_equal(part, a[2])
    c = synthetic.normal(5, 2, (4, 1000), 0.5, "f32")
    assert np.abs(a - c).max() > 0.1          # another tensor id is another stream
    d = synthetic.normal(6, 1, (4, 1000), 0.5, "f32")
    assert np.abs(a - d).max() > 0.1          # another seed is another stream


def test_distribution():
    x = synthetic.normal(9, 0, (400000,), 0.5, "f32").astype(np.float64)
    assert abs(x.mean()) < 0.005
    assert abs(x.std() - 0.5) < 0.005
    assert abs(np.mean(x > 0) - 0.5) < 0.005


def test_bf16_round_to_nearest_even_matches_torch():
    f = synthetic.normal(3, 0, (100000,), 3.0, "f32")
    bits = synthetic.normal(3, 0, (100000,), 3.0, "bf16")
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, ref)
    back = synthetic.bf16_bits_to_f32(bits)
    np.testing.assert_array_equal(back, torch.from_numpy(f).to(torch.bfloat16).float().numpy())


def test_workload_shapes():
    w = synthetic.WORKLOADS["tiny"]
    q, k, v = synthetic.qkv(w)
    assert q.shape == (1, 2, 256, 32) and q.dtype == np.float32 and v.shape == (1, 2, 256, 32)
    w = synthetic.WORKLOADS["segmented"]
    q, k, v = synthetic.qkv(w, T=64, H=2)
    assert q.shape == (2, 2, 64, 128) and q.dtype == np.uint16
    dq, dk, dv = synthetic.decode_tokens(synthetic.WORKLOADS["generation"], 3, N=4, H=2)
    assert dq.shape == (4, 2, 128) and dv.shape == (4, 2, 128)
