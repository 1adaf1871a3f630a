"""The bench's roofline accounting against the per-unit counts, restated here: forward bytes
(2d + 2dv)*2 per token and head (q, k, v read, out written) plus the state written once per
segment by the segment-wise call (4(d*dv + d) per head and segment; the final state only for a
one-segment workload or for chained segment calls, whose hand-overs between calls are not
algorithmic and count against the kernel); forward FLOPs 4*d*dv + (C+1)(d+dv) + 3d + dv +
(C+1)/2 per token and head."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synthetic  # noqa: E402


def test_segmented_workload_bytes_and_flops():
    w = synthetic.WORKLOADS["segmented"]
    byt, flops = bench.algorithmic(w)
    tokens_heads = 2 * 32 * 32768
    assert byt == tokens_heads * 512 * 2 + 16 * 2 * 32 * (128 * 128 + 128) * 4 == 2_215_116_800
    assert flops == tokens_heads * (4 * 128 * 128 + 65 * 256 + 3 * 128 + 128 + 32.5)
    assert abs(flops - 1.7348e11) / 1.7348e11 < 1e-4
    # as 16 chained calls (the final state only): one call carries a sixteenth of the bytes
    byt_calls, _ = bench.algorithmic(w, state_per_segment=False)
    assert byt_calls == tokens_heads * 512 * 2 + 2 * 32 * (128 * 128 + 128) * 4 == 2_151_710_720
    assert byt_calls // 16 == 134_481_920


def test_training_workload_bytes():
    w = synthetic.WORKLOADS["train"]
    byt, _ = bench.algorithmic(w)
    assert byt == 4 * 16 * 4096 * 256 * 2 + 4 * 16 * (64 * 64 + 64) * 4 == 135_282_688


def test_roofline_bound_is_hbm_for_every_forward_workload():
    """Arithmetic intensity far below the ridge of the measured peaks (bf16 FLOP/s / HBM B/s)."""
    hbm, tf, _ = bench.peaks()
    ridge = tf * 1e12 / (hbm * 1e9)
    for name in ("train", "segmented"):
        byt, flops = bench.algorithmic(synthetic.WORKLOADS[name])
        assert flops / byt < ridge / 3
