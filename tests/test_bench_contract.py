"""The bench's JSON line: every key the run contract names, built by the same function the
bench prints from, on a made-up timing record (no GPU): the whole-job rate, the per-launch
roofline arithmetic, the end-to-end object and the launch count."""
import os
import sys
from types import SimpleNamespace

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synthetic  # noqa: E402


def _line(world=1, with_e2e=True, status=0):
    w = synthetic.WORKLOADS["segmented"]
    K = 10
    res = {"ms_total": 5.0, "launches": K, "launches_per_step": 1, "status": status,
           "clocks": {"sm_mhz": 2032, "sm_max_mhz": 2032, "reasons": [], "samples": 5}}
    if with_e2e:
        res["e2e"] = {"steps": 2, "seconds": 0.1, "h2d": 1610612736, "d2h": 604504064}
    return w, K, bench.report_ours(SimpleNamespace(steps=K, warmup=3), w, res, world)


def test_required_keys_and_types():
    w, K, line = _line()
    for key, typ in (("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                     ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                     ("dtype", str), ("data", str), ("config", dict), ("roofline", dict), ("gpu_launches", int),
                     ("clocks", dict), ("e2e", dict)):
        assert isinstance(line[key], typ), key
    assert line["vs_baseline"] is None
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    assert line["steps"] == K and line["warmup"] == 3 and line["gpu_launches"] == K
    assert "workload" in line["config"]
    r = line["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r, key
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["traffic"] is None or (isinstance(r["traffic"], int) and r["traffic"] > 0)
    e = line["e2e"]
    assert set(e) == {"value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"}
    assert e["unit"] == line["unit"]


def test_rates_and_roofline_arithmetic():
    w, K, line = _line()
    # 5 ms for 10 steps: 0.5 ms a step, B*T tokens a step
    assert abs(line["ms_per_step"] - 0.5) < 1e-12
    assert abs(line["value"] - w.B * w.T / 0.5e-3) < 0.1
    byt, _ = bench.algorithmic(w)
    achieved = byt / 0.5e-3 / 1e9  # one launch a step
    r = line["roofline"]
    assert abs(r["achieved"] - achieved) < 0.1
    assert abs(r["frac"] - achieved / r["peak"]) < 1e-4
    # end to end: 2 steps in 0.1 s
    assert abs(line["e2e"]["value"] - w.B * w.T * 2 / 0.1) < 0.1


def test_whole_job_rate_counts_every_rank():
    _, _, one = _line(world=1)
    _, _, four = _line(world=4)
    assert abs(four["value"] - 4 * one["value"]) < 1.0
    assert four["n_gpus"] == 4 and four["config"]["global_batch"] == 4 * one["config"]["global_batch"]


def test_device_status_reported_only_when_set():
    _, _, ok = _line(status=0)
    _, _, bad = _line(status=2)
    assert "device_status" not in ok and bad["device_status"] == 2
    _, _, no_e2e = _line(with_e2e=False)
    assert "e2e" not in no_e2e
