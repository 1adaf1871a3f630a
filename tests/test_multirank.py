"""The N > 1 path of the benchmark, on CPU: two gloo ranks each run their own replica
of a (small) segmented workload through the float64 oracle, with the seed, input
layout and max-over-ranks timing reduction that bench.py uses on GPUs (weak scaling,
no data-path collective)."""
import dataclasses
import multiprocessing as mp
import os
import socket
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _small():
    import synthetic
    return dataclasses.replace(synthetic.WORKLOADS["segmented"], B=1, H=2, T=256, d=16, dv=16, segment=64)


def _replica(w, rank):
    """Segment-chained oracle outputs of rank's replica (the computation one rank times)."""
    import bench
    import oracle
    q, k, v = bench.make_inputs(w, rank)
    M = z = None
    outs = []
    for s in range(q.shape[0]):
        o, M, z = oracle.causal_fwd(q[s], k[s], v[s], M_in=M, z_in=z, eps=w.eps)
        outs.append(o)
    return q, np.stack(outs), M, z


def _worker(rank, world, port, queue):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        w = _small()
        q, outs, M, z = _replica(w, rank)
        t_max = bench.max_over_ranks(0.5 + rank, dist, "cpu")   # per-rank stand-in times
        queue.put((rank, bench.replica_seed(w, rank), t_max, q[0, 0, 0, 0, :4].tolist(), float(outs.sum()),
                   float(M.sum()), float(z.sum())))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_run_independent_replicas():
    import bench
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, seed0, t0, q0, o0, M0, z0), (r1, seed1, t1, q1, o1, M1, z1) = results
    assert (r0, r1) == (0, 1)
    assert seed0 != seed1 and q0 != q1               # each rank its own problem
    assert t0 == t1 == 1.5                           # the slowest rank's time, seen by every rank
    # each rank's result is the single-process result of its replica
    w = _small()
    for rank, o, M, z in ((0, o0, M0, z0), (1, o1, M1, z1)):
        _, outs, Mr, zr = _replica(w, rank)
        assert np.isclose(o, outs.sum(), rtol=0, atol=1e-9)
        assert np.isclose(M, Mr.sum(), rtol=0, atol=1e-9) and np.isclose(z, zr.sum(), rtol=0, atol=1e-9)
    # the whole-job rate counts every rank's tokens over the slowest time
    tokens = w.B * w.T
    assert bench.aggregate_rate(tokens, t0, 2) == 2 * tokens / 1.5


def test_single_rank_reduction_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25
    assert bench.aggregate_rate(1000, 2.0, 1) == 500.0
