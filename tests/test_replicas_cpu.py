"""The multi-process path of bench.py on CPU: replicas only (no data-path
collective), so what N > 1 adds is the job's timing -- the slowest rank's
time, world x one rank's work -- computed with a gloo process group of two
ranks here exactly as the NCCL group does it on GPUs."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as td
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    td.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) ms per step and 10 - r ms end to end
        ms, e2e = bench.max_over_ranks([1.0 + rank, 10.0 - rank])
        out.put((rank, ms, e2e, bench.whole_job_tflops(6.0e11, ms, world)))
    finally:
        td.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, e2e, tf in res:
        assert ms == 2.0 and e2e == 10.0          # both ranks see the slowest rank's times
        assert tf == pytest.approx(6.0e11 * 2 / 2.0e-3 / 1e12)


def test_single_process_is_identity():
    assert bench.max_over_ranks([3.5, 1.25]) == [3.5, 1.25]
    assert bench.whole_job_tflops(1e12, 1.0, 1) == pytest.approx(1000.0)


def test_cpu_baseline_sampler_and_config_on_cpu():
    # The oracle leg of bench.py on the tiny workload: a positive rate over
    # whole (b, h, q-block) samples, in a seeded order that resumes where it
    # stopped; the config names the workload and its geometry.
    from block_sparse_attention_plan_gb300 import workloads as W
    w = W.make_workload("tiny")
    rate, dt, done, nxt = bench.oracle_sample_rate(w, 0.2)
    assert rate > 0 and dt > 0 and done > 0 and done % 8 == 0 and nxt == done
    _, _, done2, nxt2 = bench.oracle_sample_rate(w, 0.05, start=nxt)
    assert nxt2 == nxt + done2
    cfg = bench._config(w, gpu=False)
    assert cfg["workload"] == "tiny" and cfg["active_blocks"] == w.active_blocks
    assert cfg["active_flop_per_step"] == w.active_flop


class _Ev:
    """Stand-in for a CUDA event: a timestamp in ms."""

    def __init__(self, t):
        self.t = t

    def elapsed_time(self, other):
        return other.t - self.t


def test_step_times_from_events():
    # Events of one step: start, preparation done, bounded start, bounded
    # end, step end, plan kernels done, key-norm start, key-norm end.
    step = [_Ev(t) for t in (0.0, 0.053, 0.058, 0.497, 0.508, 0.050, 0.001, 0.039)]
    ms, fwd_ms, prep_ms, bounded_ms, plan_ms, knorm_ms = bench._times([step, step])
    assert ms == pytest.approx(0.508)
    assert fwd_ms == pytest.approx(0.508 - 0.053)
    assert prep_ms == pytest.approx(0.053)
    assert bounded_ms == pytest.approx(0.497 - 0.058)
    assert plan_ms == pytest.approx(0.050)
    assert knorm_ms == pytest.approx(0.038)


def test_traffic_figure_is_keyed_to_the_kernel_sources():
    value, key = bench.NCU_TRAFFIC["video_dit"]
    assert bench._traffic("video_dit") == (value if key == bench._kernel_hash() else None)
    assert bench._traffic("no_such_workload") is None
