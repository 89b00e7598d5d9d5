"""The benchmark's host-side logic on CPU: its multi-rank timing, with two
gloo ranks, and its FLOP count.

On one GB300 per box the benchmark runs N replicas (one full SR chunk per
rank, no collective on the data path); what crosses ranks is the timing:
a barrier around the timed region and a MAX all-reduce of each rank's time,
from which the whole-job throughput is computed.  These tests run that code
in two processes over gloo on 127.0.0.1, and check the reference arm's
behaviour on ranks other than 0.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 100.0 + 25.0 * rank  # rank 1 is the slow one
        dist.barrier()
        ms = bench.max_over_ranks(my_ms, "cpu")
        value = bench.job_tflops(world, 22.61e12, 10, ms)
        results[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_is_max_and_value_counts_all_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, results), nprocs=world, start_method="spawn", join=True)
    assert set(results.keys()) == {0, 1}
    for rank in range(world):
        ms, value = results[rank]
        assert ms == 125.0  # every rank reports the slowest rank's time
        # 2 ranks x 10 chunks x 22.61 TFLOP in 0.125 s
        assert value == pytest.approx(2 * 10 * 22.61 / 0.125)


def test_single_process_timing_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(42.0) == 42.0
    assert bench.job_tflops(1, 22.61e12, 1, 14.3) == pytest.approx(22.61 / 0.0143)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    """Under torchrun only rank 0 runs and prints the reference arm."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(workloads, "generate", lambda *a, **k: called.append(1))
    assert bench.run_reference(None, workloads.get("720p")) == 0
    assert not called


def test_bench_flop_count_matches_oracle_definition():
    """The benchmark's TFLOP/s divides by visible FLOPs (4*d per visible
    (query, key) pair); its count must equal the oracle's, from the mask
    definition, on every workload."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads
    from oracle import reference as ref
    for w in workloads.WORKLOADS.values():
        want = ref.visible_flops(w.heads, w.head_dim, w.frame_tokens, w.n_frames, w.ref_frames, w.window_radius)
        assert bench.visible_flops(w) == want, w.name
