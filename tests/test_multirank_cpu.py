"""Host logic of the N > 1 benchmark path, run as two gloo ranks on the CPU:
each rank runs its own replica (weak scaling), the slowest rank's time
decides, and the whole-job value counts every rank's work."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 100.0 + 50.0 * rank  # rank 1 is the slow one
        total = bench.max_over_ranks(local_ms, dist)
        out[rank] = (total, bench.whole_job_tflops(world, 1e12, 10, total))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_takes_the_slowest_rank():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0] == out[1]
    total, value = out[0]
    assert total == pytest.approx(150.0)
    # 2 ranks x 10 steps x 1 TFLOP in 0.15 s
    assert value == pytest.approx(2 * 10 / 0.15)


def test_single_rank_is_identity():
    assert bench.max_over_ranks(12.5, None) == 12.5
    assert bench.whole_job_tflops(1, 2e12, 5, 1000.0) == pytest.approx(10.0)


def test_traffic_record_follows_the_forward_kernel_sources():
    """The per-launch DRAM traffic in the bench line is reported only while the
    forward kernel's sources are those of the capture: every listed source
    exists, and the record is found for the headline workload and variant
    only."""
    d = os.path.join(bench.ROOT, "tensorized_online_softmax_gb300", "csrc")
    for name in bench.FWD_SOURCES:
        assert os.path.isfile(os.path.join(d, name)), name
    assert len(bench.csrc_sha256()) == 64
    rec = bench.MEASURED_TRAFFIC
    if rec["csrc_sha256"] == bench.csrc_sha256():
        assert bench.measured_traffic(rec["workload"], rec["variant"]) == rec["bytes"]
    assert bench.measured_traffic(rec["workload"], "vec") is None
    assert bench.measured_traffic("no_such_workload", rec["variant"]) is None
