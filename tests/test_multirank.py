"""The N > 1 path of bench.py on CPU: two ranks over gloo (no GPU). The path shards into
independent replicas (every (sequence, head) chain is independent; there is no exchange step), so
the only multi-rank logic is the timing aggregation: the job's time is the slowest rank's, and the
job's throughput counts every rank's units."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        ms = bench.max_over_ranks(times[rank], w, torch.device("cpu"))
        out[rank] = (ms, bench.job_rate(1000, w, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_and_job_rate(world):
    times = [4.0 + 3.0 * r for r in range(world)]   # the last rank is the slowest
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), times, out), nprocs=world, start_method="spawn")
    slowest = max(times)
    for r in range(world):
        ms, rate = out[r]
        assert ms == slowest
        assert rate == pytest.approx(world * 1000 / (slowest * 1e-3))


def test_single_rank_is_local():
    assert bench.max_over_ranks(5.0, 1, torch.device("cpu")) == 5.0
    assert bench.job_rate(500, 1, 2.0) == pytest.approx(250000.0)


def test_alu_peak_from_unit_counts():
    """The fp32 CUDA-core peak of an ALU-bound line: SMs x 128 lanes x 2 flop x the maximum SM clock
    (the sampled one, else 2070 MHz)."""
    import types
    props = types.SimpleNamespace(multi_processor_count=152)
    fake = types.SimpleNamespace(cuda=types.SimpleNamespace(get_device_properties=lambda dev: props))
    peak, src = bench.alu_peak(None, fake, 2070.0)
    assert abs(peak - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9 and "152 SMs" in src
    assert bench.alu_peak(None, fake, None)[0] == peak


def test_profile_hash_ignores_comments_only():
    """The source hash that ties an ncu summary to the kernels' code sees code, not comments."""
    a = "// header\nint f(int x) {  /* multi\n line */ return x + 1;  // inc\n}\n"
    b = "// other words\nint f(int x) {  /* changed */ return x + 1;\n}\n"
    c = "// header\nint f(int x) {  /* multi\n line */ return x + 2;  // inc\n}\n"
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)
    assert "return x + 1;" in bench.code_only(a) and "header" not in bench.code_only(a)
