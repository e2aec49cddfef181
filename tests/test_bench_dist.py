"""The multi-rank path of bench.py on the CPU: two `gloo` ranks (world size 2, 127.0.0.1).

On GPUs the bench runs one replica of the workload per rank (there is no exchange step on the
attention path), takes each timing's maximum over the ranks and reports all ranks' FLOPs over
that time. Here the same functions run under a gloo process group with made-up timings, so
the reduction and the throughput formula are checked without a GPU.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    # rank r took (10 + r) ms for its timed steps and (7 - r) ms for its end-to-end step
    total_ms, e2e_ms = bench.max_over_ranks([10.0 + r, 7.0 - r], w)
    value = bench.job_tflops(w, 2.0e12, 5, total_ms)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
        f.write("%d %d %d %r %r %r\n" % (r, w, local, total_ms, e2e_ms, value))


def test_two_gloo_ranks_take_the_max_and_count_all_ranks(tmp_path):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    lines = [open(tmp_path / ("rank%d.txt" % r)).read().split() for r in range(world)]
    for r, fields in enumerate(lines):
        rank, w, local = (int(x) for x in fields[:3])
        total_ms, e2e_ms, value = (float(x) for x in fields[3:])
        assert (rank, w, local) == (r, world, r)
        assert total_ms == 11.0 and e2e_ms == 7.0      # the slowest rank's times
        # 2 ranks x 2e12 FLOP x 5 steps in 11 ms
        assert value == pytest.approx(2 * 2.0e12 * 5 / 0.011 / 1e12)


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.5], 1) == [3.0, 4.5]
    assert bench.job_tflops(1, 1.0e12, 2, 4.0) == pytest.approx(500.0)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    """Under torchrun only rank 0 times the oracle and prints; the other ranks return 0 at once
    and print nothing."""
    sys.path.insert(0, ROOT)
    import bench
    from io_aware_attention_fa2_gb300.inputs import WORKLOADS
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup, gpus, ref_total_seconds = 2, 3, 2, 1.0

    assert bench.run_reference(Args(), WORKLOADS["tiny_n256_d64"]) == 0
    assert capsys.readouterr().out == ""
