"""The bench's multi-rank path on CPU with the gloo backend, two ranks: the
timed region is the maximum over ranks, the whole-job value counts every
rank's work, and the reference arm runs on rank 0 only while the other rank
exits without work."""
import importlib.util
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_dist", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _aggregate_rank(rank, world, port, out_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    b = load_bench()
    ms = b.max_over_ranks(10.0 + 5.0 * rank, world, dist, "cpu")   # ranks time 10 and 15 ms
    value = b.whole_job_value(2.0e12, world, ms / 5)                  # 5 steps
    with open(os.path.join(out_dir, "r%d" % rank), "w") as f:
        f.write("%r %r" % (ms, value))
    dist.destroy_process_group()


def _reference_rank(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    b = load_bench()
    calls = []
    b.run_reference = lambda args: calls.append(args.gpus)
    sys.argv = ["bench.py", "--impl", "reference", "--gpus", str(world), "--steps", "1", "--warmup", "0"]
    b.main()
    with open(os.path.join(out_dir, "ref%d" % rank), "w") as f:
        f.write(repr(calls))


def test_time_is_max_over_ranks_and_value_counts_all_ranks(tmp_path):
    mp.start_processes(_aggregate_rank, args=(2, free_port(), str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for rank in range(2):
        ms, value = map(float, (tmp_path / ("r%d" % rank)).read_text().split())
        assert ms == 15.0
        assert value == pytest.approx(2.0e12 * 2 / (3.0e-3) / 1e12)


def test_reference_arm_runs_on_rank_zero_only(tmp_path):
    mp.start_processes(_reference_rank, args=(2, free_port(), str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    assert (tmp_path / "ref0").read_text() == "[2]"
    assert (tmp_path / "ref1").read_text() == "[]"
