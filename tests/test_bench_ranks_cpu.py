"""bench.py's multi-rank host logic on CPU: world size 2 over gloo (127.0.0.1),
the timing reduced to the slowest rank on every rank and the whole-job
throughput of the replicas.  No GPU: the ranks exchange plain CPU tensors."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(ws), "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench.dist_setup()
        ms = bench.max_over_ranks(dist, 100.0 + 7.0 * rank, "cpu")  # rank 1 is the slow one
        with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
            f.write(f"{got_ws} {got_rank} {got_local} {ms!r}")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    ws, port = 2, _free_port()
    mp.spawn(_rank_main, args=(ws, port, str(tmp_path)), nprocs=ws, join=True)
    for r in range(ws):
        got_ws, got_rank, got_local, ms = open(tmp_path / f"r{r}").read().split()
        assert (int(got_ws), int(got_rank), int(got_local)) == (ws, r, r)
        assert float(ms) == 107.0


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(None, 3.5, "cpu") == 3.5


def test_replica_throughput_counts_every_rank_over_the_slowest_time():
    # 2 replicas x 10 steps x 1e9 bytes in 4 s of the slowest rank
    assert bench.replica_throughput(10 ** 9, 10, 2, 4000.0) == pytest.approx(5.0)
    assert bench.replica_throughput(10 ** 9, 10, 1, 4000.0) == pytest.approx(2.5)
