"""bench.py's multi-process plumbing on CPU: two gloo ranks (127.0.0.1) set up the
process group, meet at the barrier, and take the maximum of a per-rank time; the
throughput is then the units of both ranks over that maximum (weak scaling)."""
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    dist, r, w, local = bench._dist_setup(world)
    assert dist is not None and (r, w, local) == (rank, world, rank)
    bench._barrier(dist)
    ms = 3.0 + 2.0 * rank  # a slower rank 1
    ms_max = bench._max_over_ranks(dist, ms)
    bench._barrier(dist)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(ms_max))
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max_over_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    vals = [float(open(tmp_path / f"rank{r}.txt").read()) for r in range(2)]
    assert vals == [5.0, 5.0]  # every rank sees the slowest rank's time


def test_single_process_has_no_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    sys.path.insert(0, ROOT)
    import bench

    dist, r, w, _ = bench._dist_setup(1)
    assert dist is None and (r, w) == (0, 1)
    assert bench._max_over_ranks(None, 2.5) == 2.5
