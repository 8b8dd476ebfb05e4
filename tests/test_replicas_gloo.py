"""The N > 1 replicas path of bench.py on CPU: two ranks over gloo. Each GPU runs an
independent engine; the only cross-rank steps are the barrier around the timed region,
the max over ranks of the elapsed time and the sum of committed tokens, which make
`value` = tokens of all ranks / the slowest rank's time."""
import multiprocessing as mp
import os
import socket
from types import SimpleNamespace

import bench


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE="2", RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    ws, r, _ = bench.dist_setup("gloo")
    bench.barrier(ws)
    ms = bench.barrier_max(ws, 40.0 + 5.0 * r, "cpu")          # rank 1 is the slower one
    tokens = bench.barrier_sum(ws, 100.0 + r, "cpu")
    q.put((r, ws, ms, tokens, tokens / (ms / 1e3)))
    dist.destroy_process_group()


def test_two_replicas_reduce_time_and_tokens_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest time (45 ms) and all committed tokens (201)
    assert got == [(0, 2, 45.0, 201.0, 201.0 / 0.045), (1, 2, 45.0, 201.0, 201.0 / 0.045)]


def test_reference_arm_runs_on_rank_0_only():
    args = SimpleNamespace(workload=bench.synth.TINY.name, steps=1, warmup=3, ref_budget=1.0)
    assert bench.run_reference(args, 2, 1, 1) is None


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup() == (1, 0, 0)
    assert bench.barrier_max(1, 3.5, "cpu") == 3.5
    assert bench.barrier_sum(1, 7.0, "cpu") == 7.0
