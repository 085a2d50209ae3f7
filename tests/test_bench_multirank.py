"""The benchmark's multi-rank host logic on CPU: two gloo ranks, launched the
way torchrun launches them (RANK / WORLD_SIZE / MASTER_* in the environment).

Each rank times its own replica; only the timing is reduced. These tests check
the reduction (max over ranks), the barrier, the per-rank replicas (same
shapes, different seeds) and the whole-job rate, and that the reference arm
runs on rank 0 alone.
"""

from __future__ import annotations

import io
import json
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    w_, r_, _ = bench.dist_setup()
    assert (w_, r_) == (world, rank)
    assert dist.get_backend() == "gloo"
    mine = 10.0 + 7.5 * rank            # this rank's "step time"
    top = bench.max_over_ranks(mine, world, "cpu")
    bench.barrier(world)
    w = bench.rank_workload("c2", rank)
    res = {"rank": rank, "max": top, "mine": mine,
           "lens": w.context_lens.tolist(), "q_sum": float(np.asarray(w.q, dtype=np.float64).sum()),
           "shape": list(w.q.shape), "tables": list(w.block_tables.shape)}
    Path(out_dir, f"rank{rank}.json").write_text(json.dumps(res))
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0, f"rank process exit code {p.exitcode}"
    res = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in range(world)]
    # The reduction is the max of the ranks' own numbers, seen by every rank.
    assert all(r["max"] == max(x["mine"] for x in res) for r in res)
    # Replicas: identical shapes, independent draws.
    assert res[0]["shape"] == res[1]["shape"] and res[0]["tables"] == res[1]["tables"]
    assert res[0]["lens"] != res[1]["lens"] or res[0]["q_sum"] != res[1]["q_sum"]


def test_rank0_replica_is_the_single_gpu_workload():
    """Rank 0 times the single-GPU workload: for the 64-request decode, its
    bucket of 57 sequences and 7 padded rows on the spare block."""
    a = bench.rank_workload("c3", 0)
    b = bench.inputs.make("c3", padded_rows=7)
    assert np.array_equal(a.context_lens, b.context_lens) and np.array_equal(a.block_tables, b.block_tables)
    assert a.real_rows == 57 and np.all(a.block_tables[57:] == a.spare_block)
    c = bench.rank_workload("c4", 0)
    assert np.array_equal(c.block_tables, bench.inputs.make("c4").block_tables)


def test_whole_job_rate():
    # 1 GB per rank per step, two ranks, slowest step 0.5 ms: 4000 GB/s for the job.
    assert abs(bench.whole_job_gbs(10**9, 2, 0.5) - 4000.0) < 1e-9
    assert abs(bench.whole_job_gbs(10**9, 1, 0.5) - 2000.0) < 1e-9


def test_reference_arm_runs_on_rank0_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        workload, steps, warmup = "c1", 1, 0

    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(Args())
    assert buf.getvalue() == ""
