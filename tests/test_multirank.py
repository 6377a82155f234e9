"""Multi-rank host logic of the benchmark, on the CPU with gloo ranks.

The decode indexer shards over requests with no exchange step, so a run on N
GPUs is N replicas: every rank scores its own batch and the job's time is the
slowest rank's. These tests run that host logic (rank environment, per-rank
seeds, max-over-ranks reduction, whole-job rate, rank-0-only reference arm)
in two spawned gloo processes; no GPU is involved.
"""
import json
import os
import socket
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        # rank r "measured" 10 + r ms for the timed region and 3 - r ms per e2e step
        ms, e2e_ms = bench.max_over_ranks([10.0 + r, 3.0 - r], w, "cpu")
        rate = bench.whole_job_rate(1000, 5, w, ms)
        q.put({"rank": r, "world": w, "local": local, "ms": ms, "e2e_ms": e2e_ms,
               "seed": bench.rank_seed(7, r), "rate": rate})
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    out.sort(key=lambda d: d["rank"])
    assert [d["rank"] for d in out] == [0, 1]
    assert all(d["world"] == 2 and d["local"] == d["rank"] for d in out)
    # every rank sees the slowest rank's time for both timed regions
    assert all(d["ms"] == 11.0 and d["e2e_ms"] == 3.0 for d in out)
    # 2 ranks x 5 steps x 1000 units in 11 ms
    assert all(d["rate"] == pytest.approx(2 * 5 * 1000 / 0.011) for d in out)
    # replicas draw different batches
    assert out[0]["seed"] != out[1]["seed"]


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.whole_job_rate(10, 4, 1, 2.0) == pytest.approx(20000.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    args = types.SimpleNamespace(workload="tiny", seed=1, steps=1, warmup=0, impl="reference")
    bench.run_reference(args, rank=1, world=2)  # the other ranks exit without work
    assert capsys.readouterr().out == ""


def test_reference_arm_line(capsys):
    """Rank 0 of the reference arm times the oracle and prints one JSON line."""
    pytest.importorskip("numpy")
    sys.path.insert(0, ROOT)
    import bench
    args = types.SimpleNamespace(workload="tiny", seed=1, steps=1, warmup=0, impl="reference")
    bench.run_reference(args, rank=0, world=1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "keys/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_profiled_traffic_only_for_the_profiled_kernel_code(tmp_path, monkeypatch):
    """bench.py reports the ncu DRAM bytes of a workload only while the
    kernel's code (not its comments) hashes to the value recorded with the
    capture."""
    sys.path.insert(0, ROOT)
    import shutil

    import bench
    csrc = os.path.join(ROOT, "sparse_attention_indexer_block_gb300", "csrc")
    fake = tmp_path / "sparse_attention_indexer_block_gb300" / "csrc"
    shutil.copytree(csrc, fake)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "score_select_counters.json").write_text(json.dumps(
        {"decode": {"source_sha256_16": bench.kernel_code_hash(str(tmp_path)),
                    "dram_bytes_per_launch": 1234}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_counters("decode")["dram_bytes_per_launch"] == 1234
    assert bench.profiled_counters("long") is None
    with open(fake / "common.cuh", "a") as f:
        f.write("\n// a comment only\n")
    assert bench.profiled_counters("decode")["dram_bytes_per_launch"] == 1234
    with open(fake / "common.cuh", "a") as f:
        f.write("\nconstexpr int kUnusedForTest = 1;\n")
    assert bench.profiled_counters("decode") is None
