"""The bench's multi-rank host logic on two CPU ranks (gloo): every rank gets the slowest
rank's time, the job value counts the units of all ranks over that time, and the
reference arm prints nothing on ranks other than 0.  No GPU: the data path of a rank is
an independent replica, so only this aggregation crosses ranks."""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = [40.0, 55.0][rank]
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        value = bench.job_throughput(world, 1000, 10, ms)
        q.put((rank, ms, value, bench.rank_info()))
    finally:
        dist.barrier()
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, value, info in got:
        assert ms == 55.0                                  # the slowest rank's time everywhere
        assert value == pytest.approx(2 * 1000 * 10 / 0.055)
        assert info == (rank, 2, 0)


def test_reference_arm_other_ranks_exit_quietly(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(None, bench.WORKLOADS["layer-T32"]) == 0
    assert capsys.readouterr().out == ""


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert bench.job_throughput(1, 100, 4, 2.0) == pytest.approx(200000.0)


def test_reference_arm_json_line():
    """The reference arm (the CPU oracle on a bounded sample of the workload) prints one
    JSON line with the contract's keys, on CPU."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--workload", "layer-T32",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["warmup"] >= 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "layer-T32"


def test_kernel_hash_ignores_comments(tmp_path, monkeypatch):
    """The stored gate/up DRAM-traffic capture is keyed by a hash of the kernel source that
    comments and blank lines do not change, while code does."""
    import shutil
    import bench
    root = tmp_path / "repo"
    csrc = root / "bit_expert_layer_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in ("expert_gemm.cu", "common.cuh", "gemm_common.cuh"):
        shutil.copy(os.path.join(bench.ROOT, "bit_expert_layer_gb300", "csrc", f), csrc / f)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_hash()
    p = csrc / "common.cuh"
    p.write_text(p.read_text() + "\n// a new comment\n/* and a block\n   comment */\n\n")
    assert bench.kernel_hash() == h0
    p.write_text(p.read_text() + "constexpr int UNUSED_FOR_TEST = 1;\n")
    assert bench.kernel_hash() != h0


def test_gpus_flag_starts_the_ranks():
    """``bench.py --gpus 2`` without a launcher starts two ranks itself and one JSON line
    comes out, from rank 0, with n_gpus 2 (the reference arm: no GPU needed)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR",
                                                             "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--impl", "reference",
                        "--workload", "layer-T32", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
