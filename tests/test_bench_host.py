"""Host-side logic of bench.py, on the CPU: the multi-rank reduction over a
world-size-2 gloo group, the whole-job rate, and the reference arm's rank
gating and JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's step time differs; the job takes the slowest one
        t = bench.max_over_ranks(1.5 * (rank + 1))
        dist.barrier()
        rate = bench.whole_job_rate(24, 1000, 5, world, t)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"t": t, "rate": rate}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r in res:
        assert r["t"] == 3.0
        # 2 ranks x 24 units x 1000 edges x 5 hops in 3 ms
        assert r["rate"] == pytest.approx(2 * 24 * 1000 * 5 / 3e-3)


def test_single_process_is_its_own_maximum():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.25) == 0.25
    assert bench.whole_job_rate(1, 10, 2, 1, 1.0) == pytest.approx(20_000.0)


def _run_bench(args, env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], env=env,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_other_ranks_exit_quietly():
    p = _run_bench(["--impl", "reference", "--workload", "tiny_fp32_n512", "--steps", "1"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""


def test_reference_arm_line():
    p = _run_bench(["--impl", "reference", "--workload", "tiny_fp32_n512", "--steps", "1"],
                   {"RANK": "0", "WORLD_SIZE": "1"})
    assert p.returncode == 0, p.stderr
    lines = [ln for ln in p.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "edge-hops/s" and d["value"] > 0
    assert d["warmup"] >= 3 and d["steps"] == 1 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == "tiny_fp32_n512"


def test_workload_registry():
    sys.path.insert(0, ROOT)
    from sparse_long_sequence_gb300 import workloads
    import oracle
    names = [w.name for w in workloads.ALL + workloads.VARIANTS]
    assert len(names) == len(set(names)) == len(workloads.BY_NAME)
    for w in workloads.BY_NAME.values():
        assert w.kind in ("token", "causal", "block") and w.d == 64 and w.units >= 1
        assert w.describe()["workload"] == w.name
    # the sweep keeps the text pattern; its window part is the [S] eq 6 closed form
    for w in workloads.SWEEP[:2]:
        assert (w.r, w.n_globals, w.rand_per_row, w.B, w.H) == (256, 16, 32, 2, 12)
        row_ptr, _ = oracle.token_graph(w.n, w.r, 0, 0)
        assert row_ptr[-1] == w.n * (2 * w.r + 1) - w.r * (w.r + 1)
    c = workloads.CAUSAL_TEXT
    row_ptr, _ = oracle.token_graph(c.n, c.r, 0, 0, causal=True)
    assert row_ptr[-1] == c.n * (c.r + 1) - c.r * (c.r + 1) // 2


def test_step_stats():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.step_stats([2.0])
    assert one == {"median": 2.0, "p10": 2.0, "p90": 2.0, "n": 1}
    st = bench.step_stats([float(x) for x in range(1, 12)])
    assert st["median"] == 6.0 and st["p10"] == 2.0 and st["p90"] == 10.0 and st["n"] == 11
