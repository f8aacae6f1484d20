"""The bench's multi-rank logic without a GPU: two gloo ranks on the host
(one process per GPU in a real run; replicas, so the ranks share only the
timing barrier and the max over ranks), the whole-job throughput, and the
reference arm's rank-0-only rule."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    w, r, local = bench.dist_info()
    dist = bench.init_dist(w, local)
    bench.barrier(dist)
    # each rank's "elapsed time"; the job takes the slowest
    slowest = bench.max_over_ranks(dist, 10.0 + 5.0 * r)
    bench.barrier(dist)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "backend": dist.get_backend(), "slowest": slowest}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest(tmp_path):
    port = _free_port()
    mp.spawn(_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, g in enumerate(got):
        assert g == {"world": 2, "rank": r, "backend": "gloo", "slowest": 15.0}


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    world, rank, local = bench.dist_info()
    assert (world, rank, local) == (1, 0, 0)
    assert bench.init_dist(world, local) is None
    bench.barrier(None)
    assert bench.max_over_ranks(None, 3.5) == 3.5


def test_job_value_counts_every_rank():
    # two replicas of 4096 tokens, 10 steps, slowest rank 2 s
    assert bench.job_value(2, 4096, 10, 2.0) == pytest.approx(2 * 4096 * 10 / 2.0)
    assert bench.job_value(1, 4096, 10, 2.0) * 2 == bench.job_value(2, 4096, 10, 2.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    w = bench.workload("tiny", None)

    class Args:
        steps, warmup = 1, 0

    assert bench.run_reference(Args(), w) is None
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank_zero(monkeypatch, capsys):
    # one step of the oracle arm on the small workload: one JSON line with the
    # contract's keys, its cpu_baseline and e2e carrying the line's own value
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    w = bench.workload("tiny", None)

    class Args:
        steps, warmup = 1, 0

    bench.run_reference(Args(), w)
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in line, key
    assert line["value"] > 0 and line["steps"] == 1 and line["n_gpus"] == 1
    assert line["config"]["workload"] == "tiny" and line["config"]["tokens"] == w.m
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
