"""The multi-rank host logic of bench.py (replicas only: no collective on
the data path) on CPU: two gloo ranks, each with its own timing, agree on the
slowest rank's time, the job throughput counts every rank's bytes over that
time, and the reference arm runs on rank 0 only."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, local = bench.dist_env()
    ms = bench.slowest_rank_ms(10.0 + 5.0 * rank, w, "cpu")  # rank 1 is the slow one
    gbs = bench.job_gbs(1e9, w, ms / 1e3)
    dist.destroy_process_group()
    with open(os.path.join(result_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "ms": ms, "gbs": gbs}, f)


def test_two_ranks_report_the_slowest_rank_and_the_whole_job(tmp_path):
    port = _free_port()
    mp.start_processes(_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert (d["rank"], d["world"], d["local"]) == (r, 2, r)
        assert d["ms"] == pytest.approx(15.0)        # the max over ranks, on every rank
        assert d["gbs"] == pytest.approx(2 * 1e9 / 15e-3 / 1e9)  # both ranks' bytes over the slowest time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.slowest_rank_ms(3.5, 1, "cpu") == 3.5
    assert bench.job_gbs(2e9, 1, 0.5) == pytest.approx(4.0)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:  # the arm must return at once on a rank other than 0
        layers = 1
        steps = 1
        warmup = 0

    bench.run_reference(Args(), 1, 2)
    assert capsys.readouterr().out == ""


def _fake_smi(tmp_path, util: str, pids: list[int]) -> str:
    """A stand-in nvidia-smi answering the two idle-check queries."""
    script = tmp_path / "nvidia-smi"
    pid_lines = "\n".join(str(p) for p in pids)
    script.write_text("#!/bin/sh\n"
                      "case \"$*\" in\n"
                      f"  *utilization.gpu*) echo '{util}' ;;\n"
                      f"  *compute-apps*) printf '%s\\n' '{pid_lines}' ;;\n"
                      "esac\n")
    script.chmod(0o755)
    return str(tmp_path)


def test_gpu_idle_check_reads_utilization_and_other_processes(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("PATH", _fake_smi(tmp_path, "37", [os.getpid(), 4242, 4343]) + os.pathsep +
                       os.environ.get("PATH", ""))
    got = bench.gpu_idle_check("0")
    assert got == {"util_pct": 37.0, "other_processes": 2}  # this process is not counted


def test_gpu_idle_check_without_nvidia_smi(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("PATH", str(tmp_path))  # nothing named nvidia-smi here
    assert bench.gpu_idle_check("0") == {"util_pct": None, "other_processes": None}
