"""The multi-GPU path is replicas only: N processes, one per GPU, each decoding
its own seeded sequence with no data-path collective; the job's time is the
slowest rank's, and rank 0 alone prints the line.  These tests run that host
logic as world-size-2 gloo ranks on the CPU (no GPU needed)."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    import synth.workloads as wl

    r, w, local = bench.dist_setup(world)
    dist.init_process_group("gloo", rank=r, world_size=w)
    ms = bench.max_over_ranks(10.0 + 7.5 * r, dist, device="cpu")   # rank 1 is slower
    dist.barrier()
    toks = wl.prompt_tokens(wl.LLAMA7B, r)          # each replica's own start token
    bslots = wl.slot_positions(wl.LLAMA8B_BATCHED)  # every replica serves its own B slots
    with open(os.path.join(out, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "local": local, "ms": ms, "toks": toks,
                   "nslots": len(bslots)}, f)
    dist.destroy_process_group()


def test_two_gloo_replicas_agree_on_the_slowest_time(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [r["rank"] for r in res] == [0, 1] and all(r["world"] == 2 for r in res)
    assert all(r["ms"] == 17.5 for r in res)          # the max over ranks, on every rank
    assert res[0]["toks"] != res[1]["toks"]            # replicas decode different sequences
    assert all(r["nslots"] == 64 for r in res)


def test_gpus_flag_must_match_the_world_size(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "0")
    with pytest.raises(SystemExit):
        bench.dist_setup(4)
    monkeypatch.setenv("WORLD_SIZE", "1")
    assert bench.dist_setup(1) == (0, 1, 0)
    assert bench.max_over_ranks(3.25) == 3.25


def test_reference_arm_under_torchrun_prints_once(tmp_path):
    """`bench.py --impl reference` launched as two ranks: rank 0 times the
    oracle and prints one JSON line; rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "1",
           "--workload", "tiny_llama_f32"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_reference_line_carries_the_contract_keys():
    """One process: the reference arm's line has the keys the driver reads."""
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
           "--warmup", "1", "--workload", "tiny_llama_f32"]
    p = subprocess.run(cmd, cwd=ROOT, env=dict(os.environ, OMP_NUM_THREADS="1"),
                       capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    line = json.loads([l for l in p.stdout.splitlines() if l.startswith("{")][-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
              "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["higher_is_better"] is True
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["cores"] >= 1 and "workload" in line["config"]
