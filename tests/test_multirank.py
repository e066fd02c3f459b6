"""The multi-process host path of bench.py on CPU (gloo, world size 2).

The decode and prefill workloads shard into independent replicas: every rank
times its own batch, and the job's figures are the slowest rank's time and
the units of all ranks over it (max over ranks, no data-path collective).
The reference arm (the oracle on host cores) runs and prints on rank 0
only; the other ranks exit without work."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _aggregate_worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench

    # rank r "measured" 10 (r + 1) ms for 5 steps of 32 query tokens
    total, value = bench.aggregate(10.0 * (rank + 1), 32, 5, world, device="cpu")
    q.put((rank, total, value))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_is_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_aggregate_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, value in res:
        assert total == 20.0
        assert abs(value - 2 * 32 * 5 / 0.020) < 1e-6 * value


def test_aggregate_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.aggregate(40.0, 16, 4, 1) == (40.0, 16 * 4 / 0.040)


def _bench_reference(rank: int):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1")
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                           "--warmup", "0", "--ref-sample", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=600)


def test_reference_arm_prints_on_rank0_only():
    r1 = _bench_reference(1)
    assert r1.returncode == 0, r1.stderr
    assert r1.stdout.strip() == ""
    r0 = _bench_reference(0)
    assert r0.returncode == 0, r0.stderr
    lines = [l for l in r0.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["warmup"] >= 3
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_prefill_sample():
    # the prefill's oracle baseline: sampled query rows of the 131,072-token
    # prompt, the compressor amortised to them
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "csa_prefill", "--steps", "1",
                        "--warmup", "0", "--ref-sample", "1"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr
    d = json.loads([l for l in r.stdout.splitlines() if l.strip()][-1])
    assert d["impl"] == "reference" and d["value"] > 0 and "query rows" in d["cpu_baseline"]["sample"]
    assert d["cpu_baseline"]["cores"] >= 1
