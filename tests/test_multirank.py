"""The multi-rank path of bench.py, on the host with gloo (world size 2,
rendezvous on 127.0.0.1): a weakly scaled run's throughput is the work of
all ranks over the slowest rank's time, each rank draws its own batch, and
under torchrun the reference arm runs on rank 0 alone and prints one line.
CPU only; no GPU and no NCCL."""

import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    class Args:
        impl = "reference"          # gloo: the backend of the host-only arm

    w, r, _ = bench.dist_setup(Args)
    # rank r processed 1000 (r + 1) KV bytes and 10 (r + 1) tokens per step,
    # 3 steps, in 0.5 + r seconds
    value, tok_per_s, t = bench.aggregate(1000 * (r + 1), 10 * (r + 1), 3, 0.5 + r, w)
    bench.barrier(w)
    queue.put((r, value, tok_per_s, t))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(queue.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, value, tok_per_s, t in got:
        assert t == pytest.approx(1.5)                        # the slower rank's time
        assert value == pytest.approx(3 * 3000 / 1.5 / 1e9)  # every rank's bytes
        assert tok_per_s == pytest.approx(3 * 30 / 1.5)


def test_single_rank_aggregate_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    value, tok_per_s, t = bench.aggregate(2e9, 100, 4, 2.0, 1)
    assert (value, tok_per_s, t) == (4.0, 200.0, 2.0)


def test_ranks_draw_independent_batches(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    import synthetic
    seeds = []
    monkeypatch.setattr(synthetic, "config2_gqa_batch", lambda seed: seeds.append(seed))
    monkeypatch.setattr(synthetic, "config3_mha_lognormal", lambda seed: seeds.append(seed))
    for rank in range(4):
        bench.workload("gqa4_u128_2048", seed_offset=rank)
        bench.workload("mha32_lognormal800", seed_offset=rank)
    assert len(set(seeds)) == len(seeds) == 8


def test_reference_arm_under_torchrun_two_ranks():
    """`torchrun --nproc-per-node 2 bench.py --impl reference`: rank 0 times
    the oracle and prints one JSON line; rank 1 exits 0 without work."""
    env = dict(os.environ)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--ref-sample-seqs", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_traffic_record_keys_on_code_not_comments():
    """The recorded ncu traffic is tied to the attention kernel's code: a
    comment or layout edit keeps the key, a code edit changes it."""
    sys.path.insert(0, ROOT)
    import bench
    src = "int f(int a) {  // one\n  return a + 1; /* two */ }\nconst char* s = \"x // y\";\n"
    assert bench.strip_c_comments(src) == bench.strip_c_comments(
        "int f(int a) { /* other */\n\n return a + 1;   }\n// note\nconst char* s = \"x // y\";")
    assert bench.strip_c_comments(src) != bench.strip_c_comments(src.replace("a + 1", "a + 2"))
    assert "x // y" in bench.strip_c_comments(src)
