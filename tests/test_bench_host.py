"""Host-side logic of bench.py on CPU: the max-over-ranks reduction with two
gloo ranks, and the reference arm (the FP64 oracle) under one and two ranks."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    out = bench.reduce_max([rank + 1.0, 10.0 - rank, -rank], dist)
    q.put((rank, out))
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_max_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.0, 10.0, 0.0]


def _json_lines(text):
    return [json.loads(ln) for ln in text.splitlines() if ln.startswith("{")]


def test_reference_arm_single_process():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "b1_l3297", "--steps", "3",
                        "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    ln = lines[0]
    assert ln["impl"] == "reference" and ln["value"] > 0 and ln["unit"] == "GB/s"
    assert ln["cpu_baseline"]["kind"] == "oracle" and ln["cpu_baseline"]["cores"] >= 1
    assert ln["e2e"]["h2d_bytes_per_step"] == 0 and ln["steps"] == 3 and ln["warmup"] == 3


def test_reference_arm_prefill_single_process():
    """The prefill workload's reference arm: the FP64 oracle on a bounded
    sample of output rows, reported in the prefill metric's unit."""
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "prefill_q8192_kv262144",
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    ln = lines[0]
    assert ln["impl"] == "reference" and ln["value"] > 0 and ln["unit"] == "TFLOP/s"
    assert ln["cpu_baseline"]["kind"] == "oracle" and ln["cpu_baseline"]["cores"] >= 1
    assert ln["e2e"] == {"value": ln["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_two_ranks_rank0_only():
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--workload", "b1_l3297", "--steps", "3", "--warmup", "3", "--gpus", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    assert len(_json_lines(r.stdout)) == 1


def test_warmup_floor():
    r = subprocess.run([sys.executable, "bench.py", "--warmup", "2"], cwd=ROOT, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode != 0


def test_code_hash_ignores_comments_only():
    """The recorded ncu traffic stays valid across comment edits, not code edits."""
    sys.path.insert(0, ROOT)
    import bench

    a = "int f(int x) {  // doubles x\n  return 2 * x; /* plain */\n}\n"
    b = "// a new header line\nint f(int x) {\n  /* changed\n comment */ return 2 * x;\n}\n"
    c = "int f(int x) {\n  return 3 * x;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert len(bench.kernel_source_hash()) == 16
