"""Host-side logic of bench.py: replica timing aggregation over ranks
(world size 2, gloo, CPU) and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r's replica took (r + 1) ms per step and 10 + r ms end to end
    got = bench.max_over_ranks([1.0 + rank, 10.0 + rank], torch.device("cpu"), world)
    rate = bench.whole_job_rate(1e9, got[0], world)
    out.put((rank, got, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in res:
        assert got == [2.0, 11.0]           # slowest rank's times on every rank
        assert rate == pytest.approx(2 * 1e9 / 2e-3)  # both ranks' work / slowest time


def test_reference_arm_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3", "--ref-seconds", "2"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 3
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_source_hash_ignores_comments_only():
    """The hash that ties committed profiler counters to the kernels drops
    comments and layout but keeps code and string literals (inline PTX)."""
    sys.path.insert(0, ROOT)
    import bench
    a = 'int x = 1; // note\nasm("mov.u32 %0, 1; // not a comment");\n'
    b = 'int x = 1;   /* other\nnote */\nasm("mov.u32 %0, 1; // not a comment");'
    c = 'int x = 2; // note\nasm("mov.u32 %0, 1; // not a comment");\n'
    d = 'int x = 1; // note\nasm("mov.u32 %0, 2; // not a comment");\n'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert bench._code_only(a) != bench._code_only(d)
    assert bench._code_only("char q = '\"'; // x") == "char q = '\"';"
