"""Host-side logic of bench.py's multi-GPU mode (no GPU): replicas on gloo.

With N ranks every rank runs an independent replica; the job's value is all
ranks' bytes over the slowest rank's time.  Two CPU processes (world size 2,
gloo, 127.0.0.1) check the max-over-ranks reduction and the whole-job value,
and the reference arm does no work on ranks other than 0.  The CPU baseline's
partition-split timing must give the single-threaded oracle's bits.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 * (rank + 1)           # rank 1 is the slowest
    value, max_ms = bench.whole_job_value(world, 100, 1_000_000, local_ms)
    bench.barrier(world)
    q.put((rank, value, max_ms))
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, value, max_ms in got:
        assert max_ms == 20.0
        # 2 ranks x 100 steps x 1 MB in 20 ms = 10 GB/s
        assert value == pytest.approx(10.0)


def test_reference_arm_is_silent_off_rank_zero(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.bench_reference(_args(bench))
    assert buf.getvalue() == ""


def _args(bench):
    argv = sys.argv
    try:
        sys.argv = ["bench.py", "--impl", "reference", "--gpus", "2"]
        return bench.parse_args()
    finally:
        sys.argv = argv


@pytest.mark.parametrize("cores", [1, 8, 16, 20])
def test_threaded_oracle_baseline_is_bit_identical(monkeypatch, cores):
    """The partition-split CPU baseline must produce exactly the single-threaded
    oracle's step (same per-element rank order), whatever the core count."""
    import numpy as np
    import bench
    monkeypatch.setattr(bench, "PART", 777)
    monkeypatch.setattr(bench.os, "cpu_count", lambda: cores)
    rng = np.random.default_rng(5)
    xh = [rng.integers(0, 1 << 16, size=bench.R * 777, dtype=np.uint16) & 0xBFFF
          for _ in range(bench.R)]
    _, y1, z1 = bench.run_cpu_oracle(xh, 0.0, max_reps=1)
    c2, y2, z2 = bench.run_cpu_oracle_threads(xh, 0.0, max_reps=1)
    assert c2["cores"] == min(cores, bench.R) and c2["kind"].startswith("oracle")
    assert all(np.array_equal(a, b) for a, b in zip(y1, y2))
    assert all(np.array_equal(a, b) for a, b in zip(z1, z2))


def test_sources_digest_ignores_comments_not_code():
    """The digest that ties an ncu summary's traffic to the kernel sources
    changes with the code but not with comments or layout."""
    import bench
    base = 'int f(int x) { return x + 1; } // one\n/* two */ const char* s = "a // b";\n'
    same = '/* header */\nint f(int x)\n{\n    return x + 1;   // the increment\n}\nconst char* s = "a // b";'
    other = 'int f(int x) { return x + 2; } const char* s = "a // b";'
    strs = 'int f(int x) { return x + 1; } const char* s = "a // c";'
    assert bench.code_tokens(base) == bench.code_tokens(same)
    assert bench.code_tokens(base) != bench.code_tokens(other)
    assert bench.code_tokens(base) != bench.code_tokens(strs)
    files = {f: base for f in bench.KERNEL_SOURCES["zs"]}
    d1 = bench.sources_digest("zs", read=files.get)
    d2 = bench.sources_digest("zs", read={f: same for f in files}.get)
    d3 = bench.sources_digest("zs", read={f: other for f in files}.get)
    assert d1 == d2 != d3
