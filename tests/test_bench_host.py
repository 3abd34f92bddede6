"""Host-side logic of bench.py's multi-GPU mode (no GPU): replicas on gloo.

With N ranks every rank runs an independent replica; the job's value is all
ranks' bytes over the slowest rank's time.  Two CPU processes (world size 2,
gloo, 127.0.0.1) check the max-over-ranks reduction and the whole-job value,
and the reference arm does no work on ranks other than 0.  The CPU baseline's
partition-split timing must give the single-threaded oracle's bits.
"""
import io
import json
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


def _worst_case_line(bench):
    """A result line built from stub figures with every optional part present
    and long values where values can be long."""
    per = {"reduce_scatter": {"us": 97.12345678, "gbs": 6219.123456789, "bytes": 603979776},
           "all_gather": {"us": 83.98765432, "gbs": 7191.987654321, "bytes": 603979776}}
    roofline = bench.roofline_entry(per["reduce_scatter"], 6785.9, "measured", "rs",
                                    551648256, "in step")
    e2e = {"value": 363.61234567, "unit": "GB/s", "h2d_bytes_per_step": 536870912,
           "d2h_bytes_per_step": 536870912, "ms_per_step": 3.3212345678, "steps": 20,
           "link_frac": 0.9612345678, "link": {"h2d_gbs": 209.7, "d2h_gbs": 192.3,
                                               "both_gbs": 335.1},
           "note": "a long note that must not reach the line " * 4}
    cpu = {"value": 1.7871234567, "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": "a long sample description " * 10,
           "short": "20 steps, 13.5 s, " + "x" * 16}
    lat = {"us_graph_per_launch": 1.5123456789, "us_back_to_back": 2.0}
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070, "samples": 900,
              "reasons": ["sw_power_cap"]}
    return bench.compact_line(
        world=8, steps=500, warmup=10, value=56000.123456789, ms_per_step=0.17212345678,
        variant="staged_y", roofline=roofline, per=per, e2e=e2e, cpu=cpu, parity=True,
        lat=lat, launches=1000, clocks=clocks, peak=6785.9,
        step_traffic=1141000000)


def test_result_line_is_last_short_and_parses():
    """The driver reads the benchmark's result from the end of its log: the
    result line must come last, parse alone and stay under 1000 characters,
    with the contract keys and the roofline in it; the side studies go to an
    earlier line."""
    import json
    import bench
    line = _worst_case_line(bench)
    studies = {"allreduce_sweep": [{"bytes_per_rank": 4096 << (2 * i), "us": 1.5 * i}
                                   for i in range(9)] * 50}
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.emit(line, studies)
    out = buf.getvalue().splitlines()
    assert len(out) == 2 and len(out[0]) > 1000
    last = out[-1]
    assert len(last) < 1000, len(last)
    got = json.loads(last)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "cpu_baseline", "gpu_launches", "clocks",
                "parity_vs_oracle", "allreduce_4KiB_us", "step_dram_frac"):
        assert key in got, key
    assert got["config"]["workload"]
    rf = got["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s"
    assert rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], rel=1e-3)
    # DRAM bytes over the same duration: 551648256 B / 97.12 us / 6785.9 GB/s
    assert rf["dram_frac"] == pytest.approx(551648256 / 97.12345678e-6 / 1e9 / 6785.9, rel=1e-3)
    assert got["step_dram_frac"] == pytest.approx(1141000000 / 0.17212345678e-3 / 1e9 / 6785.9,
                                                  rel=1e-3)
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step", "link_frac"):
        assert key in got["e2e"]
    assert "link" not in got["e2e"] and "note" not in got["e2e"]
    for key in ("value", "unit", "cores", "kind", "sample"):
        assert key in got["cpu_baseline"]
    assert json.loads(out[0])["studies"] == studies


def test_studies_can_go_to_a_file(tmp_path):
    import json
    import bench
    line = _worst_case_line(bench)
    path = tmp_path / "studies.json"
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.emit(line, {"cta_study": [1, 2, 3]}, str(path))
    out = buf.getvalue().splitlines()
    assert len(out) == 1 and json.loads(out[0])["metric"] == bench.METRIC
    assert json.loads(path.read_text()) == {"cta_study": [1, 2, 3]}


def test_reference_line_is_short_and_shares_the_config():
    """Both arms name one workload configuration, and the reference line is
    short as well."""
    import bench
    ours = bench.bench_config(1)
    assert ours["workload"] == bench.WORKLOAD_SHORT
    assert len(json.dumps(bench.bench_config(8))) < 200


def test_sources_digest_leaves_out_the_checked_build():
    """Code that only the checked build compiles (blocks under
    `#if defined(PURLIN_CHECKED)`, PURLIN_CHECK_* lines) does not move the
    digest; the `#else` branch of such a block and every other conditional do."""
    import bench
    base = "int f(int x) { return x + 1; }\n#if defined(FOO)\nint g;\n#endif\n"
    checked = ("#if defined(PURLIN_CHECKED)\nint chk;\n#if X\nint y;\n#endif\n#endif\n"
               "int f(int x) {\n    PURLIN_CHECK_STORE(p, 4)\n    return x + 1; }\n"
               "#if defined(FOO)\nint g;\n#endif\n")
    with_else = "#if defined(PURLIN_CHECKED)\nint chk;\n#else\nint prod;\n#endif\n" + base
    other = base.replace("FOO", "BAR")
    assert bench.code_tokens(base) == bench.code_tokens(checked)
    assert bench.code_tokens(base) != bench.code_tokens(with_else)
    assert "int prod;" in bench.code_tokens(with_else)
    assert bench.code_tokens(base) != bench.code_tokens(other)
