"""A handle's initial policy from the environment (for sweeps): PURLIN_CHUNK,
PURLIN_DEPTH, PURLIN_CTAS and PURLIN_VARIANT are read by purlin_create and act
as purlin_set_policy would; out-of-range values are ignored.  Each case runs
tests/env_policy_case.py in a child process with its own environment."""
import json
import os
import subprocess
import sys

import pytest

import reduce_datapath_gb300 as rd

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = ("PURLIN_CHUNK", "PURLIN_DEPTH", "PURLIN_CTAS", "PURLIN_VARIANT")


def _run(**env):
    rd.build()
    e = {k: v for k, v in os.environ.items() if k not in KEYS}
    e.update({k: str(v) for k, v in env.items()})
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "env_policy_case.py")],
                       env=e, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_environment_sets_the_staged_policy():
    res = _run(PURLIN_CHUNK=8192, PURLIN_DEPTH=3, PURLIN_CTAS=5,
               PURLIN_VARIANT=rd.VARIANT_STAGED)
    info = res["info"]
    assert res["parity"] and res["status"] == rd.OK
    assert info["variant"] == rd.VARIANT_STAGED
    assert info["chunk_bytes"] == 8192 and info["depth"] == 3
    assert info["grid"] == 5 * 3   # five channels of three roles


def test_values_out_of_range_are_ignored():
    res = _run(PURLIN_CHUNK=1000, PURLIN_DEPTH=99, PURLIN_CTAS=-4,
               PURLIN_VARIANT=rd.VARIANT_STAGED_Y)
    info = res["info"]
    assert res["parity"] and res["status"] == rd.OK
    assert info["variant"] == rd.VARIANT_STAGED_Y
    assert info["depth"] == 2           # the default depth
    assert info["chunk_bytes"] != 1000  # not a multiple of 16: left at the default
