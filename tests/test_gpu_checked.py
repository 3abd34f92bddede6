"""The checked build: every kernel access tested against the call's buffers.

compute-sanitizer is not available to these tests, so the library has a debug
build of its own (libpurlin_checked.so, compiled with PURLIN_CHECKED): each
global load and store of the Atom kernels -- vector, element, TMA bulk -- is
first tested against the address ranges of the call's inputs, outputs and
staging ring; one outside them is skipped and reported as PURLIN_ERR_BOUNDS
with its address (a load of an aligned block need only hold a byte of a
buffer: the shifted bodies read the aligned blocks around a segment's ends).
Here the checked build (1) runs collectives through every path and must report
nothing while matching the oracle, and (2) catches a destination, and sources,
that the debug hook moves out of range, skipping the accesses.  The
cases run in a child process (tests/checked_cases.py) that loads the checked
library in place of the product one.
"""
import json
import os
import subprocess
import sys

import pytest

import reduce_datapath_gb300 as rd

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def checked_run():
    rd.build(checked=True)
    env = dict(os.environ, PURLIN_LIBRARY="checked")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_cases.py")],
                       env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_checked_build_is_loaded(checked_run):
    assert checked_run["checked"] is True


def test_every_path_runs_clean_under_the_checks(checked_run):
    assert checked_run["clean_cases"] >= 29
    assert checked_run["clean_failures"] == [], "\n".join(checked_run["clean_failures"])


def test_a_destination_out_of_range_is_caught_and_skipped(checked_run):
    planted = checked_run["planted"]
    assert planted["status"] == rd.ERR_BOUNDS
    assert planted["violation_in_room"]
    assert planted["room_intact"]


def test_sources_out_of_range_are_caught(checked_run):
    planted = checked_run["planted_load"]
    assert planted["status"] == rd.ERR_BOUNDS
    assert planted["violation_in_room"]
