"""Run by tests/test_gpu_env_policy.py in a child process whose environment
sets a handle's initial policy (PURLIN_CHUNK, PURLIN_DEPTH, PURLIN_CTAS,
PURLIN_VARIANT): creates a handle, runs one AllReduce and prints the launch
record and whether the result matched the oracle, as one JSON object."""
import json
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import oracle  # noqa: E402
import reduce_datapath_gb300 as rd  # noqa: E402
from helpers import host_bits, inputs, same_bits  # noqa: E402


def main():
    R, n = 4, (1 << 19) + 3
    h = rd.purlin_create(R)
    try:
        x = inputs(R, n, "bf16", seed=11)
        out = [torch.empty_like(t) for t in x]
        rd.purlin_all_reduce(h, x, out, n, "bf16")
        torch.cuda.synchronize()
        info = rd.purlin_last_launch(h)
        want = oracle.all_reduce([host_bits(t) for t in x], dtype="bf16")
        ok = all(same_bits(host_bits(out[j]), want[j]) for j in range(R))
        print(json.dumps({"info": info, "parity": ok, "status": int(rd.purlin_query_status(h))}))
    finally:
        rd.purlin_destroy(h)


if __name__ == "__main__":
    main()
