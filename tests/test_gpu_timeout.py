"""Bounded waits of the SNAC kernel: a wait that runs out is reported, not hung.

purlin_debug_inject makes the producer of channel 0 skip one notify, so a
consumer waits on a flag that nothing sets.  With a 50 ms limit the waiting CTA
records PURLIN_ERR_TIMEOUT, every other CTA leaves at its next wait, the kernel
returns, the host reads the status -- and the context stays usable: the next
call on the same handle is correct.  No fault, trap or endless loop is involved.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import reduce_datapath_gb300 as rd
from helpers import host_bits, inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", [rd.VARIANT_STAGED, rd.VARIANT_STAGED_Y])
@pytest.mark.parametrize("coll", ["all_reduce", "reduce_scatter", "all_gather"])
def test_wait_that_runs_out_reports_timeout(coll, variant):
    rd.build()
    R, c = 4, 1 << 14
    h = rd.purlin_create(R)
    try:
        rd.purlin_set_policy(h, 4096, 2, 2, variant)
        rd.purlin_set_timeout(h, 50_000_000)
        x = inputs(R, R * c, "bf16", seed=4)
        small = [t[:c] for t in x]

        def call():
            if coll == "all_reduce":
                out = [torch.empty_like(t) for t in x]
                rd.purlin_all_reduce(h, x, out, R * c, "bf16")
                return out, oracle.all_reduce([host_bits(t) for t in x], dtype="bf16")
            if coll == "reduce_scatter":
                out = [torch.empty(c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
                rd.purlin_reduce_scatter(h, x, out, [c] * R, None, "bf16")
                return out, oracle.reduce_scatter([host_bits(t) for t in x], [c] * R, dtype="bf16")
            out = [torch.empty(R * c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
            rd.purlin_all_gather(h, small, out, [c] * R, None, "bf16")
            return out, oracle.all_gather([host_bits(t) for t in small])

        rd.purlin_debug_inject(h, 1)
        t0 = time.monotonic()
        call()
        torch.cuda.synchronize()
        elapsed = time.monotonic() - t0
        assert rd.purlin_query_status(h) == rd.ERR_TIMEOUT
        assert elapsed < 10.0
        # the hook cleared itself, the status word was cleared by the query,
        # and the context still works
        out, want = call()
        torch.cuda.synchronize()
        assert rd.purlin_query_status(h) == rd.OK
        for j in range(R):
            assert np.array_equal(host_bits(out[j]), want[j])
    finally:
        rd.purlin_destroy(h)
