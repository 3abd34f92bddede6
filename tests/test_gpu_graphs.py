"""Collectives captured in a CUDA graph and replayed.

A graph freezes kernel parameters at capture time.  The staged (SNAC) kernels
keep their flag epoch in device memory, so every replay runs with a fresh epoch
and must give the right answer; zero-staging kernels hold no state.  Each case
captures ReduceScatter -> AllGather and an AllReduce, then replays the graph
three times with new input contents, comparing every replay with the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import reduce_datapath_gb300 as rd
import workloads
from helpers import host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("variant", [rd.VARIANT_ZS, rd.VARIANT_STAGED, rd.VARIANT_STAGED_Y])
def test_replayed_graph_matches_oracle_every_time(variant):
    rd.build()
    R, c = 8, 40000
    n = R * c
    x = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    y = [torch.empty(c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    z = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    a = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    h = rd.purlin_create(R)
    try:
        rd.purlin_set_policy(h, 0 if variant == rd.VARIANT_ZS else 4096, 2, 3, variant)
        for t in x:
            t.zero_()
        stream = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            rd.purlin_reduce_scatter(h, x, y, [c] * R, None, "bf16")
            rd.purlin_all_gather(h, y, z, [c] * R, None, "bf16")
            rd.purlin_all_reduce(h, x, a, n, "bf16")
        for replay in range(3):
            fresh = workloads.rank_buffers("rs_ag_r8_bf16", R, n, "bf16", role=10 + replay,
                                           device="cuda")
            for dst, src in zip(x, fresh):
                dst.copy_(src)
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            assert rd.purlin_query_status(h) == rd.OK
            xs = [host_bits(t) for t in x]
            want_y = oracle.reduce_scatter(xs, [c] * R, dtype="bf16")
            want_a = oracle.all_reduce(xs, dtype="bf16")
            for k in range(R):
                assert np.array_equal(host_bits(y[k]), want_y[k]), (replay, k)
                assert np.array_equal(host_bits(z[k]), np.concatenate(want_y)), (replay, k)
                assert np.array_equal(host_bits(a[k]), want_a[k]), (replay, k)
        del g
    finally:
        torch.cuda.synchronize()
        rd.purlin_destroy(h)


@pytest.mark.parametrize("atom", [rd.ATOM_COPY_ENGINE, rd.ATOM_BULK])
def test_replayed_graph_with_other_copy_atoms(atom):
    """The copy-engine Atom (memcpy nodes, no kernel) and the TMA bulk Atom inside
    a captured graph: every replay copies the buffers' current contents."""
    rd.build()
    R, c = 8, 30001
    y = [torch.empty(c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    z = [torch.empty(R * c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    h = rd.purlin_create(R)
    try:
        rd.purlin_set_policy(h, 0, 0, 0, rd.VARIANT_ZS)
        rd.purlin_set_atom(h, atom)
        stream = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            rd.purlin_all_gather(h, y, z, [c] * R, None, "bf16")
        for replay in range(3):
            fresh = workloads.rank_buffers("rs_ag_r8_bf16", R, c, "bf16", role=20 + replay,
                                           device="cuda")
            for dst, src in zip(y, fresh):
                dst.copy_(src)
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            assert rd.purlin_query_status(h) == rd.OK
            want = np.concatenate([host_bits(t) for t in y])
            for k in range(R):
                assert np.array_equal(host_bits(z[k]), want), (replay, k)
        del g
    finally:
        torch.cuda.synchronize()
        rd.purlin_destroy(h)
