"""Plans (purlin_plan_begin / _end / _launch / _destroy): a collective checked
and laid out once, launched many times.

Every launch of a plan must give the oracle's bits for whatever the buffers hold
at launch time, through every datapath (one-warp and 256-thread zero staging,
the TMA bulk and copy-engine Atoms, SNAC); the policy in force when the plan was
made is the one it keeps; misuse is reported, not ignored; plan launches can be
captured in a CUDA graph.
"""
import numpy as np
import pytest
import torch

import oracle
import reduce_datapath_gb300 as rd
import workloads
from helpers import close_handles, handle, host_bits, inputs, same_bits, set_variant

pytestmark = pytest.mark.gpu

POLICIES = {
    "zs": (rd.VARIANT_ZS,),
    "zs_large": (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_AUTO, rd.DIRECTION_AUTO, rd.SMALL_TILES_NEVER),
    "zs_bulk": (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_BULK),
    "zs_copy_engine": (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_COPY_ENGINE),
    "snac": (rd.VARIANT_STAGED,),
    "snac_y": (rd.VARIANT_STAGED_Y,),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rd.build()
    yield
    torch.cuda.synchronize()
    close_handles()


def _refill(bufs, dtype, seed):
    for r, t in enumerate(bufs):
        t.copy_(inputs(1, t.numel(), dtype, seed=seed * 17 + r)[0])


def _ok(h):
    torch.cuda.synchronize()
    assert rd.purlin_query_status(h) == rd.OK


@pytest.mark.parametrize("policy", list(POLICIES))
@pytest.mark.parametrize("coll", ["rs", "ag", "ar", "a2av", "a2a"])
def test_plan_launches_match_the_oracle(policy, coll):
    R, c, dtype = 8, 3001, "bf16"
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    try:
        if coll == "rs":
            x = inputs(R, R * c, dtype, seed=1)
            outs = [torch.empty(c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
            p = rd.plan(rd.purlin_reduce_scatter, h, x, outs, [c] * R, None, dtype)
            want = lambda: oracle.reduce_scatter([host_bits(t) for t in x], [c] * R, dtype=dtype)
        elif coll == "ag":
            x = inputs(R, c, dtype, seed=2)
            outs = [torch.empty(R * c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
            p = rd.plan(rd.purlin_all_gather, h, x, outs, [c] * R, None, dtype)
            want = lambda: oracle.all_gather([host_bits(t) for t in x])
        elif coll == "ar":
            x = inputs(R, c, dtype, seed=3)
            outs = [torch.empty(c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
            p = rd.plan(rd.purlin_all_reduce, h, x, outs, c, dtype)
            want = lambda: oracle.all_reduce([host_bits(t) for t in x], dtype=dtype)
        elif coll == "a2av":
            C = workloads.zipf_pair_counts(R, 300, workloads.ZIPF_S, 99) * 16
            x = [inputs(1, int(C[s].sum()), dtype, seed=40 + s)[0] for s in range(R)]
            outs = [torch.empty(int(C[:, j].sum()), dtype=torch.bfloat16, device="cuda")
                    for j in range(R)]
            p = rd.plan(rd.purlin_all_to_all_v, h, x, outs, C, None, None, dtype)
            want = lambda: oracle.all_to_all_v([host_bits(t) for t in x], C)
        else:
            x = inputs(R, R * c, dtype, seed=5)
            outs = [torch.empty(R * c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
            p = rd.plan(rd.purlin_all_to_all, h, x, outs, c, dtype)
            want = lambda: oracle.all_to_all_v([host_bits(t) for t in x], np.full((R, R), c))
        torch.cuda.synchronize()
        for rep in range(3):          # new contents each time: the plan reads them at launch
            _refill(x, dtype, seed=100 * rep + len(coll))
            p()
            _ok(h)
            w = want()
            for j in range(R):
                assert same_bits(host_bits(outs[j]), w[j]), (rep, j)
        p.destroy()
    finally:
        set_variant(h, rd.VARIANT_AUTO)


def test_plan_keeps_the_policy_it_was_made_with():
    R, n = 8, 1 << 20
    h = handle(R)
    set_variant(h, rd.VARIANT_ZS)
    x = inputs(R, n, "bf16", seed=7)
    out = [torch.empty_like(t) for t in x]
    p = rd.plan(rd.purlin_all_reduce, h, x, out, n, "bf16")
    try:
        set_variant(h, rd.VARIANT_STAGED)
        p()
        _ok(h)
        assert rd.purlin_last_launch(h)["variant"] == rd.VARIANT_ZS
        rd.purlin_all_reduce(h, x, out, n, "bf16")
        _ok(h)
        assert rd.purlin_last_launch(h)["variant"] == rd.VARIANT_STAGED
    finally:
        p.destroy()
        set_variant(h, rd.VARIANT_AUTO)


def test_plan_misuse_is_reported():
    R, n = 4, 1000
    h = handle(R)
    x = inputs(R, n, "f32", seed=8)
    out = [torch.empty_like(t) for t in x]
    with pytest.raises(rd.PurlinError):           # end without begin
        rd.purlin_plan_end(h)
    rd.purlin_plan_begin(h)
    with pytest.raises(rd.PurlinError):           # begin twice
        rd.purlin_plan_begin(h)
    with pytest.raises(rd.PurlinError):           # nothing recorded
        rd.purlin_plan_end(h)
    rd.purlin_plan_begin(h)
    rd.purlin_all_reduce(h, x, out, n, "f32")     # recorded, not launched
    with pytest.raises(rd.PurlinError) as e:      # a second call in one plan
        rd.purlin_all_reduce(h, x, out, n, "f32")
    assert e.value.status == rd.ERR_INVALID_ARG
    plan = rd.purlin_plan_end(h)
    assert plan
    rd.purlin_plan_destroy(plan)
    rd.purlin_plan_begin(h)                       # an invalid call records nothing
    with pytest.raises(rd.PurlinError):
        rd.purlin_all_reduce(h, x, [out[0]] * R, n, "f32")   # outputs overlap
    with pytest.raises(rd.PurlinError):
        rd.purlin_plan_end(h)
    with pytest.raises(rd.PurlinError):
        rd.purlin_plan_launch(None)
    rd.purlin_plan_destroy(None)
    # recording left nothing behind: the next call launches as usual
    out[0].zero_()
    rd.purlin_all_reduce(h, x, out, n, "f32")
    _ok(h)
    assert same_bits(host_bits(out[0]), oracle.all_reduce([host_bits(t) for t in x], "f32")[0])


def test_recorded_call_enqueues_nothing():
    R, n = 2, 4096
    h = handle(R)
    x = inputs(R, n, "f32", seed=9)
    out = [torch.zeros_like(t) for t in x]
    rd.purlin_plan_begin(h)
    rd.purlin_all_reduce(h, x, out, n, "f32")
    plan = rd.purlin_plan_end(h)
    torch.cuda.synchronize()
    assert all(int(torch.count_nonzero(o)) == 0 for o in out)
    rd.purlin_plan_launch(plan)
    _ok(h)
    rd.purlin_plan_destroy(plan)
    assert same_bits(host_bits(out[1]), oracle.all_reduce([host_bits(t) for t in x], "f32")[1])


@pytest.mark.parametrize("variant", [rd.VARIANT_ZS, rd.VARIANT_STAGED])
def test_plan_launches_in_a_cuda_graph(variant):
    R, c = 8, 20000
    h = handle(R)
    set_variant(h, variant)
    x = [torch.zeros(R * c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    y = [torch.empty(c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    z = [torch.empty(R * c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    stream = torch.cuda.Stream()
    rs = rd.plan(rd.purlin_reduce_scatter, h, x, y, [c] * R, None, "bf16", stream=stream)
    ag = rd.plan(rd.purlin_all_gather, h, y, z, [c] * R, None, "bf16", stream=stream)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            rs()
            ag()
        for rep in range(3):
            _refill(x, "bf16", seed=300 + rep)
            torch.cuda.synchronize()
            g.replay()
            _ok(h)
            want_y = oracle.reduce_scatter([host_bits(t) for t in x], [c] * R, dtype="bf16")
            for k in range(R):
                assert same_bits(host_bits(y[k]), want_y[k])
                assert same_bits(host_bits(z[k]), np.concatenate(want_y))
        del g
    finally:
        rs.destroy()
        ag.destroy()
        set_variant(h, rd.VARIANT_AUTO)


def test_two_launch_plan_all_reduce_in_a_cuda_graph():
    """An AllReduce into outputs on different alignments plans two kernels (a
    sum into output 0, then copies): a kept plan launches both, each launch and
    each replay of a captured graph gives the oracle's bits."""
    R, n, dtype = 8, 50000 + 5, "bf16"
    h = handle(R)
    set_variant(h, rd.VARIANT_ZS)
    x = [inputs(1, n, dtype, seed=70 + r, offset=r % 2)[0] for r in range(R)]
    full = [torch.zeros(n + 8, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    out = [t[j % 3:j % 3 + n] for j, t in enumerate(full)]
    stream = torch.cuda.Stream()
    p = rd.plan(rd.purlin_all_reduce, h, x, out, n, dtype, stream=stream)
    try:
        for rep in range(2):
            _refill(x, dtype, seed=700 + rep)
            torch.cuda.synchronize()
            p()
            _ok(h)
            assert rd.purlin_last_launch(h)["kernels"] == 2
            want = oracle.all_reduce([host_bits(t) for t in x], dtype=dtype)
            for j in range(R):
                assert same_bits(host_bits(out[j]), want[j]), (rep, j)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            p()
        for rep in range(2):
            _refill(x, dtype, seed=710 + rep)
            torch.cuda.synchronize()
            g.replay()
            _ok(h)
            want = oracle.all_reduce([host_bits(t) for t in x], dtype=dtype)
            for j in range(R):
                assert same_bits(host_bits(out[j]), want[j]), (rep, j)
        del g
    finally:
        p.destroy()
