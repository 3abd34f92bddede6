"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle.

Every collective, dtype, datapath variant (zero staging and SNAC staged, at
several chunk sizes / depths / CTA counts) and layout (packed, explicit
displacements, zero counts, unaligned starts, in-place forms) must match the
oracle BIT FOR BIT: copies are permutations of bytes, and sums follow one fixed
rank order with binary32 accumulation and a single rounding.  Every output is
surrounded by canary guards that must survive.
"""
import numpy as np
import pytest
import torch

import oracle
import reduce_datapath_gb300 as rd
import workloads
from helpers import (TORCH, Guarded, close_handles, handle, host_bits, inputs, same_bits,
                     set_variant)

pytestmark = pytest.mark.gpu

POLICIES = {
    "zs": (rd.VARIANT_ZS, 0, 0, 0),
    "zs_3ctas": (rd.VARIANT_ZS, 0, 0, 3),
    # 256-thread CTAs at every size (small messages otherwise run one-warp CTAs)
    "zs_large": (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_AUTO, rd.DIRECTION_AUTO, rd.SMALL_TILES_NEVER),
    "zs_large_3ctas": (rd.VARIANT_ZS, 0, 0, 3, rd.ATOM_AUTO, rd.DIRECTION_AUTO,
                       rd.SMALL_TILES_NEVER),
    # one-warp CTAs at every size
    "zs_small": (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_AUTO, rd.DIRECTION_AUTO, 1 << 30),
    "zs_bulk": (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_BULK),
    "zs_bulk_3ctas": (rd.VARIANT_ZS, 0, 0, 3, rd.ATOM_BULK),
    "zs_copy_engine": (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_COPY_ENGINE),
    "zs_pull": (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_VECTOR, rd.DIRECTION_PULL),
    "zs_pull_bulk_3ctas": (rd.VARIANT_ZS, 0, 0, 3, rd.ATOM_BULK, rd.DIRECTION_PULL),
    "snac_tiny_chunks": (rd.VARIANT_STAGED, 256, 2, 3),
    "snac_default": (rd.VARIANT_STAGED, 0, 0, 0),
    "snac_deep": (rd.VARIANT_STAGED, 4096, 8, 5),
    # sums reduced by the producer, the reduced chunk staged
    "snac_y_default": (rd.VARIANT_STAGED_Y, 0, 0, 0),
    "snac_y_tiny_chunks": (rd.VARIANT_STAGED_Y, 256, 3, 3),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rd.build()
    yield
    torch.cuda.synchronize()
    close_handles()


def run_ok(h):
    torch.cuda.synchronize()
    st = rd.purlin_query_status(h)
    assert st == rd.OK, rd.purlin_status_string(st)


def oracle_in(bufs):
    return [host_bits(b) for b in bufs]


# ------------------------------------------------------------------ AllReduce

@pytest.mark.parametrize("policy", list(POLICIES))
@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("R", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("n", [0, 1, 7, 33, 4096, 70001])
def test_all_reduce(policy, dtype, R, n):
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    x = inputs(R, n, dtype, seed=n + 7 * R)
    outs = [Guarded(n, dtype) for _ in range(R)]
    rd.purlin_all_reduce(h, x, [o.view for o in outs], n, dtype)
    run_ok(h)
    want = oracle.all_reduce(oracle_in(x), dtype=dtype)
    for j in range(R):
        assert same_bits(host_bits(outs[j].view), want[j]), (j,)
        assert outs[j].guards_intact()


@pytest.mark.parametrize("policy", ["zs", "zs_large", "snac_tiny_chunks", "snac_y_tiny_chunks"])
@pytest.mark.parametrize("offset", [1, 3, 8])
def test_all_reduce_unaligned_streams(policy, offset):
    """Streams starting at different offsets force element-wise segments."""
    R, n, dtype = 4, 5000, "bf16"
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    x = [inputs(1, n, dtype, seed=100 + r, offset=(offset * r) % 16)[0] for r in range(R)]
    outs = [Guarded(n, dtype, offset=offset) for _ in range(R)]
    rd.purlin_all_reduce(h, x, [o.view for o in outs], n, dtype)
    run_ok(h)
    want = oracle.all_reduce(oracle_in(x), dtype=dtype)
    for j in range(R):
        assert same_bits(host_bits(outs[j].view), want[j])
        assert outs[j].guards_intact()


@pytest.mark.parametrize("policy", ["zs", "zs_large", "snac_tiny_chunks", "snac_y_tiny_chunks"])
def test_all_reduce_in_place(policy):
    R, n, dtype = 8, 12345, "f32"
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    x = inputs(R, n, dtype, seed=5)
    want = oracle.all_reduce(oracle_in(x), dtype=dtype)
    rd.purlin_all_reduce(h, x, x, n, dtype)
    run_ok(h)
    for j in range(R):
        assert same_bits(host_bits(x[j]), want[j])


# ------------------------------------------------------------- ReduceScatter

def _rs_case(R, seed, explicit):
    counts = workloads.random_counts(R, 3000, seed)
    if explicit:   # partitions in a shuffled order with gaps
        rng = np.random.default_rng(seed)
        displs = np.zeros(R, dtype=np.int64)
        pos = 0
        for k in rng.permutation(R):
            displs[k] = pos
            pos += counts[k] + int(rng.integers(0, 9))
        return counts, displs, int(pos)
    return counts, None, int(counts.sum())


@pytest.mark.parametrize("policy", list(POLICIES))
@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("R", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("explicit", [False, True])
def test_reduce_scatter_v(policy, dtype, R, explicit):
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    seed = 11 * R + explicit
    counts, displs, total = _rs_case(R, seed, explicit)
    x = inputs(R, total, dtype, seed=seed)
    outs = [Guarded(int(c), dtype) for c in counts]
    rd.purlin_reduce_scatter(h, x, [o.view for o in outs], counts, displs, dtype)
    run_ok(h)
    want = oracle.reduce_scatter(oracle_in(x), counts, displs, dtype=dtype)
    for k in range(R):
        assert same_bits(host_bits(outs[k].view), want[k]), k
        assert outs[k].guards_intact()


@pytest.mark.parametrize("policy", ["zs", "zs_large", "snac_tiny_chunks", "snac_y_tiny_chunks"])
def test_reduce_scatter_in_place(policy):
    R, c, dtype = 8, 1001, "bf16"
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    x = inputs(R, R * c, dtype, seed=77)
    want = oracle.reduce_scatter(oracle_in(x), [c] * R, dtype=dtype)
    outs = [x[k][k * c:(k + 1) * c] for k in range(R)]
    rd.purlin_reduce_scatter(h, x, outs, [c] * R, None, dtype)
    run_ok(h)
    for k in range(R):
        assert same_bits(host_bits(outs[k]), want[k])


@pytest.mark.parametrize("policy", ["zs", "zs_large", "snac_tiny_chunks", "snac_y_tiny_chunks"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_reduce_scatter_unaligned_partitions(policy, dtype):
    """Partitions at odd element offsets: heads and tails are element-wise."""
    R = 5
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    counts = np.array([1023, 1, 0, 517, 2049])
    displs = np.array([3, 1031, 1040, 1100, 1701])
    x = inputs(R, 3800, dtype, seed=3, offset=1)
    outs = [Guarded(int(c), dtype, offset=3) for c in counts]
    rd.purlin_reduce_scatter(h, x, [o.view for o in outs], counts, displs, dtype)
    run_ok(h)
    want = oracle.reduce_scatter(oracle_in(x), counts, displs, dtype=dtype)
    for k in range(R):
        assert same_bits(host_bits(outs[k].view), want[k])
        assert outs[k].guards_intact()


@pytest.mark.parametrize("coll", ["all_reduce", "reduce_scatter"])
@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("R", [2, 3, 4, 5])
@pytest.mark.parametrize("offset", [0, 1, 4, 8])
def test_sums_of_few_ranks_over_many_tiles(coll, dtype, R, offset):
    """Sums of 2 to 4 ranks take 2 or 4 units per thread: messages of several
    such tiles (256 threads x 4 x 32 B = 32 KiB) with a ragged tail; streams
    `offset` elements into their allocations leave 32-byte, 16-byte or
    element-wise bodies."""
    esize = 4 if dtype == "f32" else 2
    n = (5 * 32768 + 4 * 777) // esize + 3
    h = handle(R)
    set_variant(h, *POLICIES["zs_large"])
    x = [inputs(1, n, dtype, seed=900 + 10 * R + r, offset=offset)[0] for r in range(R)]
    if coll == "all_reduce":
        outs = [Guarded(n, dtype, offset=offset) for _ in range(R)]
        rd.purlin_all_reduce(h, x, [o.view for o in outs], n, dtype)
        want = oracle.all_reduce(oracle_in(x), dtype=dtype)
    else:
        counts = np.full(R, n // R)
        counts[-1] += n - int(counts.sum())
        outs = [Guarded(int(c), dtype, offset=offset) for c in counts]
        rd.purlin_reduce_scatter(h, x, [o.view for o in outs], counts, None, dtype)
        want = oracle.reduce_scatter(oracle_in(x), counts, None, dtype=dtype)
    run_ok(h)
    for j in range(R):
        assert same_bits(host_bits(outs[j].view), want[j]), j
        assert outs[j].guards_intact()


# ------------------------------------------------------------------ AllGather

@pytest.mark.parametrize("policy", list(POLICIES))
@pytest.mark.parametrize("dtype", ["bf16", "f32", "u8"])
@pytest.mark.parametrize("R", [1, 3, 8])
@pytest.mark.parametrize("explicit", [False, True])
def test_all_gather_v(policy, dtype, R, explicit):
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    seed = 13 * R + explicit
    counts, displs, total = _rs_case(R, seed, explicit)
    x = [inputs(1, int(c), dtype, seed=seed + k)[0] for k, c in enumerate(counts)]
    outs = [Guarded(total, dtype) for _ in range(R)]
    for o in outs:   # gaps between blocks keep their initial value in both sides
        o.view.zero_()
    rd.purlin_all_gather(h, x, [o.view for o in outs], counts, displs, dtype)
    run_ok(h)
    want = oracle.all_gather(oracle_in(x), counts, displs, out_count=total)
    for j in range(R):
        assert same_bits(host_bits(outs[j].view), want[j]), j
        assert outs[j].guards_intact()


@pytest.mark.parametrize("policy", ["zs", "zs_large", "zs_bulk", "zs_copy_engine", "zs_pull", "snac_tiny_chunks"])
def test_all_gather_in_place(policy):
    R, c, dtype = 8, 999, "bf16"
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    outs = inputs(R, R * c, dtype, seed=9)
    ins = [outs[k][k * c:(k + 1) * c] for k in range(R)]
    want = oracle.all_gather([host_bits(i) for i in ins])
    rd.purlin_all_gather(h, ins, outs, [c] * R, None, dtype)
    run_ok(h)
    for j in range(R):
        assert same_bits(host_bits(outs[j]), want[j])


@pytest.mark.parametrize("policy", ["zs", "zs_large", "zs_bulk", "zs_copy_engine", "zs_pull", "snac_tiny_chunks"])
def test_all_gather_bytes_at_odd_offsets(policy):
    """u8 payloads at odd byte offsets use narrow copy units."""
    R = 3
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    counts = np.array([4097, 31, 1000])
    x = [inputs(1, int(c), "u8", seed=k, offset=k + 1)[0] for k, c in enumerate(counts)]
    outs = [Guarded(int(counts.sum()), "u8", offset=5) for _ in range(R)]
    rd.purlin_all_gather(h, x, [o.view for o in outs], counts, None, "u8")
    run_ok(h)
    want = oracle.all_gather(oracle_in(x), counts)
    for j in range(R):
        assert same_bits(host_bits(outs[j].view), want[j])
        assert outs[j].guards_intact()


# ------------------------------------------------------------------ AllToAll(V)

@pytest.mark.parametrize("policy", list(POLICIES))
@pytest.mark.parametrize("dtype", ["bf16", "u8", "f32"])
@pytest.mark.parametrize("R", [1, 2, 8])
@pytest.mark.parametrize("explicit", [False, True])
def test_all_to_all_v(policy, dtype, R, explicit):
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    seed = 17 * R + explicit
    C = workloads.random_pair_counts(R, 700, seed)
    sd = rdsp = None
    if explicit:   # reversed packing on both sides
        sd = np.zeros((R, R), dtype=np.int64)
        rdsp = np.zeros((R, R), dtype=np.int64)
        for s in range(R):
            pos = 0
            for j in reversed(range(R)):
                sd[s, j] = pos
                pos += C[s, j]
        for j in range(R):
            pos = 0
            for s in reversed(range(R)):
                rdsp[j, s] = pos
                pos += C[s, j]
    x = [inputs(1, int(C[s].sum()), dtype, seed=seed + s)[0] for s in range(R)]
    outs = [Guarded(int(C[:, j].sum()), dtype) for j in range(R)]
    rd.purlin_all_to_all_v(h, x, [o.view for o in outs], C, sd, rdsp, dtype)
    run_ok(h)
    want = oracle.all_to_all_v(oracle_in(x), C, sd, rdsp)
    for j in range(R):
        assert same_bits(host_bits(outs[j].view), want[j]), j
        assert outs[j].guards_intact()


@pytest.mark.parametrize("policy", ["zs", "zs_large", "zs_bulk", "zs_copy_engine", "snac_tiny_chunks"])
def test_all_to_all_fixed_twice_is_identity(policy):
    R, c, dtype = 8, 3001, "bf16"
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    x = inputs(R, R * c, dtype, seed=21)
    mid = [torch.empty_like(t) for t in x]
    back = [torch.empty_like(t) for t in x]
    rd.purlin_all_to_all(h, x, mid, c, dtype)
    rd.purlin_all_to_all(h, mid, back, c, dtype)
    run_ok(h)
    want = oracle.all_to_all_v(oracle_in(x), np.full((R, R), c))
    for j in range(R):
        assert same_bits(host_bits(mid[j]), want[j])
        assert same_bits(host_bits(back[j]), host_bits(x[j]))


# ------------------------------------------------------------- tree order

def _as_f64(bits, dtype):
    if dtype == "f32":
        return bits.astype(np.float64)
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("policy", ["zs", "zs_large", "snac_tiny_chunks", "snac_y_tiny_chunks"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("R", [3, 8])
def test_tree_order(policy, dtype, R):
    """The pairwise order is bit-exact to the oracle's pairwise fold.  Against
    the fixed rank order it may differ by the reordering error of binary32 adds,
    2(R-1) 2^-24 sum|x|, plus one unit in the last place of the output type:
    1e-6 relative to sum|x| for fp32, 1 ulp plus that for bf16."""
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    c = 4000
    x = inputs(R, R * c, dtype, seed=31 + R)
    outs = [torch.empty(c, dtype=x[0].dtype, device="cuda") for _ in range(R)]
    rd.purlin_set_reduce_order(h, rd.ORDER_TREE)
    try:
        rd.purlin_reduce_scatter(h, x, outs, [c] * R, None, dtype)
        run_ok(h)
    finally:
        rd.purlin_set_reduce_order(h, rd.ORDER_FIXED)
    xin = oracle_in(x)
    tree = oracle.reduce_scatter(xin, [c] * R, dtype=dtype, order="tree")
    fixed = oracle.reduce_scatter(xin, [c] * R, dtype=dtype)
    mag = np.sum([np.abs(_as_f64(a, dtype)) for a in xin], axis=0)
    for k in range(R):
        got = host_bits(outs[k])
        assert same_bits(got, tree[k])
        g, f = _as_f64(got, dtype), _as_f64(fixed[k], dtype)
        scale = mag[k * c:(k + 1) * c]
        reorder = 2 * (R - 1) * 2.0 ** -24 * scale
        if dtype == "f32":
            assert np.all(np.abs(g - f) <= 1e-6 * scale + 1e-38)
        else:
            ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(f), 2.0 ** -126))) - 7)
            assert np.all(np.abs(g - f) <= ulp + reorder)


@pytest.mark.parametrize("policy", ["zs", "zs_large", "zs_small", "snac_default", "snac_tiny_chunks",
                                    "snac_y_default", "snac_y_tiny_chunks"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("R", [3, 5, 8])
@pytest.mark.parametrize("layout", ["partitions_off_grid", "ranks_on_different_grids"])
def test_tree_order_shifted_bodies(policy, dtype, R, layout):
    """The pairwise order on layouts off the vector grid (shifted bodies):
    partitions whose starts sit off the outputs' 16-byte grid, or ranks' inputs
    r % 4 elements into their allocations.  Bit-exact to the oracle's pairwise
    fold, for a ReduceScatter and an AllReduce."""
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    c = 5 * 1024 + 3
    n = R * c
    off = (lambda r: r % 4) if layout == "ranks_on_different_grids" else (lambda r: 0)
    x = [inputs(1, n, dtype, seed=1200 + 7 * R + r, offset=off(r))[0] for r in range(R)]
    xin = oracle_in(x)
    rs_out = [Guarded(c, dtype) for _ in range(R)]
    ar_out = [Guarded(n, dtype, offset=1) for _ in range(R)]
    rd.purlin_set_reduce_order(h, rd.ORDER_TREE)
    try:
        rd.purlin_reduce_scatter(h, x, [o.view for o in rs_out], [c] * R, None, dtype)
        rd.purlin_all_reduce(h, x, [o.view for o in ar_out], n, dtype)
        run_ok(h)
    finally:
        rd.purlin_set_reduce_order(h, rd.ORDER_FIXED)
    want = oracle.reduce_scatter(xin, [c] * R, dtype=dtype, order="tree")
    whole = np.concatenate(want)
    for k in range(R):
        assert same_bits(host_bits(rs_out[k].view), want[k]), k
        assert rs_out[k].guards_intact()
    for j in range(R):
        assert same_bits(host_bits(ar_out[j].view), whole), j
        assert ar_out[j].guards_intact()


@pytest.mark.parametrize("coll", ["all_gather", "all_to_all_v"])
def test_bulk_atom_hands_off_grid_layouts_to_shifted_bodies(coll):
    """Under the TMA bulk Atom a layout whose sources and destinations sit on
    different 16-byte alignments runs on the vector kernels (shifted bodies,
    256-thread CTAs); an aligned layout stays on the one-warp bulk CTAs."""
    R = 4
    h = handle(R)
    # 256-thread CTAs at every size, so that the vector kernels are told apart
    # from the one-warp bulk CTAs
    set_variant(h, rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_BULK, rd.DIRECTION_AUTO, rd.SMALL_TILES_NEVER)
    try:
        for counts, want_block in (([20000 + 13 * k + 3 for k in range(R)], 256),
                                   ([16384] * R, 32)):
            if coll == "all_gather":
                x = [inputs(1, c, "bf16", seed=70 + k)[0] for k, c in enumerate(counts)]
                outs = [Guarded(sum(counts), "bf16") for _ in range(R)]
                rd.purlin_all_gather(h, x, [o.view for o in outs], counts, None, "bf16")
                want = oracle.all_gather(oracle_in(x))
            else:
                C = np.array([[counts[(s + j) % R] // R for j in range(R)] for s in range(R)])
                x = [inputs(1, int(C[s].sum()), "bf16", seed=80 + s)[0] for s in range(R)]
                outs = [Guarded(int(C[:, j].sum()), "bf16") for j in range(R)]
                rd.purlin_all_to_all_v(h, x, [o.view for o in outs], C, None, None, "bf16")
                want = oracle.all_to_all_v(oracle_in(x), C)
            run_ok(h)
            assert rd.purlin_last_launch(h)["block"] == want_block
            for j in range(R):
                assert same_bits(host_bits(outs[j].view), want[j]), j
                assert outs[j].guards_intact()
    finally:
        set_variant(h, *POLICIES["zs"])


# ------------------------------------------------------------ argument errors

def test_argument_errors_enqueue_nothing():
    R, n = 2, 64
    h = handle(R)
    set_variant(h, rd.VARIANT_ZS)
    x = inputs(R, n, "f32", seed=1)
    out = [torch.zeros(n, device="cuda") for _ in range(R)]
    with pytest.raises(rd.PurlinError) as e:   # outputs overlap
        rd.purlin_all_reduce(h, x, [out[0], out[0]], n, "f32")
    assert e.value.status == rd.ERR_INVALID_ARG
    with pytest.raises(rd.PurlinError) as e:   # an output inside another rank's input
        rd.purlin_all_reduce(h, x, [x[1], out[1]], n, "f32")
    assert e.value.status == rd.ERR_INVALID_ARG
    with pytest.raises(rd.PurlinError) as e:   # copy op is not a reduction
        rd.purlin_all_reduce(h, x, out, n, "f32", op="copy")
    assert e.value.status == rd.ERR_UNSUPPORTED
    with pytest.raises(rd.PurlinError) as e:   # misaligned float stream
        rd.purlin_all_reduce(h, [x[0].data_ptr() + 1, x[1]], out, n - 1, "f32")
    assert e.value.status == rd.ERR_INVALID_ARG
    with pytest.raises(rd.PurlinError) as e:   # null buffer with a non-zero count
        rd.purlin_all_reduce(h, [None, x[1]], out, n, "f32")
    assert e.value.status == rd.ERR_INVALID_ARG
    with pytest.raises(rd.PurlinError) as e:   # overlapping AllGather blocks
        rd.purlin_all_gather(h, x, out, [8, 8], [0, 4], "f32")
    assert e.value.status == rd.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[1]) == 0
    with pytest.raises(rd.PurlinError) as e:
        rd.purlin_create(9)
    assert e.value.status == rd.ERR_INVALID_ARG


def test_last_launch_reports_the_call():
    R, n = 8, 1 << 20
    h = handle(R)
    set_variant(h, rd.VARIANT_ZS)
    x = inputs(R, n, "bf16", seed=2)
    out = [torch.empty_like(t) for t in x]
    rd.purlin_all_reduce(h, x, out, n, "bf16")
    info = rd.purlin_last_launch(h)
    assert info["variant"] == rd.VARIANT_ZS and info["kernels"] == 1
    assert info["bytes_moved"] == 2 * R * n * 2
    assert 1 <= info["grid"] and info["block"] == 256 and info["sms"] > 100
    set_variant(h, rd.VARIANT_STAGED)
    rd.purlin_all_reduce(h, x, out, n, "bf16")
    info = rd.purlin_last_launch(h)
    assert info["variant"] == rd.VARIANT_STAGED and info["grid"] % 3 == 0
    run_ok(h)


def test_prepared_call_repeats_the_same_collective():
    """rd.prepare marshals once; every repeat must give the same bits as a
    fresh call, and see policy changes made on the handle in between."""
    R, n = 4, 50001
    h = handle(R)
    set_variant(h, rd.VARIANT_ZS)
    x = inputs(R, n, "bf16", seed=61)
    out = [torch.empty_like(t) for t in x]
    want = oracle.all_reduce(oracle_in(x), dtype="bf16")
    call = rd.prepare(rd.purlin_all_reduce, h, x, out, n, "bf16")
    for variant in (rd.VARIANT_ZS, rd.VARIANT_STAGED, rd.VARIANT_ZS):
        for o in out:
            o.zero_()
        rd.purlin_set_policy(h, 0, 0, 0, variant)
        call()
        run_ok(h)
        for j in range(R):
            assert same_bits(host_bits(out[j]), want[j])
    set_variant(h, rd.VARIANT_ZS)


@pytest.mark.parametrize("fp8", ["float8_e4m3fn", "float8_e5m2"])
def test_fp8_payloads_move_as_bytes(fp8):
    """fp8 (or packed fp4) token payloads of an AllToAllV dispatch are 1-byte
    copies: the binding maps torch's fp8 dtypes to the byte type."""
    if not hasattr(torch, fp8):
        pytest.skip("torch has no " + fp8)
    R = 8
    h = handle(R)
    set_variant(h, rd.VARIANT_ZS)
    C = np.random.default_rng(5).integers(0, 300, size=(R, R)) * 64
    x = [torch.randn(int(C[s].sum()), device="cuda").to(getattr(torch, fp8)) for s in range(R)]
    out = [torch.empty(int(C[:, j].sum()), dtype=x[0].dtype, device="cuda") for j in range(R)]
    rd.purlin_all_to_all_v(h, x, out, C, None, None, x[0].dtype)
    run_ok(h)
    want = oracle.all_to_all_v([t.view(torch.uint8).cpu().numpy() for t in x], C)
    for j in range(R):
        assert same_bits(out[j].view(torch.uint8).cpu().numpy(), want[j])


@pytest.mark.parametrize("policy", ["zs", "zs_large", "snac_default"])
def test_nvfp4_dispatch_and_combine(policy):
    """An NVFP4 MoE dispatch: each token is 7168 e2m1 values packed two per byte
    (3584 payload bytes) plus one e4m3 scale per 16 values (448 bytes).  Both
    streams move as byte AllToAllV copies with per-token byte counts; the
    inverse AllToAllV must give every source its tokens back."""
    R, T, H = 8, 512, workloads.HIDDEN
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    C = workloads.zipf_pair_counts(R, T, workloads.ZIPF_S, workloads.seed_for("moe_a2av_r8", 21))
    g = torch.Generator().manual_seed(77)
    for per_token in (H // 2, H // 16):          # payload, then block scales
        x = [torch.randint(0, 256, (T * per_token,), generator=g, dtype=torch.uint8).cuda()
             for _ in range(R)]
        recv = [torch.empty(int(C[:, j].sum()) * per_token, dtype=torch.uint8, device="cuda")
                for j in range(R)]
        rd.purlin_all_to_all_v(h, x, recv, C * per_token, None, None, "u8")
        back = [torch.empty_like(t) for t in x]
        rd.purlin_all_to_all_v(h, recv, back, C.T * per_token, None, None, "u8")
        run_ok(h)
        want = oracle.all_to_all_v([host_bits(t) for t in x], C * per_token)
        for j in range(R):
            assert same_bits(host_bits(recv[j]), want[j]), (per_token, j)
        for s in range(R):
            assert same_bits(host_bits(back[s]), host_bits(x[s])), (per_token, s)


# Special values of each type as raw bits: signed zeros, the smallest and largest
# subnormals, the smallest normal, the largest finite value, infinities, a quiet
# NaN, and ordinary values near 1 (ties in the final rounding).
SPECIAL_BITS = {
    "f32": [0x00000000, 0x80000000, 0x00000001, 0x807FFFFF, 0x00800000, 0x7F7FFFFF,
            0xFF7FFFFF, 0x7F800000, 0xFF800000, 0x7FC00000, 0x3F800000, 0x3F800001,
            0x33800000, 0xBF800000],
    "bf16": [0x0000, 0x8000, 0x0001, 0x807F, 0x0080, 0x7F7F, 0xFF7F, 0x7F80, 0xFF80, 0x7FC0,
             0x3F80, 0x3F81, 0x3B80, 0xBF80],
    "f16": [0x0000, 0x8000, 0x0001, 0x83FF, 0x0400, 0x7BFF, 0xFBFF, 0x7C00, 0xFC00, 0x7E00,
            0x3C00, 0x3C01, 0x1400, 0xBC00],
}


def _is_nan(bits, dtype):
    if dtype == "f32":
        return np.isnan(bits.view(np.float32))
    exp_mask, man_mask = (0x7F80, 0x007F) if dtype == "bf16" else (0x7C00, 0x03FF)
    b = bits.view(np.uint16)
    return ((b & exp_mask) == exp_mask) & ((b & man_mask) != 0)


@pytest.mark.parametrize("policy", ["zs", "zs_large", "snac_default", "snac_y_default"])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("R", [2, 3, 8])
def test_special_values_sum(policy, dtype, R):
    """Sums over signed zeros, subnormals, overflow to infinity, inf - inf and
    NaN: every non-NaN output bit-exact to the oracle (fold from rank 0's value,
    subnormals kept, one round to nearest even), and NaN exactly where the
    oracle has NaN (payloads are not compared)."""
    n = 3000
    rng = np.random.default_rng(R * 7 + len(dtype))
    pool = np.array(SPECIAL_BITS[dtype], dtype=np.uint32 if dtype == "f32" else np.uint16)
    host = [pool[rng.integers(0, len(pool), size=n)] for _ in range(R)]
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    x = [torch.from_numpy(b.view(np.int32 if dtype == "f32" else np.int16).copy()).cuda()
         .view(TORCH[dtype]) for b in host]
    ar = [Guarded(n, dtype) for _ in range(R)]
    rd.purlin_all_reduce(h, x, [o.view for o in ar], n, dtype)
    run_ok(h)
    want = oracle.all_reduce([host_bits(t) for t in x], dtype=dtype)
    for j in range(R):
        got = host_bits(ar[j].view)
        gi = got.view(np.uint32 if dtype == "f32" else np.uint16)
        wi = want[j].view(np.uint32 if dtype == "f32" else np.uint16)
        nan_w = _is_nan(wi, dtype)
        assert np.array_equal(_is_nan(gi, dtype), nan_w), j
        assert np.array_equal(gi[~nan_w], wi[~nan_w]), j
        assert ar[j].guards_intact()


def test_staged_kinds_share_a_handle():
    """Calls of every staged kind alternate on one handle: each kind's flag words
    (ready / free tags, the y part's tags, the reduced-chunk kinds' step words)
    must never release a wait of another kind (every tag is above 2^32, every
    step word below it)."""
    R, n = 8, 300_000
    h = handle(R)
    x = inputs(R, n, "bf16", seed=61)
    want_ar = oracle.all_reduce(oracle_in(x), dtype="bf16")
    c = n // R
    want_rs = oracle.reduce_scatter(oracle_in(x), [c] * R, dtype="bf16")
    try:
        for rep in range(3):
            for variant, chunk in ((rd.VARIANT_STAGED_Y, 4096), (rd.VARIANT_STAGED, 4096),
                                   (rd.VARIANT_STAGED_Y, 0), (rd.VARIANT_STAGED, 0)):
                set_variant(h, variant, chunk, 2, 0)
                out = [torch.empty_like(t) for t in x]
                rd.purlin_all_reduce(h, x, out, n, "bf16")
                ys = [torch.empty(c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
                rd.purlin_reduce_scatter(h, x, ys, [c] * R, None, "bf16")
                run_ok(h)
                for j in range(R):
                    assert same_bits(host_bits(out[j]), want_ar[j]), (rep, variant, chunk, j)
                    assert same_bits(host_bits(ys[j]), want_rs[j]), (rep, variant, chunk, j)
    finally:
        set_variant(h, rd.VARIANT_AUTO)


@pytest.mark.parametrize("coll,nbytes,small,R", [
    ("ar", 4096, True, 8), ("ar", 1 << 20, True, 8), ("ar", 4 << 20, False, 8),
    ("rs", 256 << 10, True, 8), ("rs", 1 << 20, False, 8),
    ("ag", 1 << 20, True, 8), ("ag", 16 << 20, False, 8),
    # sums of 2 ranks run 4 units per thread; the switch stays at the same size
    ("ar", 1 << 20, True, 2), ("ar", 4 << 20, False, 2),
    ("rs", 256 << 10, True, 2), ("rs", 1 << 20, False, 2),
])
def test_launch_shape_follows_message_size(coll, nbytes, small, R):
    """One-warp CTAs below the per-collective threshold (AllReduce: 256 tiles of
    256 x 32 B; the others: 64 tiles), 256-thread CTAs above it; the result is
    the oracle's either way."""
    n = nbytes // 2
    c = n // R
    h = handle(R)
    set_variant(h, rd.VARIANT_ZS)
    x = inputs(R, n if coll != "ag" else c, "bf16", seed=nbytes % 1000 + len(coll))
    if coll == "ar":
        out = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        rd.purlin_all_reduce(h, x, out, n, "bf16")
        want = oracle.all_reduce(oracle_in(x), dtype="bf16")
    elif coll == "rs":
        out = [torch.empty(c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        rd.purlin_reduce_scatter(h, x, out, [c] * R, None, "bf16")
        want = oracle.reduce_scatter(oracle_in(x), [c] * R, dtype="bf16")
    else:
        out = [torch.empty(R * c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        rd.purlin_all_gather(h, x, out, [c] * R, None, "bf16")
        want = oracle.all_gather(oracle_in(x))
    run_ok(h)
    info = rd.purlin_last_launch(h)
    assert info["block"] == (32 if small else 256), info
    for j in range(R):
        assert same_bits(host_bits(out[j]), want[j]), j


# ------------------------------------------------------------ shifted bodies

@pytest.mark.parametrize("policy", ["zs", "zs_large", "zs_small", "snac_default", "snac_tiny_chunks", "snac_deep", "snac_y_default", "snac_y_tiny_chunks"])
@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("R", [2, 3, 5, 8])
def test_reduce_scatter_shifted_partitions(policy, dtype, R):
    """Partitions whose starts sit off the 32-byte grid while the outputs are
    aligned: the bodies are summed at the sources' alignment and realigned to
    the outputs' (several tiles of warps, a ragged end)."""
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    c = 9 * 1024 + 7 if dtype != "f32" else 5 * 1024 + 3
    x = inputs(R, R * c, dtype, seed=31 * R + len(dtype))
    outs = [Guarded(c, dtype) for _ in range(R)]
    rd.purlin_reduce_scatter(h, x, [o.view for o in outs], [c] * R, None, dtype)
    run_ok(h)
    want = oracle.reduce_scatter(oracle_in(x), [c] * R, dtype=dtype)
    for k in range(R):
        assert same_bits(host_bits(outs[k].view), want[k]), k
        assert outs[k].guards_intact()


@pytest.mark.parametrize("policy", ["zs", "zs_large", "zs_small", "snac_default", "snac_tiny_chunks", "snac_deep", "snac_y_default", "snac_y_tiny_chunks"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("R", [2, 4, 8])
@pytest.mark.parametrize("offset", [1, 3, 6])
def test_all_reduce_shifted_outputs(policy, dtype, R, offset):
    """Aligned inputs, outputs `offset` elements into their allocations."""
    n = 40000 + 11
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    x = inputs(R, n, dtype, seed=700 + R + offset)
    outs = [Guarded(n, dtype, offset=offset) for _ in range(R)]
    rd.purlin_all_reduce(h, x, [o.view for o in outs], n, dtype)
    run_ok(h)
    want = oracle.all_reduce(oracle_in(x), dtype=dtype)
    for j in range(R):
        assert same_bits(host_bits(outs[j].view), want[j]), j
        assert outs[j].guards_intact()


@pytest.mark.parametrize("policy", ["zs", "zs_large", "zs_small", "zs_pull", "snac_default", "snac_tiny_chunks", "snac_deep", "snac_y_default", "snac_y_tiny_chunks"])
@pytest.mark.parametrize("R", [2, 3, 8])
@pytest.mark.parametrize("dtype", ["bf16", "u8"])
def test_all_gather_shifted_blocks(policy, R, dtype):
    """Blocks of lengths that place each rank's block off the 32-byte grid of
    the outputs (copies realigned in registers), several tiles long."""
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    counts = [20000 + 13 * k + (5 if dtype == "u8" else 3) for k in range(R)]
    x = [inputs(1, c, dtype, seed=50 + k)[0] for k, c in enumerate(counts)]
    total = sum(counts)
    outs = [Guarded(total, dtype) for _ in range(R)]
    rd.purlin_all_gather(h, x, [o.view for o in outs], counts, None, dtype)
    run_ok(h)
    want = oracle.all_gather(oracle_in(x))
    for j in range(R):
        assert same_bits(host_bits(outs[j].view), want[j]), j
        assert outs[j].guards_intact()


@pytest.mark.parametrize("policy", ["zs", "zs_large", "zs_small", "snac_default", "snac_tiny_chunks", "snac_deep", "snac_y_default", "snac_y_tiny_chunks"])
@pytest.mark.parametrize("R", [3, 8])
def test_all_to_all_v_shifted_blocks(policy, R):
    """Per-pair counts that are not multiples of 16 bytes: send and receive
    offsets fall on different residues."""
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    rng = np.random.default_rng(R)
    C = rng.integers(3000, 9000, size=(R, R)) | 1
    x = [inputs(1, int(C[s].sum()), "bf16", seed=90 + s)[0] for s in range(R)]
    outs = [Guarded(int(C[:, j].sum()), "bf16") for j in range(R)]
    rd.purlin_all_to_all_v(h, x, [o.view for o in outs], C, None, None, "bf16")
    run_ok(h)
    want = oracle.all_to_all_v(oracle_in(x), C)
    for j in range(R):
        assert same_bits(host_bits(outs[j].view), want[j]), j
        assert outs[j].guards_intact()


@pytest.mark.parametrize("policy", ["zs", "zs_large", "zs_small", "snac_default", "snac_tiny_chunks", "snac_deep", "snac_y_default", "snac_y_tiny_chunks"])
@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("R", [2, 3, 5, 8])
@pytest.mark.parametrize("coll", ["reduce_scatter", "all_reduce"])
def test_sums_with_sources_on_different_grids(policy, dtype, R, coll):
    """Each rank's input `r % 4` elements into its allocation: the ranks' shifts
    differ, so each rank's blocks are realigned on their own before the fold."""
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    c = 6 * 1024 + 5
    n = R * c
    x = [inputs(1, n, dtype, seed=400 + 7 * R + r, offset=r % 4)[0] for r in range(R)]
    if coll == "reduce_scatter":
        outs = [Guarded(c, dtype) for _ in range(R)]
        rd.purlin_reduce_scatter(h, x, [o.view for o in outs], [c] * R, None, dtype)
        want = oracle.reduce_scatter(oracle_in(x), [c] * R, dtype=dtype)
    else:
        outs = [Guarded(n, dtype, offset=1) for _ in range(R)]
        rd.purlin_all_reduce(h, x, [o.view for o in outs], n, dtype)
        want = oracle.all_reduce(oracle_in(x), dtype=dtype)
    run_ok(h)
    for j in range(R):
        assert same_bits(host_bits(outs[j].view), want[j]), j
        assert outs[j].guards_intact()


@pytest.mark.parametrize("policy", ["zs", "zs_large", "zs_small"])
@pytest.mark.parametrize("R", [2, 3, 8])
@pytest.mark.parametrize("dtype", ["bf16", "u8"])
def test_all_gather_outputs_on_different_grids(policy, R, dtype):
    """Outputs `j % 5` elements into their allocations: the gather runs by
    destination, each block realigned to its own output."""
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    counts = [12000 + 7 * k for k in range(R)]
    x = [inputs(1, c, dtype, seed=60 + k)[0] for k, c in enumerate(counts)]
    total = sum(counts)
    outs = [Guarded(total, dtype, offset=j % 5) for j in range(R)]
    rd.purlin_all_gather(h, x, [o.view for o in outs], counts, None, dtype)
    run_ok(h)
    want = oracle.all_gather(oracle_in(x))
    for j in range(R):
        assert same_bits(host_bits(outs[j].view), want[j]), j
        assert outs[j].guards_intact()


@pytest.mark.parametrize("policy", ["zs", "zs_large", "zs_small"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("R", [2, 3, 8])
def test_all_reduce_outputs_on_different_grids(policy, dtype, R):
    """Outputs `j % 3` elements into their allocations (and inputs `r % 2`):
    the sum goes to output 0, then copies to the others -- two launches."""
    n = 30000 + 7
    h = handle(R)
    set_variant(h, *POLICIES[policy])
    x = [inputs(1, n, dtype, seed=800 + 3 * R + r, offset=r % 2)[0] for r in range(R)]
    outs = [Guarded(n, dtype, offset=j % 3) for j in range(R)]
    rd.purlin_all_reduce(h, x, [o.view for o in outs], n, dtype)
    run_ok(h)
    assert rd.purlin_last_launch(h)["kernels"] == 2
    want = oracle.all_reduce(oracle_in(x), dtype=dtype)
    for j in range(R):
        assert same_bits(host_bits(outs[j].view), want[j]), j
        assert outs[j].guards_intact()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_all_reduce_in_place_on_different_grids(dtype):
    """In place (out[r] is in[r]) with the ranks' buffers on different offsets."""
    R, n = 8, 20000 + 3
    h = handle(R)
    set_variant(h, *POLICIES["zs"])
    x = [inputs(1, n, dtype, seed=900 + r, offset=r % 3)[0] for r in range(R)]
    want = oracle.all_reduce(oracle_in(x), dtype=dtype)
    rd.purlin_all_reduce(h, x, x, n, dtype)
    run_ok(h)
    for j in range(R):
        assert same_bits(host_bits(x[j]), want[j]), j


# ------------------------------------------------- staged steps vs channels

@pytest.mark.parametrize("variant", [rd.VARIANT_STAGED, rd.VARIANT_STAGED_Y])
@pytest.mark.parametrize("steps", [3, 4, 5, 8, 9])
def test_staged_steps_around_the_channel_count(variant, steps):
    """A staged call on 4 channels of 4 KiB chunks whose step count sits below,
    at and above the channel count: with one step per channel every role leaves
    after its step, otherwise the channels take further steps from the device
    counter.  AllReduce (the whole vector in `steps` chunks), ReduceScatter and
    AllGather (one piece per rank, `steps` chunks in all where R divides it)."""
    R, chunk = 4, 4096
    h = handle(R)
    set_variant(h, variant, chunk=chunk, depth=2, ctas=4)
    try:
        _staged_steps_case(h, R, chunk, steps)
    finally:
        set_variant(h, rd.VARIANT_AUTO)


def _staged_steps_case(h, R, chunk, steps):
    n = steps * chunk // 2 - 3   # bf16 elements: the last chunk is ragged
    x = inputs(R, n, "bf16", seed=300 + steps)
    out = [Guarded(n, "bf16") for _ in range(R)]
    rd.purlin_all_reduce(h, x, [o.view for o in out], n, "bf16")
    run_ok(h)
    assert rd.purlin_last_launch(h)["chunk_bytes"] == chunk
    want = oracle.all_reduce(oracle_in(x), dtype="bf16")
    for j in range(R):
        assert same_bits(host_bits(out[j].view), want[j]) and out[j].guards_intact()
    # one piece of ceil(steps / R) chunks per rank
    c = -(-steps // R) * chunk // 2 - 1
    x = inputs(R, R * c, "bf16", seed=400 + steps)
    rs = [Guarded(c, "bf16") for _ in range(R)]
    rd.purlin_reduce_scatter(h, x, [o.view for o in rs], [c] * R, None, "bf16")
    run_ok(h)
    want = oracle.reduce_scatter(oracle_in(x), [c] * R, dtype="bf16")
    for j in range(R):
        assert same_bits(host_bits(rs[j].view), want[j]) and rs[j].guards_intact()
    ag = [Guarded(R * c, "bf16") for _ in range(R)]
    rd.purlin_all_gather(h, [o.view for o in rs], [o.view for o in ag], [c] * R, None, "bf16")
    run_ok(h)
    want = np.concatenate([host_bits(o.view) for o in rs])
    for j in range(R):
        assert same_bits(host_bits(ag[j].view), want) and ag[j].guards_intact()


@pytest.mark.parametrize("variant", [rd.VARIANT_STAGED, rd.VARIANT_STAGED_Y])
def test_staged_calls_on_two_handles_at_once(variant):
    """Two handles (each with its own ring, flags and status word) run staged
    AllReduces on two streams at the same time, several calls deep: every call
    must finish and give the oracle's bits.  (The allocation-free AllReduce,
    whose one static array all calls share, is the documented exception.)"""
    R, n = 8, (4 << 20) // 2 + 5
    hs = [rd.purlin_create(R), rd.purlin_create(R)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    try:
        xs = [inputs(R, n, "bf16", seed=500 + k) for k in range(2)]
        wants = [oracle.all_reduce(oracle_in(x), dtype="bf16") for x in xs]
        outs = [[[torch.empty_like(t) for t in xs[k]] for _ in range(3)] for k in range(2)]
        for h in hs:
            set_variant(h, variant)
        torch.cuda.synchronize()
        for rep in range(3):
            for k in range(2):
                with torch.cuda.stream(streams[k]):
                    rd.purlin_all_reduce(hs[k], xs[k], outs[k][rep], n, "bf16",
                                         stream=streams[k])
        torch.cuda.synchronize()
        for k in range(2):
            run_ok(hs[k])
            for rep in range(3):
                for j in range(R):
                    assert same_bits(host_bits(outs[k][rep][j]), wants[k][j]), (k, rep, j)
    finally:
        for h in hs:
            rd.purlin_destroy(h)
