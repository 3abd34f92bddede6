"""Randomized parity: many small random layouts through the C ABI.

Each case draws a collective, R, a dtype, per-rank counts (zeros included), an
element offset for every buffer (unaligned heads and tails), optional explicit
displacements, a datapath (zero staging with one of three copy Atoms, or SNAC
with a random chunk, depth and channel count), the launch shape (one-warp or
256-thread CTAs) and, for sums, the rank order.
The outputs must equal the oracle's bit for bit and the canary guards around
every output must survive.  Run with PURLIN_LIBRARY=checked (after
reduce_datapath_gb300.build(checked=True)) the same cases also assert that no
kernel access left the call's buffers.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import reduce_datapath_gb300 as rd
from helpers import Guarded, close_handles, handle, host_bits, inputs, same_bits

pytestmark = pytest.mark.gpu

# PURLIN_FUZZ_CASES widens the sweep for a soak run (the default keeps the suite
# to seconds).
CASES = int(os.environ.get("PURLIN_FUZZ_CASES", "240"))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rd.build()
    yield
    torch.cuda.synchronize()
    close_handles()


def _layout(rng, counts, gaps):
    """Partition starts in a random order, with random gaps between them."""
    R = len(counts)
    starts = np.zeros(R, dtype=np.int64)
    pos = 0
    for k in rng.permutation(R):
        starts[k] = pos
        pos += int(counts[k]) + (int(rng.integers(0, 5)) if gaps else 0)
    return starts, int(pos)


def _policy(rng, h, copy):
    if rng.random() < 0.5:
        rd.purlin_set_policy(h, 0, 0, int(rng.choice([0, 1, 3, 17])), rd.VARIANT_ZS)
        rd.purlin_set_atom(h, int(rng.choice([rd.ATOM_VECTOR, rd.ATOM_BULK, rd.ATOM_COPY_ENGINE]))
                           if copy else rd.ATOM_AUTO)
        rd.purlin_set_direction(h, int(rng.choice([rd.DIRECTION_PUSH, rd.DIRECTION_PULL])))
        rd.purlin_set_small_tiles(h, int(rng.choice([rd.SMALL_TILES_NEVER, rd.SMALL_TILES_DEFAULT,
                                                     1 << 30])))
    else:
        chunk = int(rng.choice([256, 512, 4096, 16384, 65536]))
        rd.purlin_set_policy(h, chunk, int(rng.integers(1, 9)), int(rng.choice([0, 1, 2, 5])),
                             int(rng.choice([rd.VARIANT_STAGED, rd.VARIANT_STAGED_Y])))
        rd.purlin_set_atom(h, rd.ATOM_AUTO)


@pytest.mark.parametrize("seed", range(CASES))
def test_random_layout(seed):
    _case(seed, 1)


# Fewer, 100x larger cases: many SNAC steps per channel, many tiles per CTA.
LARGE_CASES = int(os.environ.get("PURLIN_FUZZ_LARGE_CASES", "16"))


@pytest.mark.parametrize("seed", range(LARGE_CASES))
def test_random_layout_large(seed):
    _case(50_000 + seed, 100)


def _case(seed, scale):
    rng = np.random.default_rng(1000 + seed)
    coll = ["rs", "ag", "ar", "a2av"][seed % 4]
    R = int(rng.integers(1, 9))
    copy = coll in ("ag", "a2av")
    dtype = str(rng.choice(["f32", "bf16", "f16", "u8"] if copy else ["f32", "bf16", "f16"]))
    h = handle(R)
    _policy(rng, h, copy)
    order = rd.ORDER_TREE if (not copy and rng.random() < 0.3) else rd.ORDER_FIXED
    rd.purlin_set_reduce_order(h, order)
    off = lambda: int(rng.integers(0, 18))
    try:
        if coll == "ar":
            n = int(rng.integers(0, 20000 * scale))
            x = [inputs(1, n, dtype, seed=seed * 10 + r, offset=off())[0] for r in range(R)]
            outs = [Guarded(n, dtype, offset=off()) for _ in range(R)]
            rd.purlin_all_reduce(h, x, [o.view for o in outs], n, dtype)
            xs = [host_bits(t) for t in x]
            if order == rd.ORDER_TREE:
                # pairwise order: the oracle's pairwise sum of the whole vector,
                # placed at every rank
                y = oracle.reduce_scatter(xs, [n] + [0] * (R - 1), dtype=dtype, order="tree")[0]
                want = [y] * R
            else:
                want = oracle.all_reduce(xs, dtype=dtype)
        elif coll == "rs":
            counts = rng.integers(0, 3000 * scale, size=R)
            counts[rng.random(R) < 0.2] = 0
            explicit = rng.random() < 0.5
            displs, total = _layout(rng, counts, explicit) if explicit else (None, int(counts.sum()))
            x = [inputs(1, total, dtype, seed=seed * 10 + r, offset=off())[0] for r in range(R)]
            outs = [Guarded(int(c), dtype, offset=off()) for c in counts]
            rd.purlin_reduce_scatter(h, x, [o.view for o in outs], counts, displs, dtype)
            want = oracle.reduce_scatter([host_bits(t) for t in x], counts, displs, dtype=dtype,
                                         order="tree" if order == rd.ORDER_TREE else "fixed")
        elif coll == "ag":
            counts = rng.integers(0, 3000 * scale, size=R)
            counts[rng.random(R) < 0.2] = 0
            explicit = rng.random() < 0.5
            displs, total = _layout(rng, counts, explicit) if explicit else (None, int(counts.sum()))
            x = [inputs(1, int(c), dtype, seed=seed * 10 + k, offset=off())[0]
                 for k, c in enumerate(counts)]
            outs = [Guarded(total, dtype, offset=off()) for _ in range(R)]
            for o in outs:
                o.view.view(torch.uint8).zero_()
            rd.purlin_all_gather(h, x, [o.view for o in outs], counts, displs, dtype)
            want = oracle.all_gather([host_bits(t) for t in x], counts, displs, out_count=total)
        else:
            C = rng.integers(0, 600 * scale, size=(R, R))
            C[rng.random((R, R)) < 0.25] = 0
            x = [inputs(1, int(C[s].sum()), dtype, seed=seed * 10 + s, offset=off())[0]
                 for s in range(R)]
            outs = [Guarded(int(C[:, j].sum()), dtype, offset=off()) for j in range(R)]
            rd.purlin_all_to_all_v(h, x, [o.view for o in outs], C, None, None, dtype)
            want = oracle.all_to_all_v([host_bits(t) for t in x], C)
        torch.cuda.synchronize()
        assert rd.purlin_query_status(h) == rd.OK
        # under the checked build (PURLIN_LIBRARY=checked) no access may leave
        # the call's buffers; the product build reports 0
        assert rd.purlin_debug_violation(h) == 0
        for j in range(R):
            assert same_bits(host_bits(outs[j].view), want[j]), (coll, R, dtype, j)
            assert outs[j].guards_intact()
    finally:
        rd.purlin_set_reduce_order(h, rd.ORDER_FIXED)
        rd.purlin_set_atom(h, rd.ATOM_AUTO)
        rd.purlin_set_direction(h, rd.DIRECTION_AUTO)
        rd.purlin_set_small_tiles(h, rd.SMALL_TILES_DEFAULT)
        rd.purlin_set_policy(h, 0, 0, 0, rd.VARIANT_AUTO)
