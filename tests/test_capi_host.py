"""Host-side tests of the C-ABI library (no GPU, no kernel launches).

* libpurlin.so loads and exports every symbol that include/*.h declares;
* the layout module's plan (purlin_plan_segments, host only) covers every
  output byte exactly once, maps it to the right source byte per the Figure 4
  layouts, and splits pieces so each access unit is aligned for every stream;
* argument errors are reported as such.
"""
import glob
import os
import re

import numpy as np
import pytest

import reduce_datapath_gb300 as rd
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    rd.build()
    return rd.lib()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"PURLIN_API\s+[\w\s\*]+?\b(purlin_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(rd.EXPORTED)


def test_version_and_status_strings(lib):
    assert rd.purlin_version() >> 16 == 1
    for s in range(7):
        assert rd.purlin_status_string(s) != "unknown status"
    assert rd.purlin_status_string(99) == "unknown status"


def test_null_handle_is_invalid(lib):
    assert lib.purlin_set_policy(None, 0, 0, 0, 0) == rd.ERR_INVALID_ARG
    assert lib.purlin_query_status(None) == rd.ERR_INVALID_ARG
    assert lib.purlin_destroy(None) == rd.OK
    assert lib.purlin_all_reduce(None, None, None, 4, rd.F32, rd.OP_SUM, None) == rd.ERR_INVALID_ARG
    for setter in (lib.purlin_set_atom, lib.purlin_set_direction, lib.purlin_set_small_tiles,
                   lib.purlin_set_reduce_order, lib.purlin_debug_inject):
        assert setter(None, 0) == rd.ERR_INVALID_ARG
    assert lib.purlin_set_timeout(None, 1) == rd.ERR_INVALID_ARG
    assert lib.purlin_last_launch(None, None) == rd.ERR_INVALID_ARG
    # plans: no handle, no plan
    assert lib.purlin_plan_begin(None) == rd.ERR_INVALID_ARG
    assert lib.purlin_plan_end(None, None) == rd.ERR_INVALID_ARG
    assert lib.purlin_plan_launch(None, None) == rd.ERR_INVALID_ARG
    assert lib.purlin_plan_destroy(None) == rd.OK


def test_product_build_is_not_the_checked_one(lib):
    # the checked build (bounds tests in every kernel access) is a separate
    # library; the product one reports itself as unchecked
    assert lib.purlin_debug_checked() == 0
    assert lib.purlin_debug_violation(None, None) == rd.ERR_INVALID_ARG


# ----------------------------------------------------------------- plan tests

def _packed(counts):
    out, s = [], 0
    for c in counts:
        out.append(s)
        s += int(c)
    return out


def expected_map(coll, R, counts, da, db, count, esz):
    """For every output rank: {dst byte -> (src rank or -1, src byte)} from the
    Figure 4 definitions, written as plain loops over partitions."""
    want = [dict() for _ in range(R)]
    if coll == rd.COLL_REDUCE_SCATTER:
        d = da if da is not None else _packed(counts)
        for k in range(R):
            for i in range(int(counts[k]) * esz):
                want[k][i] = (-1, int(d[k]) * esz + i)
    elif coll == rd.COLL_ALL_GATHER:
        D = da if da is not None else _packed(counts)
        for j in range(R):
            for k in range(R):
                for i in range(int(counts[k]) * esz):
                    want[j][int(D[k]) * esz + i] = (k, i)
    elif coll == rd.COLL_ALL_REDUCE:
        for j in range(R):
            for i in range(count * esz):
                want[j][i] = (-1, i)
    else:
        C = np.asarray(counts).reshape(R, R)
        for j in range(R):
            pos = 0
            for s in range(R):
                sd = int(da[s * R + j]) if da is not None else int(sum(C[s, :j]))
                rdsp = int(db[j * R + s]) if db is not None else pos
                for i in range(int(C[s, j]) * esz):
                    want[j][rdsp * esz + i] = (s, sd * esz + i)
                pos += int(C[s, j])
    return want


def plan_map(segs, R):
    got = [dict() for _ in range(R)]
    for s in segs:
        dsts = range(R) if s["dst_rank"] == -1 else [s["dst_rank"]]
        for j in dsts:
            for b in range(s["bytes"]):
                key = s["dst_off"] + b
                assert key not in got[j], "output byte written twice"
                got[j][key] = (s["src_rank"], s["src_off"] + b)
    return got


def check_alignment(segs, R, in_addr, out_addr, reduce, esz):
    if reduce and any(s["shift"] for s in segs):
        # a sum plan holding a shifted body has 16-byte vector bodies throughout
        assert all(s["unit"] in (esz, 16) for s in segs), segs
    for s in segs:
        u = s["unit"]
        assert s["bytes"] % u == 0
        srcs = [in_addr[r] + s["src_off"] for r in range(R)] if s["src_rank"] == -1 \
            else [in_addr[s["src_rank"]] + s["src_off"]]
        dsts = [out_addr[r] + s["dst_off"] for r in range(R)] if s["dst_rank"] == -1 \
            else [out_addr[s["dst_rank"]] + s["dst_off"]]
        if s["shift"]:
            # shifted body: destinations aligned; the first source off their grid
            # is `shift` past a boundary (a copy's one source; a sum's sources
            # each on their own offset, element-aligned)
            assert u in (16, 32) and 0 < s["shift"] < u, s
            for a in dsts:
                assert a % u == 0, (s, a)
            first = next(a % u for a in srcs if a % u)
            assert first == s["shift"], s
            if reduce:
                assert all(a % esz == 0 for a in srcs), s
            else:
                assert len(srcs) == 1
            continue
        for a in srcs + dsts:
            assert a % u == 0, (s, a)
        if reduce:
            assert u in (esz, 16, 32)


def check_tiles(segs, ntiles, reduce, R):
    # sums in the fixed rank order: 4 units per thread for R <= 2, 2 for R <= 4
    unroll = (4 if R <= 2 else 2 if R <= 4 else 1) if reduce else 4
    t = 0
    for s in segs:
        assert s["tile0"] == t
        units = 256 * unroll
        if s["shift"]:
            units = units // 32 * 31   # each warp writes 31 units of 32 lanes' blocks
        tb = units * s["unit"]
        t += -(-s["bytes"] // tb)
    assert t == ntiles


def _addrs(rng, R, misalign, esz):
    base = [(1 << 30) * (r + 1) for r in range(R)]
    if misalign:
        base = [b + int(rng.integers(0, 16)) * esz for b in base]
    return base


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("coll", [rd.COLL_REDUCE_SCATTER, rd.COLL_ALL_GATHER,
                                  rd.COLL_ALL_REDUCE, rd.COLL_ALL_TO_ALL_V])
@pytest.mark.parametrize("dtype", ["bf16", "f32", "u8"])
def test_plan_covers_every_output_byte_once(lib, coll, dtype, seed):
    reduce = coll in (rd.COLL_REDUCE_SCATTER, rd.COLL_ALL_REDUCE)
    if reduce and dtype == "u8":
        pytest.skip("sums take float types only")
    esz = rd.ELEM_BYTES[rd.DTYPES[dtype]]
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, 9))
    misalign = seed % 2 == 1
    in_addr = _addrs(rng, R, misalign, esz)
    out_addr = _addrs(rng, R, misalign, esz)
    counts = da = db = None
    count = 0
    if coll == rd.COLL_ALL_REDUCE:
        count = int(rng.integers(0, 3000))
    elif coll == rd.COLL_ALL_TO_ALL_V:
        counts = workloads.random_pair_counts(R, 300, seed)
        if seed % 3 == 2:   # explicit displacements: reversed packing
            C = counts.reshape(R, R)
            da = np.zeros((R, R), dtype=np.int64)
            db = np.zeros((R, R), dtype=np.int64)
            for s in range(R):
                pos = 0
                for j in reversed(range(R)):
                    da[s, j] = pos
                    pos += C[s, j]
            for j in range(R):
                pos = 0
                for s in reversed(range(R)):
                    db[j, s] = pos
                    pos += C[s, j]
            da, db = da.reshape(-1), db.reshape(-1)
        counts = counts.reshape(-1)
    else:
        counts = workloads.random_counts(R, 700, seed)
        if seed % 3 == 2:
            perm = rng.permutation(R)
            starts = np.zeros(R, dtype=np.int64)
            pos = 0
            for k in perm:
                starts[k] = pos
                pos += counts[k] + int(rng.integers(0, 5))
            da = starts
    segs, ntiles = rd.purlin_plan_segments(coll, R, in_addr, out_addr, counts, da, db, count,
                                           dtype)
    check_alignment(segs, R, in_addr, out_addr, reduce, esz)
    check_tiles(segs, ntiles, reduce, R)
    got = plan_map(segs, R)
    want = expected_map(coll, R, counts, da, db, count, esz)
    assert got == want


def test_aligned_bodies_use_wide_units(lib):
    R = 8
    n = 1 << 16
    in_addr = [(1 << 32) * (r + 1) for r in range(R)]
    out_addr = [(1 << 32) * (r + 9) for r in range(R)]
    segs, _ = rd.purlin_plan_segments(rd.COLL_ALL_REDUCE, R, in_addr, out_addr, count=n,
                                      dtype="bf16")
    assert len(segs) == 1 and segs[0]["unit"] == 32 and segs[0]["bytes"] == 2 * n
    segs, _ = rd.purlin_plan_segments(rd.COLL_ALL_REDUCE, R, in_addr, out_addr, count=n,
                                      dtype="bf16", max_unit=16)
    assert segs[0]["unit"] == 16
    # one source off by one element: a 16-byte body shifted for that rank
    in_addr[3] += 2
    segs, _ = rd.purlin_plan_segments(rd.COLL_ALL_REDUCE, R, in_addr, out_addr, count=n,
                                      dtype="bf16")
    assert [(s["unit"], s["shift"]) for s in segs] == [(16, 2)]
    check_alignment(segs, R, in_addr, out_addr, True, 2)
    # outputs on different alignments: no body fits all of them, element units
    out_addr[5] += 2
    segs, _ = rd.purlin_plan_segments(rd.COLL_ALL_REDUCE, R, in_addr, out_addr, count=n,
                                      dtype="bf16")
    assert [s["unit"] for s in segs] == [2]


def test_plan_rejects_bad_arguments(lib):
    a = [1 << 20, 2 << 20]
    with pytest.raises(rd.PurlinError) as e:
        rd.purlin_plan_segments(rd.COLL_ALL_REDUCE, 9, a * 5, a * 5, count=4, dtype="f32")
    assert e.value.status == rd.ERR_INVALID_ARG
    with pytest.raises(rd.PurlinError) as e:   # misaligned sum stream
        rd.purlin_plan_segments(rd.COLL_ALL_REDUCE, 2, [a[0] + 1, a[1]], a, count=4, dtype="f32")
    assert e.value.status == rd.ERR_INVALID_ARG
    with pytest.raises(rd.PurlinError) as e:   # sums of bytes are not served
        rd.purlin_plan_segments(rd.COLL_ALL_REDUCE, 2, a, a, count=4, dtype="u8")
    assert e.value.status == rd.ERR_UNSUPPORTED
    with pytest.raises(rd.PurlinError) as e:   # counts missing
        rd.purlin_plan_segments(rd.COLL_REDUCE_SCATTER, 2, a, a, None, dtype="f32")
    assert e.value.status == rd.ERR_INVALID_ARG
    with pytest.raises(rd.PurlinError) as e:   # byte count overflows 64 bits
        rd.purlin_plan_segments(rd.COLL_ALL_GATHER, 2, a, a, [2 ** 63, 1], dtype="f32")
    assert e.value.status == rd.ERR_INVALID_ARG


def test_plan_at_maximum_sizes(lib):
    """Huge messages plan without overflow, and a tile count beyond 32 bits is
    refused rather than wrapped."""
    a = [1 << 44, 2 << 44, 3 << 44, 4 << 44, 5 << 44, 6 << 44, 7 << 44, 8 << 44]
    b = [x + (1 << 43) for x in a]
    # 64 GiB of bf16 per rank: 2^23 tiles of 8 KiB at 32-byte units
    segs, nt = rd.purlin_plan_segments(rd.COLL_ALL_REDUCE, 8, a, b, count=1 << 35, dtype="bf16")
    assert len(segs) == 1 and segs[0]["bytes"] == 1 << 36 and nt == (1 << 36) // 8192
    # 2^45 bytes at 32-byte copy units -> 2^32 tiles of 32 KiB: refused
    with pytest.raises(rd.PurlinError) as e:
        rd.purlin_plan_segments(rd.COLL_ALL_GATHER, 1, a[:1], b[:1], [1 << 47], dtype="u8")
    assert e.value.status == rd.ERR_UNSUPPORTED
    # R * R pieces with 3 segments each fit the largest plan
    R = 8
    odd = [x + 1 for x in a]
    C = np.full(R * R, 1001)
    segs, _ = rd.purlin_plan_segments(rd.COLL_ALL_TO_ALL_V, R, odd, b, C, dtype="u8")
    assert len(segs) <= 3 * R * R


def test_offset_partitions_get_shifted_bodies(lib):
    """ReduceScatter of 3 ranks whose partitions start 20 bytes past a 32-byte
    boundary: aligned outputs take 16-byte vector bodies that read the sources
    shifted by 4 (not element by element), and the plan's other bodies are
    16-byte too; the aligned partition 0 is plain.  AllGather placing such
    blocks, the copy analogue, keeps 32-byte units."""
    R, esz = 3, 2
    c = 16 * 1000 + 10                          # 32,020 B per partition: 20 mod 32
    in_addr = [(1 << 32) * (r + 1) for r in range(R)]
    out_addr = [(1 << 32) * (r + 9) for r in range(R)]
    segs, ntiles = rd.purlin_plan_segments(rd.COLL_REDUCE_SCATTER, R, in_addr, out_addr,
                                           [c] * R, dtype="bf16")
    check_alignment(segs, R, in_addr, out_addr, True, esz)
    check_tiles(segs, ntiles, True, R)
    assert all(s["unit"] in (esz, 16) for s in segs)
    body = {s["dst_rank"]: s for s in segs if s["unit"] == 16}
    assert body[0]["shift"] == 0 and body[0]["bytes"] >= c * esz - 16
    for k in (1, 2):
        assert body[k]["shift"] == (k * c * esz) % 16 and body[k]["shift"] != 0
        assert body[k]["bytes"] >= c * esz - 32     # only a sub-vector head and tail
    assert plan_map(segs, R) == expected_map(rd.COLL_REDUCE_SCATTER, R, [c] * R, None, None, 0,
                                             esz)
    # the copy back (AllGather of those partitions into packed outputs): 32-byte
    # bodies shifted by the partitions' offsets
    segs, ntiles = rd.purlin_plan_segments(rd.COLL_ALL_GATHER, R, out_addr, in_addr, [c] * R,
                                           dtype="bf16")
    check_alignment(segs, R, out_addr, in_addr, False, esz)
    check_tiles(segs, ntiles, False, R)
    assert any(s["unit"] == 32 and s["shift"] for s in segs)
