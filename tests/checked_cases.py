"""Cases run against the checked build of the library (every kernel access
tested against the call's buffers).  Run as a script with PURLIN_LIBRARY=checked
by tests/test_gpu_checked.py; prints one JSON object.

clean: collectives through every path -- zero staging (vector, TMA bulk and
    copy-engine copies, one-warp and 256-thread CTAs), both staged kinds, the
    pairwise order, shifted bodies, the allocation-free AllReduce -- must give
    the oracle's bits and report no access outside their buffers.
planted: a zero-staging ReduceScatter whose first segment's destination the
    debug hook moves one output extent too far, on outputs with room behind
    them: the checked kernel must skip every such store, report
    PURLIN_ERR_BOUNDS and the first address it met, and leave the room behind
    the outputs as it was.
planted_load: the same with the first segment's sources moved one input
    extent too far (inputs with room behind them): the loads are caught and
    the address reported lies in that room.
"""
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import oracle  # noqa: E402
import reduce_datapath_gb300 as rd  # noqa: E402
from helpers import Guarded, host_bits, inputs, same_bits  # noqa: E402

POLICIES = [
    ("zs", (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_AUTO, rd.SMALL_TILES_DEFAULT)),
    ("zs_large", (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_AUTO, rd.SMALL_TILES_NEVER)),
    ("zs_small", (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_AUTO, 1 << 30)),
    ("zs_bulk", (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_BULK, rd.SMALL_TILES_DEFAULT)),
    ("zs_copy_engine", (rd.VARIANT_ZS, 0, 0, 0, rd.ATOM_COPY_ENGINE, rd.SMALL_TILES_DEFAULT)),
    ("snac", (rd.VARIANT_STAGED, 4096, 2, 3, rd.ATOM_AUTO, rd.SMALL_TILES_DEFAULT)),
    ("snac_y", (rd.VARIANT_STAGED_Y, 4096, 3, 3, rd.ATOM_AUTO, rd.SMALL_TILES_DEFAULT)),
]


def set_policy(h, pol):
    variant, chunk, depth, ctas, atom, small = pol
    rd.purlin_set_policy(h, chunk, depth, ctas, variant)
    rd.purlin_set_atom(h, atom)
    rd.purlin_set_small_tiles(h, small)


def report(h, what, failures, buffers):
    """Status and violation of the collective just launched; a violation is
    named by the buffer it falls nearest to."""
    torch.cuda.synchronize()
    st = rd.purlin_query_status(h)
    bad = rd.purlin_debug_violation(h)
    if st == rd.OK and bad == 0:
        return True
    where = ""
    if bad:
        near = min(((abs(bad - t.data_ptr()), name, bad - t.data_ptr(), t.numel() * t.element_size())
                    for name, ts in buffers.items() for t in ts), default=None)
        if near:
            where = f" ({near[2]:+d} B from {near[1]}, {near[3]} B)"
    failures.append(f"{what}: status {st} bad {bad:#x}{where}")
    return False


def clean_cases():
    failures = []
    count = 0
    R = 4
    h = rd.purlin_create(R)
    try:
        for name, pol in POLICIES:
            set_policy(h, pol)
            for order in (rd.ORDER_FIXED, rd.ORDER_TREE):
                rd.purlin_set_reduce_order(h, order)
                for off in (0, 3):   # 3: partitions and buffers off the vector grid
                    c = 3000 + 7 * off
                    x = [inputs(1, R * c, "bf16", seed=40 + r, offset=(r * off) % 4)[0]
                         for r in range(R)]
                    xs = [host_bits(t) for t in x]
                    o = "tree" if order == rd.ORDER_TREE else "fixed"
                    case = f"{name} order {order} offset {off}"
                    rs = [Guarded(c, "bf16") for _ in range(R)]
                    rd.purlin_reduce_scatter(h, x, [g.view for g in rs], [c] * R, None, "bf16")
                    ok = report(h, case + " ReduceScatter", failures,
                                {"input": x, "output": [g.view for g in rs]})
                    ar = [Guarded(R * c, "bf16", offset=off) for _ in range(R)]
                    rd.purlin_all_reduce(h, x, [g.view for g in ar], R * c, "bf16")
                    ok &= report(h, case + " AllReduce", failures,
                                 {"input": x, "output": [g.view for g in ar]})
                    ag = [Guarded(R * c, "bf16", offset=off) for _ in range(R)]
                    rd.purlin_all_gather(h, [g.view for g in rs], [g.view for g in ag], [c] * R,
                                         None, "bf16")
                    ok &= report(h, case + " AllGather", failures,
                                 {"input": [g.view for g in rs], "output": [g.view for g in ag]})
                    C = np.array([[(c // R) + s + j for j in range(R)] for s in range(R)])
                    xa = [inputs(1, int(C[s].sum()), "bf16", seed=60 + s, offset=off)[0]
                          for s in range(R)]
                    a2 = [Guarded(int(C[:, j].sum()), "bf16") for j in range(R)]
                    rd.purlin_all_to_all_v(h, xa, [g.view for g in a2], C, None, None, "bf16")
                    ok &= report(h, case + " AllToAllV", failures,
                                 {"input": xa, "output": [g.view for g in a2]})
                    want_rs = oracle.reduce_scatter(xs, [c] * R, dtype="bf16", order=o)
                    want_ar = np.concatenate(want_rs)
                    want_a2 = oracle.all_to_all_v([host_bits(t) for t in xa], C)
                    bits = True
                    for j in range(R):
                        bits &= same_bits(host_bits(rs[j].view), want_rs[j])
                        bits &= same_bits(host_bits(ar[j].view), want_ar)
                        bits &= same_bits(host_bits(ag[j].view), want_ar)
                        bits &= same_bits(host_bits(a2[j].view), want_a2[j])
                        bits &= all(g.guards_intact() for g in (rs[j], ar[j], ag[j], a2[j]))
                    count += 1
                    if ok and not bits:
                        failures.append(f"{case}: results differ from the oracle")
            rd.purlin_set_reduce_order(h, rd.ORDER_FIXED)
    finally:
        rd.purlin_destroy(h)
    # the allocation-free AllReduce
    n = 40000 + 11
    x = [inputs(1, n, "bf16", seed=90 + r)[0] for r in range(R)]
    out = [torch.empty_like(t) for t in x]
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rd.purlin_all_reduce_noalloc(x, out, n, "bf16", chunk_bytes=4096, device_status=status)
    torch.cuda.synchronize()
    want = oracle.all_reduce([host_bits(t) for t in x], dtype="bf16")
    count += 1
    if int(status.item()) != 0 or not all(same_bits(host_bits(out[j]), want[j]) for j in range(R)):
        failures.append(f"noalloc: status {int(status.item())}")
    return count, failures


def planted_load_case():
    """The first segment's sources one input extent too far: every load there
    lies wholly outside the inputs and must be caught (aligned blocks that only
    straddle a buffer's end are allowed; these do not touch it)."""
    R, c = 4, 8192 + 5
    h = rd.purlin_create(R)
    try:
        set_policy(h, POLICIES[1][1])
        n = R * c
        full = [torch.zeros(3 * n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        for r in range(R):
            full[r][:n].copy_(inputs(1, n, "bf16", seed=80 + r)[0])
        x = [t[:n] for t in full]
        outs = [torch.full((c,), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        rd.purlin_debug_inject(h, 3)
        rd.purlin_reduce_scatter(h, x, outs, [c] * R, None, "bf16")
        torch.cuda.synchronize()
        st = rd.purlin_query_status(h)
        bad = rd.purlin_debug_violation(h)
        ext = n * 2
        in_room = any(t.data_ptr() + ext <= bad < t.data_ptr() + 2 * ext for t in full)
        return {"status": int(st), "violation_in_room": bool(in_room)}
    finally:
        rd.purlin_destroy(h)


def planted_case():
    R, c = 4, 8192 + 5
    h = rd.purlin_create(R)
    try:
        set_policy(h, POLICIES[1][1])
        x = [inputs(1, R * c, "bf16", seed=70 + r)[0] for r in range(R)]
        # each output is the first third of its allocation; the planted
        # destination lands in the second third
        full = [torch.full((3 * c,), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
        outs = [t[:c] for t in full]
        rd.purlin_debug_inject(h, 2)
        rd.purlin_reduce_scatter(h, x, outs, [c] * R, None, "bf16")
        torch.cuda.synchronize()
        st = rd.purlin_query_status(h)
        bad = rd.purlin_debug_violation(h)
        bases = [t.data_ptr() for t in full]
        ext = c * 2
        in_room = any(b + ext <= bad < b + 2 * ext for b in bases)
        room_intact = all(bool(torch.all(t[c:] == 7.0).item()) for t in full)
        return {"status": int(st), "violation_in_room": bool(in_room),
                "room_intact": room_intact}
    finally:
        rd.purlin_destroy(h)


def main():
    rd.lib()
    result = {"checked": rd.purlin_debug_checked()}
    count, failures = clean_cases()
    result["clean_cases"] = count
    result["clean_failures"] = failures
    result["planted"] = planted_case()
    result["planted_load"] = planted_load_case()
    print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()
