"""Parity at the workloads' full sizes, in the launch configurations the
benchmark times.

  allreduce_r2_f32     AllReduce R=2 fp32 4096 integers in [-8, 8] (exact sums),
                       plus ReduceScatter + AllGather on the same inputs.
  rs_ag_r8_bf16        ReduceScatter then AllGather, R=8 bf16, 64 MiB per rank:
                       compared in full with the oracle; the same size summed
                       over 2 and 4 ranks (bf16 and fp32), in full.
  allreduce_sweep_r8   AllReduce R=8 bf16, 4 KiB .. 256 MiB per rank, zero staging
                       and SNAC chunks of 64 KiB .. 2 MiB: in full up to 16 MiB
                       per rank, sampled above (the oracle recomputes sampled
                       elements from the gathered inputs), plus "all R outputs
                       are identical" in full.
  moe_a2av_r8          AllToAllV dispatch, R=8, 4096 tokens x 7168 bf16 per
                       source, Zipf(1.2) destinations: in full, then the inverse
                       AllToAllV must give back every source buffer.
  dp_attn_agv_rsv_r8   AllGatherV + ReduceScatterV with token counts uniform in
                       [1, 2048] x 7168 bf16: in full; plus a 1 GiB-per-rank
                       output AllGather and a 1 GiB-per-rank AllReduce, sampled
                       plus full-size layout properties.
"""
import numpy as np
import pytest
import torch

import oracle
import reduce_datapath_gb300 as rd
import workloads
from helpers import host_bits

pytestmark = pytest.mark.gpu

MiB = 1 << 20
GiB = 1 << 30


@pytest.fixture(scope="module", autouse=True)
def _lib():
    rd.build()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _ok(h):
    torch.cuda.synchronize()
    assert rd.purlin_query_status(h) == rd.OK


def _bits_equal(a, b):
    return a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8))


def _sample_idx(n, k, seed):
    rng = np.random.default_rng(seed)
    idx = np.unique(rng.integers(0, n, size=k))
    idx = np.concatenate([[0, n - 1], idx])
    return torch.from_numpy(np.unique(idx)).cuda()


# --------------------------------------------------------------- allreduce_r2_f32

@pytest.mark.parametrize("variant", [rd.VARIANT_ZS, rd.VARIANT_STAGED, rd.VARIANT_STAGED_Y])
def test_allreduce_r2_f32_integers(variant):
    R, n = 2, 4096
    x = workloads.rank_buffers("allreduce_r2_f32", R, n, "f32", device="cuda", values="int")
    h = rd.purlin_create(R)
    try:
        rd.purlin_set_policy(h, 0, 0, 0, variant)
        ar = [torch.empty(n, device="cuda") for _ in range(R)]
        rd.purlin_all_reduce(h, x, ar, n, "f32")
        y = [torch.empty(n // R, device="cuda") for _ in range(R)]
        z = [torch.empty(n, device="cuda") for _ in range(R)]
        rd.purlin_reduce_scatter(h, x, y, [n // R] * R, None, "f32")
        rd.purlin_all_gather(h, y, z, [n // R] * R, None, "f32")
        _ok(h)
    finally:
        rd.purlin_destroy(h)
    xs = [host_bits(t) for t in x]
    exact = np.sum(np.stack(xs).astype(np.int64), axis=0)
    want = oracle.all_reduce(xs, dtype="f32")
    for j in range(R):
        got = host_bits(ar[j])
        assert _bits_equal(got, want[j])
        assert np.array_equal(got.astype(np.int64), exact)
        assert _bits_equal(host_bits(z[j]), got)       # AR == AG(RS)


# -------------------------------------------------------------- rs_ag_r8_bf16

@pytest.mark.parametrize("variant", [rd.VARIANT_ZS, rd.VARIANT_STAGED, rd.VARIANT_STAGED_Y])
def test_rs_ag_r8_bf16_64MiB_full(variant):
    R, n = 8, 64 * MiB // 2
    c = n // R
    x = workloads.rank_buffers("rs_ag_r8_bf16", R, n, "bf16", device="cuda")
    y = [torch.empty(c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    z = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    h = rd.purlin_create(R)
    try:
        rd.purlin_set_policy(h, 0, 0, 0, variant)
        rd.purlin_reduce_scatter(h, x, y, [c] * R, None, "bf16")
        rd.purlin_all_gather(h, y, z, [c] * R, None, "bf16")
        _ok(h)
    finally:
        rd.purlin_destroy(h)
    xs = [host_bits(t) for t in x]
    del x
    want_y = oracle.reduce_scatter(xs, [c] * R, dtype="bf16")
    del xs
    for k in range(R):
        assert _bits_equal(host_bits(y[k]), want_y[k]), k
    want_z = np.concatenate(want_y)
    for j in range(R):
        assert _bits_equal(host_bits(z[j]), want_z), j



# ----------------------------------------------------- sums of 2 and 4 ranks

@pytest.mark.parametrize("coll", ["all_reduce", "reduce_scatter"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("R", [2, 4])
def test_rank_count_sums_64MiB_full(R, dtype, coll):
    """The benchmark's rank-count study (64 MiB per rank, zero staging, 4 or 2
    units per thread), compared in full with the oracle."""
    esz = 2 if dtype == "bf16" else 4
    n = 64 * MiB // esz
    c = n // R
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = workloads.rank_buffers("rs_ag_r8_bf16", R, n, dtype, role=10 + R, device="cuda")
    h = rd.purlin_create(R)
    try:
        if coll == "all_reduce":
            out = [torch.empty(n, dtype=tdt, device="cuda") for _ in range(R)]
            rd.purlin_all_reduce(h, x, out, n, dtype)
        else:
            out = [torch.empty(c, dtype=tdt, device="cuda") for _ in range(R)]
            rd.purlin_reduce_scatter(h, x, out, [c] * R, None, dtype)
        _ok(h)
        assert rd.purlin_last_launch(h)["block"] == 256
    finally:
        rd.purlin_destroy(h)
    xs = [host_bits(t) for t in x]
    del x
    if coll == "all_reduce":
        want = oracle.all_reduce(xs, dtype=dtype)
    else:
        want = oracle.reduce_scatter(xs, [c] * R, dtype=dtype)
    for j in range(R):
        assert _bits_equal(host_bits(out[j]), want[j]), j

# ---------------------------------------------------------- allreduce_sweep_r8

def _check_allreduce(x, out, n, sampled, seed):
    R = len(x)
    for j in range(1, R):   # any size: every rank holds the same result
        assert torch.equal(out[j].view(torch.int16), out[0].view(torch.int16))
    if not sampled:
        want = oracle.all_reduce([host_bits(t) for t in x], dtype="bf16")
        assert _bits_equal(host_bits(out[0]), want[0])
        return
    idx = _sample_idx(n, 1 << 16, seed)
    mini = [host_bits(t[idx]) for t in x]
    want = oracle.all_reduce(mini, dtype="bf16")
    assert _bits_equal(host_bits(out[0][idx]), want[0])


SWEEP = [(b, v, ch) for b in workloads.SWEEP_BYTES for (v, ch) in
         [(rd.VARIANT_ZS, 0), (rd.VARIANT_STAGED, 0), (rd.VARIANT_STAGED, 64 * 1024),
          (rd.VARIANT_STAGED, 256 * 1024), (rd.VARIANT_STAGED, 1 * MiB), (rd.VARIANT_STAGED, 2 * MiB),
          (rd.VARIANT_STAGED_Y, 0), (rd.VARIANT_STAGED_Y, 64 * 1024),
          (rd.VARIANT_STAGED_Y, 2 * MiB)]]


@pytest.fixture(scope="module")
def sweep_handle():
    # room for 2 MiB chunks: depth 2 x (8 + 1) parts x 2 MiB = 36 MiB per channel
    h = rd.purlin_create(8, 160 * MiB)
    yield h
    torch.cuda.synchronize()
    rd.purlin_destroy(h)


@pytest.mark.parametrize("nbytes,variant,chunk", SWEEP,
                         ids=[f"{b >> 10}KiB-{ {1: 'zs', 2: 'snac', 3: 'snac_y'}[v] }-{c >> 10}K"
                              for b, v, c in SWEEP])
def test_allreduce_sweep_r8(sweep_handle, nbytes, variant, chunk):
    R, n = 8, nbytes // 2
    h = sweep_handle
    rd.purlin_set_policy(h, chunk, 0, 0, variant)
    x = workloads.rank_buffers("allreduce_sweep_r8", R, n, "bf16", device="cuda",
                               role=nbytes.bit_length())
    out = [torch.empty_like(t) for t in x]
    rd.purlin_all_reduce(h, x, out, n, "bf16")
    _ok(h)
    _check_allreduce(x, out, n, sampled=nbytes > 16 * MiB, seed=nbytes)


@pytest.mark.parametrize("variant", [rd.VARIANT_ZS, rd.VARIANT_STAGED, rd.VARIANT_STAGED_Y])
def test_allreduce_sweep_256MiB_full(sweep_handle, variant):
    """The largest point of the AllReduce sweep (256 MiB per rank, R=8, bf16)
    compared in full with the oracle, not on a sample."""
    R, n = 8, 256 * MiB // 2
    h = sweep_handle
    rd.purlin_set_policy(h, 0, 0, 0, variant)
    x = workloads.rank_buffers("allreduce_sweep_r8", R, n, "bf16", device="cuda",
                               role=(256 * MiB).bit_length())
    out = [torch.empty_like(t) for t in x]
    rd.purlin_all_reduce(h, x, out, n, "bf16")
    _ok(h)
    for j in range(1, R):
        assert torch.equal(out[j].view(torch.int16), out[0].view(torch.int16)), j
    xs = [host_bits(t) for t in x]
    del x
    want = oracle.all_reduce(xs, dtype="bf16")
    del xs
    assert _bits_equal(host_bits(out[0]), want[0])


# ---------------------------------------------------------------- moe_a2av_r8

ATOMS = [(rd.VARIANT_ZS, rd.ATOM_VECTOR), (rd.VARIANT_ZS, rd.ATOM_BULK),
         (rd.VARIANT_ZS, rd.ATOM_COPY_ENGINE), (rd.VARIANT_STAGED, rd.ATOM_AUTO),
         (rd.VARIANT_STAGED_Y, rd.ATOM_AUTO)]


@pytest.mark.parametrize("variant,atom", ATOMS)
def test_moe_a2av_r8_dispatch_and_inverse(variant, atom):
    R, T, H = 8, 4096, workloads.HIDDEN
    C = workloads.zipf_pair_counts(R, T, workloads.ZIPF_S, workloads.seed_for("moe_a2av_r8", 9))
    assert (C.sum(axis=1) == T).all()
    x = workloads.rank_buffers("moe_a2av_r8", R, T * H, "bf16", device="cuda")
    recv = [torch.empty(int(C[:, j].sum()) * H, dtype=torch.bfloat16, device="cuda")
            for j in range(R)]
    back = [torch.empty_like(t) for t in x]
    h = rd.purlin_create(R)
    try:
        rd.purlin_set_policy(h, 0, 0, 0, variant)
        rd.purlin_set_atom(h, atom)
        rd.purlin_all_to_all_v(h, x, recv, C * H, None, None, "bf16")
        rd.purlin_all_to_all_v(h, recv, back, C.T * H, None, None, "bf16")
        _ok(h)
    finally:
        rd.purlin_destroy(h)
    for s in range(R):   # the inverse gives every token back to its source
        assert torch.equal(back[s].view(torch.int16), x[s].view(torch.int16)), s
    want = oracle.all_to_all_v([host_bits(t) for t in x], C * H)
    for j in range(R):
        assert _bits_equal(host_bits(recv[j]), want[j]), j
    # the skew the workload asks for: rank 0 receives the most tokens
    assert C[:, 0].sum() == C.sum(axis=0).max()


# ---------------------------------------------------------- dp_attn_agv_rsv_r8

@pytest.mark.parametrize("variant", [rd.VARIANT_ZS, rd.VARIANT_STAGED, rd.VARIANT_STAGED_Y])
def test_dp_attention_agv_rsv(variant):
    R, H = 8, workloads.HIDDEN
    tok = workloads.uniform_token_counts(R, 1, 2048, workloads.seed_for("dp_attn_agv_rsv_r8", 9))
    counts = tok * H
    T = int(counts.sum())
    ag_in = [workloads.normal_buffer(int(counts[k]), "bf16",
                                     workloads.seed_for("dp_attn_agv_rsv_r8", 1, k), "cuda")
             for k in range(R)]
    ag_out = [torch.empty(T, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    rs_in = workloads.rank_buffers("dp_attn_agv_rsv_r8", R, T, "bf16", role=2, device="cuda")
    rs_out = [torch.empty(int(c), dtype=torch.bfloat16, device="cuda") for c in counts]
    h = rd.purlin_create(R)
    try:
        rd.purlin_set_policy(h, 0, 0, 0, variant)
        rd.purlin_all_gather(h, ag_in, ag_out, counts, None, "bf16")
        rd.purlin_reduce_scatter(h, rs_in, rs_out, counts, None, "bf16")
        _ok(h)
    finally:
        rd.purlin_destroy(h)
    want = oracle.all_gather([host_bits(t) for t in ag_in], counts)
    for j in range(R):
        assert _bits_equal(host_bits(ag_out[j]), want[j])
    want = oracle.reduce_scatter([host_bits(t) for t in rs_in], counts, dtype="bf16")
    for k in range(R):
        assert _bits_equal(host_bits(rs_out[k]), want[k])


@pytest.mark.parametrize("variant,atom", ATOMS)
def test_allgather_1GiB_out_per_rank(variant, atom):
    R = 8
    c = 128 * MiB // 2
    x = workloads.rank_buffers("dp_attn_agv_rsv_r8", R, c, "bf16", role=3, device="cuda")
    out = [torch.empty(R * c, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    h = rd.purlin_create(R)
    try:
        rd.purlin_set_policy(h, 0, 0, 0, variant)
        rd.purlin_set_atom(h, atom)
        rd.purlin_all_gather(h, x, out, [c] * R, None, "bf16")
        _ok(h)
    finally:
        rd.purlin_destroy(h)
    for j in range(R):   # full size: every block where Figure 4 puts it
        for k in range(R):
            assert torch.equal(out[j][k * c:(k + 1) * c].view(torch.int16), x[k].view(torch.int16))
    idx = _sample_idx(c, 1 << 14, 5)
    mini = [host_bits(t[idx]) for t in x]
    want = oracle.all_gather(mini)
    S = idx.numel()
    for j in range(R):
        got = np.concatenate([host_bits(out[j][k * c + idx]) for k in range(R)])
        assert _bits_equal(got, want[j])
    del out, x
    torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", [rd.VARIANT_ZS, rd.VARIANT_STAGED, rd.VARIANT_STAGED_Y])
def test_allreduce_1GiB_per_rank(variant):
    R, n = 8, GiB // 2
    x = workloads.rank_buffers("dp_attn_agv_rsv_r8", R, n, "bf16", role=4, device="cuda")
    out = [torch.empty_like(t) for t in x]
    h = rd.purlin_create(R)
    try:
        rd.purlin_set_policy(h, 0, 0, 0, variant)
        rd.purlin_all_reduce(h, x, out, n, "bf16")
        _ok(h)
    finally:
        rd.purlin_destroy(h)
    _check_allreduce(x, out, n, sampled=True, seed=11)
    del out, x
    torch.cuda.empty_cache()
