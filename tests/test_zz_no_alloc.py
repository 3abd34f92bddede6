"""The AllReduce entry point that allocates nothing, called through the C ABI.

Some callers cannot call cudaMalloc: a host framework that keeps the GPU's memory
in its own pool, a plugin that may not own device memory, or a latency-critical
path that cannot take the synchronization an allocation may cause.
purlin_all_reduce_noalloc serves them from a fixed static device array.  Here it
must give the same bits as the handle-based purlin_all_reduce and as the CPU
oracle (every sum test in this suite is bit-exact: all follow the fixed rank
order with binary32 accumulation and one rounding) on two calls in a row -- the
second call runs on whatever the first left in the shared array -- and it must
refuse a staging ring that does not fit in that array.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
import reduce_datapath_gb300 as rd
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h8():
    rd.build()
    h = rd.purlin_create(8)
    yield h
    torch.cuda.synchronize()
    rd.purlin_destroy(h)


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


@pytest.mark.parametrize("dtype,n", [("bf16", (1 << 20) + 77), ("f32", 300001)])
def test_matches_all_reduce_on_two_calls_in_a_row(h8, dtype, n):
    R = 8
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rd.purlin_set_policy(h8, 0, 0, 0, rd.VARIANT_ZS)
    for call in range(2):
        x = [workloads.normal_buffer(n, dtype, 9000 + 100 * call + r, device="cuda")
             for r in range(R)]
        want = [torch.empty_like(t) for t in x]
        got = [torch.full_like(t, float("nan")) for t in x]
        rd.purlin_all_reduce(h8, x, want, n, dtype)
        rd.purlin_all_reduce_noalloc(x, got, n, dtype, device_status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        for j in range(R):
            assert torch.equal(_bits(got[j]), _bits(want[j])), (call, j)
        # and directly against the CPU oracle
        ref = oracle.all_reduce([_host(t) for t in x], dtype=dtype)
        for j in (0, R - 1):
            assert np.array_equal(_host(got[j]).view(np.uint8), ref[j].view(np.uint8)), (call, j)


def test_in_place_small_chunks_deep_ring(h8):
    R, n = 4, 123457
    x = [workloads.normal_buffer(n, "f16", 77 + r, device="cuda") for r in range(R)]
    h4 = rd.purlin_create(R)
    try:
        want = [torch.empty_like(t) for t in x]
        rd.purlin_all_reduce(h4, x, want, n, "f16")
        rd.purlin_all_reduce_noalloc(x, x, n, "f16", chunk_bytes=1024, depth=8)
        torch.cuda.synchronize()
        for j in range(R):
            assert torch.equal(_bits(x[j]), _bits(want[j]))
    finally:
        rd.purlin_destroy(h4)


def test_rejects_a_ring_beyond_the_static_array():
    R, n = 8, 1024
    x = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    out = [torch.zeros_like(t) for t in x]
    # 8 slots * 1 MiB = 8 MiB > the 8 MiB array less its 64 KiB of flags
    with pytest.raises(rd.PurlinError) as e:
        rd.purlin_all_reduce_noalloc(x, out, n, "bf16", chunk_bytes=1 << 20, depth=8)
    assert e.value.status == rd.ERR_INVALID_ARG
    with pytest.raises(rd.PurlinError) as e:   # overlapping outputs
        rd.purlin_all_reduce_noalloc(x, [out[0]] * R, n, "bf16")
    assert e.value.status == rd.ERR_INVALID_ARG


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_inputs_off_the_vector_grid_match_the_oracle(dtype):
    """Each rank's input sits r % 4 elements into its allocation, so the ranks'
    sources sit on different alignments; two calls in a row, each checked bit
    for bit against the CPU oracle."""
    R, n = 8, 50000 + 13
    for call in range(2):
        x = []
        for r in range(R):
            full = torch.empty(n + r % 4, dtype=_TORCH[dtype], device="cuda")
            full[r % 4:].copy_(workloads.normal_buffer(n, dtype, 5000 + 50 * call + r,
                                                       device="cuda"))
            x.append(full[r % 4:])
        out = [torch.full((n,), float("nan"), dtype=_TORCH[dtype], device="cuda")
               for _ in range(R)]
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        rd.purlin_all_reduce_noalloc(x, out, n, dtype, device_status=status)
        torch.cuda.synchronize()
        assert status.item() == 0
        want = oracle.all_reduce([_host(t) for t in x], dtype=dtype)
        for j in range(R):
            assert np.array_equal(_host(out[j]).view(np.uint8), want[j].view(np.uint8)), (call, j)


_TORCH = {"bf16": torch.bfloat16, "f32": torch.float32}


def _host(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()
