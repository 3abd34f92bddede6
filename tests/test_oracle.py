"""Pins for the CPU oracle (runs without a GPU).

The oracle is trusted only because of these tests, which check it against things
other than itself:
  * library codecs (torch's and numpy's float narrowing/widening) for the
    bfloat16/float16 conversions, exhaustively where the domain is small;
  * hand-worked examples from the pages' Figure 4/6 layouts (tests/golden/);
  * hand-derived IEEE cases that fix the fold order, the start value and the
    single rounding (tests/golden/fold_rounding.json);
  * exact integer sums, an error bound against the exact (float64) sum, and the
    invariants AR == AG(RS), A2A(A2A) == id, A2AV followed by its inverse == id,
    "V with equal counts == fixed", R = 1 == copy.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_torch_bf16(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


def same_bits_or_both_nan(a_bits, b_bits, a_float, b_float):
    nan_a, nan_b = np.isnan(a_float), np.isnan(b_float)
    assert np.array_equal(nan_a, nan_b)
    assert np.array_equal(a_bits[~nan_a], b_bits[~nan_b])


def _f32_probe_bits(rng, n_random):
    """Random binary32 bit patterns plus patterns around every rounding boundary."""
    rand = rng.integers(0, 2 ** 32, size=n_random, dtype=np.uint64).astype(np.uint32)
    special = np.array([0x00000000, 0x80000000, 0x7f800000, 0xff800000, 0x7fc00000,
                        0x7f800001, 0xffc00001, 0x00000001, 0x807fffff, 0x7f7fffff,
                        0xff7fffff, 0x477fe000, 0x477fefff, 0x477ff000, 0x477ff001,
                        0x38800000, 0x387fffff, 0x33800000, 0x33000000, 0x33000001,
                        0x337fffff, 0x32ffffff], dtype=np.uint32)
    return np.concatenate([rand, special])


class TestCodecs:
    def test_bf16_widen_exhaustive(self):
        bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
        ours = oracle.bf16_to_f32(bits)
        ref = bits_to_torch_bf16(bits).float().numpy()
        same_bits_or_both_nan(ours.view(np.uint32), ref.view(np.uint32), ours, ref)

    def test_f16_widen_exhaustive(self):
        bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
        ours = oracle.f16_to_f32(bits)
        ref = bits.view(np.float16).astype(np.float32)
        same_bits_or_both_nan(ours.view(np.uint32), ref.view(np.uint32), ours, ref)

    def test_bf16_narrow_matches_torch(self):
        rng = np.random.default_rng(1)
        # every bfloat16 value, the exact midpoint above it and one ulp either side
        hi = np.arange(1 << 16, dtype=np.uint32) << 16
        around = np.concatenate([hi, hi | 0x8000, hi | 0x7fff, hi | 0x8001, hi | 0x0001])
        probe = np.concatenate([_f32_probe_bits(rng, 1 << 20), around]).view(np.float32)
        ours = oracle.f32_to_bf16(probe)
        ref = bf16_bits(torch.from_numpy(probe.copy()).to(torch.bfloat16))
        same_bits_or_both_nan(ours, ref, oracle.bf16_to_f32(ours), oracle.bf16_to_f32(ref))
        assert np.array_equal(np.isnan(oracle.bf16_to_f32(ours)), np.isnan(probe))

    def test_f16_narrow_matches_numpy(self):
        rng = np.random.default_rng(2)
        # every float16 value widened, the midpoint to its successor and +-1 ulp of it
        vals = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
        vals = vals[np.isfinite(vals)].astype(np.float64)
        vals = np.unique(vals)
        mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
        m = mids.view(np.uint32)
        around = np.concatenate([vals.astype(np.float32).view(np.uint32), m, m + 1, m - 1])
        # the overflow threshold and the subnormal range, densely
        dense = np.arange(0x477fe000, 0x47800100, dtype=np.uint32)
        tiny = np.arange(0x32f00000, 0x33900000, 97, dtype=np.uint32)
        probe = np.concatenate([_f32_probe_bits(rng, 1 << 20), around, dense, tiny,
                                dense | 0x80000000]).view(np.float32)
        ours = oracle.f32_to_f16(probe)
        with np.errstate(over="ignore", invalid="ignore"):
            ref = probe.astype(np.float16).view(np.uint16)
        same_bits_or_both_nan(ours, ref, ours.view(np.float16), ref.view(np.float16))
        assert np.array_equal(np.isnan(ours.view(np.float16)), np.isnan(probe))


# ----------------------------------------------------------------------------- golden

def _as(dtype, values):
    if dtype == "f32":
        return np.asarray(values, dtype=np.float32)
    raise AssertionError(dtype)


class TestGolden:
    def test_fig4_three_ranks(self):
        g = _golden("fig4_three_ranks.json")
        x = [_as("f32", v) for v in g["x"]]
        y = oracle.reduce_scatter(x, g["reduce_scatter"]["recv_counts"], dtype="f32")
        assert [list(v) for v in y] == g["reduce_scatter"]["y"]
        ag = oracle.all_gather(y)
        assert [list(v) for v in ag] == g["all_gather_of_y"]["out"]
        ar = oracle.all_reduce(x, dtype="f32")
        assert [list(v) for v in ar] == g["all_reduce"]["out"]
        R = g["R"]
        c = g["all_to_all"]["count_per_pair"]
        a2a = oracle.all_to_all_v(x, np.full((R, R), c))
        assert [list(v) for v in a2a] == g["all_to_all"]["out"]

    def test_two_rank_sum(self):
        g = _golden("two_rank_sum.json")
        x = [_as("f32", v) for v in g["x"]]
        y = oracle.reduce_scatter(x, g["reduce_scatter"]["recv_counts"], dtype="f32")
        assert [list(v) for v in y] == g["reduce_scatter"]["y"]
        ar = oracle.all_reduce(x, dtype="f32")
        assert [list(v) for v in ar] == g["all_reduce"]["out"]

    def test_variable_length(self):
        g = _golden("variable_length.json")
        for case in g["reduce_scatter_v"]:
            x = [_as("f32", v) for v in case["x"]]
            y = oracle.reduce_scatter(x, case["recv_counts"], case["in_displs"], dtype="f32")
            assert [list(v) for v in y] == case["y"]
        for case in g["all_gather_v"]:
            ins = [_as("f32", v) for v in case["in"]]
            out = oracle.all_gather(ins, case["counts"], case["out_displs"])
            assert [list(v) for v in out] == case["out"]
        for case in g["all_to_all_v"]:
            ins = [_as("f32", v) for v in case["in"]]
            out = oracle.all_to_all_v(ins, case["send_counts"], case["send_displs"],
                                      case["recv_displs"])
            assert [list(v) for v in out] == case["out"]

    @pytest.mark.parametrize("order", ["fixed", "tree"])
    def test_fold_rounding(self, order):
        g = _golden("fold_rounding.json")
        for case in g["cases"]:
            dt = case["dtype"]
            if dt == "f32":
                x = [np.asarray([v], dtype=np.float32) for v in case["x"]]
            else:
                x = [np.asarray([int(b, 16)], dtype=np.uint16) for b in case["x_bits"]]
            R = len(x)
            counts = [0] * R
            counts[0] = 1
            y = oracle.reduce_scatter(x, counts, dtype=dt, order=order)[0]
            want = int(case[order + "_bits"], 16)
            got = int(y.view(np.uint32 if dt == "f32" else np.uint16)[0])
            assert got == want, (case["name"], order, hex(got))
            if order == "fixed":
                ar = oracle.all_reduce(x, dtype=dt)
                for o in ar:
                    assert int(o.view(np.uint32 if dt == "f32" else np.uint16)[0]) == want


# ------------------------------------------------------------------------- invariants

def _normal(rng, n, dtype):
    f = rng.standard_normal(n).astype(np.float32)
    if dtype == "f32":
        return f
    if dtype == "bf16":
        return bf16_bits(torch.from_numpy(f).to(torch.bfloat16))
    return f.astype(np.float16).view(np.uint16)


def _to_f64(a, dtype):
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "bf16":
        return bits_to_torch_bf16(a).double().numpy()
    return a.view(np.float16).astype(np.float64)


def _packed(counts):
    return list(np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int64))


class TestInvariants:
    @pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
    @pytest.mark.parametrize("R", [1, 2, 3, 5, 8])
    def test_allreduce_equals_allgather_of_reducescatter(self, R, dtype):
        rng = np.random.default_rng(10 + R)
        counts = rng.integers(0, 40, size=R)
        N = int(counts.sum())
        x = [_normal(rng, N, dtype) for _ in range(R)]
        ar = oracle.all_reduce(x, dtype=dtype)
        y = oracle.reduce_scatter(x, counts, dtype=dtype)
        ag = oracle.all_gather(y, counts, out_count=N)
        for j in range(R):
            assert np.array_equal(ar[j], ag[j])

    @pytest.mark.parametrize("R", [1, 2, 4, 7, 8])
    def test_alltoall_twice_is_identity(self, R):
        rng = np.random.default_rng(20 + R)
        c = 5
        ins = [rng.integers(0, 2 ** 16, size=R * c, dtype=np.uint16) for _ in range(R)]
        C = np.full((R, R), c)
        once = oracle.all_to_all_v(ins, C)
        twice = oracle.all_to_all_v(once, C)
        for j in range(R):
            assert np.array_equal(twice[j], ins[j])
        if R > 1:  # and once is not the identity
            assert any(not np.array_equal(once[j], ins[j]) for j in range(R))

    @pytest.mark.parametrize("R", [2, 3, 8])
    def test_alltoallv_then_inverse_is_identity(self, R):
        rng = np.random.default_rng(30 + R)
        C = rng.integers(0, 9, size=(R, R))
        ins = [rng.integers(0, 2 ** 16, size=int(C[s].sum()), dtype=np.uint16)
               for s in range(R)]
        fwd = oracle.all_to_all_v(ins, C)
        back = oracle.all_to_all_v(fwd, C.T)
        for s in range(R):
            assert np.array_equal(back[s], ins[s])

    @pytest.mark.parametrize("R", [2, 5, 8])
    def test_v_with_equal_counts_matches_fixed(self, R):
        rng = np.random.default_rng(40 + R)
        c = 6
        x = [_normal(rng, R * c, "bf16") for _ in range(R)]
        fixed = oracle.reduce_scatter(x, [c] * R, None, dtype="bf16")
        v = oracle.reduce_scatter(x, [c] * R, [k * c for k in range(R)], dtype="bf16")
        for k in range(R):
            assert np.array_equal(fixed[k], v[k])
        ag_f = oracle.all_gather(fixed)
        ag_v = oracle.all_gather(fixed, [c] * R, [k * c for k in range(R)])
        for j in range(R):
            assert np.array_equal(ag_f[j], ag_v[j])
        ins = [rng.integers(0, 2 ** 16, size=R * c, dtype=np.uint16) for _ in range(R)]
        C = np.full((R, R), c)
        sd = np.tile(np.arange(R) * c, (R, 1))
        a_f = oracle.all_to_all_v(ins, C)
        a_v = oracle.all_to_all_v(ins, C, sd, sd)
        for j in range(R):
            assert np.array_equal(a_f[j], a_v[j])

    @pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
    @pytest.mark.parametrize("R", [2, 3, 8])
    def test_integer_inputs_sum_exactly(self, R, dtype):
        rng = np.random.default_rng(50 + R)
        n = 257
        ints = [rng.integers(-8, 9, size=R * n) for _ in range(R)]
        if dtype == "f32":
            x = [a.astype(np.float32) for a in ints]
        elif dtype == "bf16":
            x = [bf16_bits(torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16))
                 for a in ints]
        else:
            x = [a.astype(np.float16).view(np.uint16) for a in ints]
        exact = np.sum(np.stack(ints), axis=0)
        y = oracle.reduce_scatter(x, [n] * R, dtype=dtype)
        for k in range(R):
            assert np.array_equal(_to_f64(y[k], dtype), exact[k * n:(k + 1) * n].astype(np.float64))

    @pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
    def test_one_rank_is_a_copy(self, dtype):
        rng = np.random.default_rng(60)
        x = [_normal(rng, 33, dtype)]
        assert np.array_equal(oracle.reduce_scatter(x, [33], dtype=dtype)[0], x[0])
        assert np.array_equal(oracle.all_reduce(x, dtype=dtype)[0], x[0])
        assert np.array_equal(oracle.all_gather(x)[0], x[0])
        assert np.array_equal(oracle.all_to_all_v(x, [[33]])[0], x[0])

    @pytest.mark.parametrize("dtype,unit", [("f32", 2.0 ** -24), ("bf16", 2.0 ** -8),
                                            ("f16", 2.0 ** -11)])
    @pytest.mark.parametrize("order", ["fixed", "tree"])
    def test_within_error_bound_of_exact_sum(self, dtype, unit, order):
        """|y - S| <= u_out*|S| + 2*(R-1)*2^-24*sum|x_r| (+ the output type's
        smallest subnormal spacing), S the exact sum (float64 is exact here)."""
        rng = np.random.default_rng(70)
        R, n = 8, 4096
        x = [_normal(rng, R * n, dtype) for _ in range(R)]
        xs = np.stack([_to_f64(a, dtype) for a in x])
        S = xs.sum(axis=0)
        mag = np.abs(xs).sum(axis=0)
        y = np.concatenate([_to_f64(v, dtype) for v in
                            oracle.reduce_scatter(x, [n] * R, dtype=dtype, order=order)])
        tiny = {"f32": 2.0 ** -149, "bf16": 2.0 ** -133, "f16": 2.0 ** -24}[dtype]
        bound = unit * np.abs(S) + 2 * (R - 1) * 2.0 ** -24 * mag + tiny
        assert np.all(np.abs(y - S) <= bound)
        # and the bound is not vacuous: most results are not bit-identical to the
        # result of a different (reversed) order in binary32
        if dtype == "f32":
            rev = np.zeros_like(S, dtype=np.float32)
            acc = xs[R - 1].astype(np.float32)
            for r in range(R - 2, -1, -1):
                acc = acc + xs[r].astype(np.float32)
            rev = acc
            assert np.mean(rev != y.astype(np.float32)) > 0.05

    def test_fixed_order_matches_torch_elementwise_fold(self):
        """Library special case: torch's binary32 adds and its bf16 narrowing."""
        rng = np.random.default_rng(80)
        R, n = 8, 10000
        x = [_normal(rng, R * n, "bf16") for _ in range(R)]
        y = np.concatenate(oracle.reduce_scatter(x, [n] * R, dtype="bf16"))
        acc = bits_to_torch_bf16(x[0]).float()
        for r in range(1, R):
            acc = acc + bits_to_torch_bf16(x[r]).float()
        ref = bf16_bits(acc.to(torch.bfloat16))
        assert np.array_equal(y, ref)

    def test_fsum_agreement_f32(self):
        """For binary32 with two ranks the fold is a single correctly rounded add."""
        rng = np.random.default_rng(90)
        x = [rng.standard_normal(1000).astype(np.float32) for _ in range(2)]
        y = oracle.all_reduce(x, dtype="f32")[0]
        for i in range(0, 1000, 37):
            assert y[i] == np.float32(math.fsum([float(x[0][i]), float(x[1][i])]))
