"""CPU oracle for the Purlin collectives -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The CUDA library
and its Python binding never import it; the oracle imports nothing from them.

The arithmetic lives in ``purlin_oracle.c`` (plain C99, single-threaded scalar
loops); this module compiles it with gcc and marshals numpy arrays through
ctypes.  Semantics follow the page "Purlin: Separating Orchestration from the
Datapath of Collectives": Figure 4 (ReduceScatter, AllGather, AllToAll layouts on
three ranks), Figure 6 (AllReduce composed of ReduceScatter and AllGather) and
Table 2 ("(V)" = variable-length variant).

Data convention: float32 buffers are ``np.float32`` arrays; bfloat16 and
float16 buffers are ``np.uint16`` arrays holding the raw 16-bit words.  Counts and
displacements are in elements; ``None`` displacements mean packed layouts.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "purlin_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpurlin_oracle.so")

DTYPES = {"f32": 0, "bf16": 1, "f16": 2}
CFLAGS = ["-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libpurlin_oracle.so`` (gcc)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
             and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(
                 os.path.join(_HERE, "purlin_oracle.h")))
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", *CFLAGS, "-o", tmp, _SRC]
    subprocess.run(cmd, check=True, cwd=_HERE)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # PURLIN_ORACLE_LIB lets the mutation tests load a deliberately broken
        # build of this oracle in a child process.
        override = os.environ.get("PURLIN_ORACLE_LIB")
        lib = ctypes.CDLL(override if override else build())
        vp, u64p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint64)
        pp = ctypes.POINTER(ctypes.c_void_p)
        for name in ("oracle_bf16_to_f32_n", "oracle_f32_to_bf16_n",
                     "oracle_f16_to_f32_n", "oracle_f32_to_f16_n"):
            getattr(lib, name).argtypes = [vp, vp, ctypes.c_size_t]
            getattr(lib, name).restype = None
        lib.oracle_reduce_scatter.argtypes = [ctypes.c_int, pp, pp, u64p, u64p, ctypes.c_int]
        lib.oracle_reduce_scatter_tree.argtypes = [ctypes.c_int, pp, pp, u64p, u64p,
                                                   ctypes.c_int]
        lib.oracle_all_gather.argtypes = [ctypes.c_int, pp, pp, u64p, u64p, ctypes.c_size_t]
        lib.oracle_all_reduce.argtypes = [ctypes.c_int, pp, pp, ctypes.c_uint64, ctypes.c_int]
        lib.oracle_all_to_all_v.argtypes = [ctypes.c_int, pp, pp, u64p, u64p, u64p,
                                            ctypes.c_size_t]
        for name in ("oracle_reduce_scatter", "oracle_reduce_scatter_tree",
                     "oracle_all_gather", "oracle_all_reduce", "oracle_all_to_all_v"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


# --------------------------------------------------------------------------- helpers

def _ptrs(arrays):
    for a in arrays:
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("oracle buffers must be C-contiguous")
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


def _u64(values):
    if values is None:
        return None
    flat = np.ascontiguousarray(np.asarray(values, dtype=np.uint64).reshape(-1))
    return flat, flat.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64))


def _np_type(dtype: str):
    return np.float32 if dtype == "f32" else np.uint16


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: arguments rejected")


def _packed(counts):
    starts, s = [], 0
    for c in counts:
        starts.append(s)
        s += int(c)
    return starts


# --------------------------------------------------------------------------- codecs

def _codec(name, src, out_dtype):
    lib = _load()
    src = np.ascontiguousarray(src)
    out = np.empty(src.shape, dtype=out_dtype)
    getattr(lib, name)(src.ctypes.data, out.ctypes.data, src.size)
    return out


def bf16_to_f32(h):
    return _codec("oracle_bf16_to_f32_n", np.asarray(h, dtype=np.uint16), np.float32)


def f32_to_bf16(f):
    return _codec("oracle_f32_to_bf16_n", np.asarray(f, dtype=np.float32), np.uint16)


def f16_to_f32(h):
    return _codec("oracle_f16_to_f32_n", np.asarray(h, dtype=np.uint16), np.float32)


def f32_to_f16(f):
    return _codec("oracle_f32_to_f16_n", np.asarray(f, dtype=np.float32), np.uint16)


# ----------------------------------------------------------------------- collectives

def reduce_scatter(x, recv_counts, in_displs=None, dtype="bf16", order="fixed"):
    """ReduceScatter(V) (Figure 4, top): returns [y_0, ..., y_{R-1}] with
    y_k[i] = sum_r x_r[d_k + i] folded in rank order (``order="tree"``: pairwise)."""
    lib = _load()
    R = len(x)
    counts, counts_p = _u64(recv_counts)
    displs = _u64(in_displs)
    y = [np.empty(int(c), dtype=_np_type(dtype)) for c in counts]
    fn = lib.oracle_reduce_scatter if order == "fixed" else lib.oracle_reduce_scatter_tree
    _check(fn(R, _ptrs(x), _ptrs(y), counts_p, displs[1] if displs else None,
              DTYPES[dtype]), "reduce_scatter")
    return y


def all_gather(inputs, counts=None, out_displs=None, out_count=None):
    """AllGather(V) (Figure 4, top): every output holds every input, in rank order."""
    lib = _load()
    R = len(inputs)
    counts = [a.size for a in inputs] if counts is None else list(counts)
    starts = list(out_displs) if out_displs is not None else _packed(counts)
    if out_count is None:
        out_count = max([int(s) + int(c) for s, c in zip(starts, counts)] + [0])
    out = [np.zeros(int(out_count), dtype=inputs[0].dtype) for _ in range(R)]
    cnt, cnt_p = _u64(counts)
    displs = _u64(out_displs)
    _check(lib.oracle_all_gather(R, _ptrs(inputs), _ptrs(out), cnt_p,
                                 displs[1] if displs else None, inputs[0].itemsize),
           "all_gather")
    return out


def all_reduce(x, dtype="bf16"):
    """AllReduce (Figure 6): every output is the rank-order sum of all inputs."""
    lib = _load()
    R = len(x)
    n = x[0].size
    out = [np.empty(n, dtype=_np_type(dtype)) for _ in range(R)]
    _check(lib.oracle_all_reduce(R, _ptrs(x), _ptrs(out), n, DTYPES[dtype]), "all_reduce")
    return out


def all_to_all_v(inputs, send_counts, send_displs=None, recv_displs=None, recv_lens=None):
    """AllToAll(V) (Figure 4, bottom): rank j gets partition j of every source in
    source order.  ``send_counts[s][j]`` elements go from source s to rank j."""
    lib = _load()
    R = len(inputs)
    C = np.asarray(send_counts, dtype=np.uint64).reshape(R, R)
    if recv_lens is None:
        recv_lens = []
        for j in range(R):
            if recv_displs is None:
                recv_lens.append(int(C[:, j].sum()))
            else:
                rd = np.asarray(recv_displs, dtype=np.uint64).reshape(R, R)
                recv_lens.append(max([int(rd[j, s]) + int(C[s, j]) for s in range(R)] + [0]))
    out = [np.zeros(int(n), dtype=inputs[0].dtype) for n in recv_lens]
    cnt, cnt_p = _u64(C)
    sd = _u64(send_displs)
    rd_ = _u64(recv_displs)
    _check(lib.oracle_all_to_all_v(R, _ptrs(inputs), _ptrs(out), cnt_p,
                                   sd[1] if sd else None, rd_[1] if rd_ else None,
                                   inputs[0].itemsize), "all_to_all_v")
    return out
