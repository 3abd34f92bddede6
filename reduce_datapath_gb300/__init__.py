"""Python binding of the Purlin collective datapath C ABI (``include/purlin.h``).

Argument marshalling only: every entry point forwards to ``libpurlin.so``, whose
CUDA kernels do all the work.  There is no Python or CPU fallback: if the
library is missing, the first call raises ``PurlinLibraryError``.

The functions keep the C names.  Buffers are passed as sequences of R device
tensors (anything with ``data_ptr()``) or raw integer device addresses; counts
and displacements as sequences of ints (R, or R*R for AllToAllV, row-major);
``dtype`` as ``"f32" | "bf16" | "f16" | "u8"`` or a torch dtype; ``stream`` as a
``torch.cuda.Stream``, a raw ``cudaStream_t`` integer, or None for torch's current
stream.  A non-OK status raises ``PurlinError`` carrying the status code.

Page: "Purlin: Separating Orchestration from the Datapath of Collectives"
(abstract; Figure 4 layouts; Figure 6 composed AllReduce; Table 2 "(V)").
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
# PURLIN_LIBRARY=checked selects the checked build (every kernel access tested
# against the call's buffers; for tests) in place of the product build.
LIB_PATH = os.path.join(_HERE, "lib", "libpurlin_checked.so"
                        if os.environ.get("PURLIN_LIBRARY") == "checked" else "libpurlin.so")

# purlin_status_t
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_OOM, ERR_BOUNDS = range(7)
# purlin_dtype_t
F32, BF16, F16, U8 = range(4)
DTYPES = {"f32": F32, "bf16": BF16, "f16": F16, "u8": U8}
ELEM_BYTES = {F32: 4, BF16: 2, F16: 2, U8: 1}
# purlin_op_t
OP_COPY, OP_SUM = 0, 1
# purlin_variant_t
VARIANT_AUTO, VARIANT_ZS, VARIANT_STAGED, VARIANT_STAGED_Y = 0, 1, 2, 3
# purlin_order_t
ORDER_FIXED, ORDER_TREE = 0, 1
# purlin_atom_t
ATOM_AUTO, ATOM_VECTOR, ATOM_BULK, ATOM_COPY_ENGINE = 0, 1, 2, 3
# purlin_direction_t
DIRECTION_AUTO, DIRECTION_PUSH, DIRECTION_PULL = 0, 1, 2
# purlin_set_small_tiles: library default / never
SMALL_TILES_DEFAULT, SMALL_TILES_NEVER = -1, 0
# purlin_collective_t
COLL_REDUCE_SCATTER, COLL_ALL_GATHER, COLL_ALL_REDUCE, COLL_ALL_TO_ALL_V = range(4)
MAX_RANKS = 8

# Every symbol the headers under include/ declare.
EXPORTED = (
    "purlin_create", "purlin_destroy", "purlin_reduce_scatter", "purlin_all_gather",
    "purlin_all_reduce", "purlin_all_to_all", "purlin_all_to_all_v", "purlin_set_policy",
    "purlin_set_reduce_order", "purlin_set_atom", "purlin_set_direction", "purlin_set_small_tiles",
    "purlin_set_timeout", "purlin_query_status", "purlin_plan_begin", "purlin_plan_end",
    "purlin_plan_launch", "purlin_plan_destroy",
    "purlin_last_launch", "purlin_status_string", "purlin_version", "purlin_plan_segments",
    "purlin_debug_inject", "purlin_debug_checked", "purlin_debug_violation",
    "purlin_all_reduce_noalloc",
)


class PurlinLibraryError(RuntimeError):
    """libpurlin.so is missing or does not load."""


class PurlinError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_text(status)} (status {status})")


class LaunchInfo(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("kernels", ctypes.c_int), ("grid", ctypes.c_int),
                ("block", ctypes.c_int), ("sms", ctypes.c_int), ("depth", ctypes.c_int),
                ("chunk_bytes", ctypes.c_size_t), ("bytes_moved", ctypes.c_size_t)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class Segment(ctypes.Structure):
    _fields_ = [("src_off", ctypes.c_uint64), ("dst_off", ctypes.c_uint64),
                ("bytes", ctypes.c_uint64), ("src_rank", ctypes.c_int32),
                ("dst_rank", ctypes.c_int32), ("unit", ctypes.c_int32),
                ("tile0", ctypes.c_uint32), ("shift", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False, checked: bool = False) -> str:
    """Compile libpurlin.so in-tree (nvcc, sm_103a); checked=True: the checked
    build libpurlin_checked.so instead."""
    from . import _build
    return _build.build(force=force, checked=checked)


def lib():
    """The loaded libpurlin.so (raises PurlinLibraryError if it is not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise PurlinLibraryError(
                f"{LIB_PATH} is not built; run reduce_datapath_gb300.build() first")
        try:
            L = ctypes.CDLL(LIB_PATH)
        except OSError as e:
            raise PurlinLibraryError(f"cannot load {LIB_PATH}: {e}") from e
        vp, sz, i32, u64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_uint64
        pp = ctypes.POINTER(ctypes.c_void_p)
        szp = ctypes.POINTER(ctypes.c_size_t)
        u64p = ctypes.POINTER(ctypes.c_uint64)
        sigs = {
            "purlin_create": [ctypes.POINTER(vp), i32, sz, i32],
            "purlin_destroy": [vp],
            "purlin_reduce_scatter": [vp, pp, pp, szp, szp, i32, i32, vp],
            "purlin_all_gather": [vp, pp, pp, szp, szp, i32, vp],
            "purlin_all_reduce": [vp, pp, pp, sz, i32, i32, vp],
            "purlin_all_to_all": [vp, pp, pp, sz, i32, vp],
            "purlin_all_to_all_v": [vp, pp, pp, szp, szp, szp, i32, vp],
            "purlin_set_policy": [vp, sz, i32, i32, i32],
            "purlin_set_reduce_order": [vp, i32],
            "purlin_set_atom": [vp, i32],
            "purlin_set_direction": [vp, i32],
            "purlin_set_small_tiles": [vp, i32],
            "purlin_plan_begin": [vp],
            "purlin_plan_end": [vp, ctypes.POINTER(vp)],
            "purlin_plan_launch": [vp, vp],
            "purlin_plan_destroy": [vp],
            "purlin_set_timeout": [vp, u64],
            "purlin_query_status": [vp],
            "purlin_last_launch": [vp, ctypes.POINTER(LaunchInfo)],
            "purlin_status_string": [i32],
            "purlin_version": [],
            "purlin_plan_segments": [i32, i32, u64p, u64p, szp, szp, szp, sz, i32, i32,
                                     ctypes.POINTER(Segment), i32, ctypes.POINTER(i32),
                                     ctypes.POINTER(ctypes.c_uint32)],
            "purlin_debug_inject": [vp, i32],
            "purlin_debug_checked": [],
            "purlin_debug_violation": [vp, u64p],
            "purlin_all_reduce_noalloc": [pp, pp, i32, sz, i32, sz, i32, vp, vp],
        }
        for name, args in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = i32
        L.purlin_status_string.restype = ctypes.c_char_p
        _lib = L
        return L


def status_text(status: int) -> str:
    try:
        return lib().purlin_status_string(int(status)).decode()
    except PurlinLibraryError:
        return "status %d" % status


# ------------------------------------------------------------------ marshalling

def _check(status: int, where: str):
    if status != OK:
        raise PurlinError(status, where)


def _ptr(x) -> int:
    if x is None:
        return 0
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    return int(x)


def _ptrs(bufs):
    vals = [_ptr(b) for b in bufs]
    return (ctypes.c_void_p * len(vals))(*vals)


def _sizes(vals):
    if vals is None:
        return None
    if hasattr(vals, "__array_interface__"):
        # a numpy array: a ctypes view of a contiguous size_t copy (the view
        # keeps that array alive for the call)
        import numpy as np
        arr = np.ascontiguousarray(np.asarray(vals).reshape(-1), dtype=_SIZE_T_NP)
        if not arr.flags.writeable:
            arr = arr.copy()
        return (ctypes.c_size_t * arr.size).from_buffer(arr)
    flat = [int(v) for v in (vals.reshape(-1).tolist() if hasattr(vals, "reshape") else vals)]
    return (ctypes.c_size_t * len(flat))(*flat)


_SIZE_T_NP = "u%d" % ctypes.sizeof(ctypes.c_size_t)


def _dtype(dt) -> int:
    if isinstance(dt, int):
        return dt
    if isinstance(dt, str):
        return DTYPES[dt]
    import torch
    table = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16, torch.uint8: U8,
             torch.int8: U8}
    fp8 = [getattr(torch, n) for n in ("float8_e4m3fn", "float8_e5m2") if hasattr(torch, n)]
    for t in fp8:
        table[t] = U8
    return table[dt]


def _op(op) -> int:
    if isinstance(op, int):
        return op
    return {"sum": OP_SUM, "copy": OP_COPY}[op]


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if hasattr(stream, "cuda_stream"):
        return int(stream.cuda_stream)
    return int(stream)


# ------------------------------------------------------------------- the ABI

def purlin_version() -> int:
    return lib().purlin_version()


def purlin_create(R: int, staging_bytes: int = 0, device: int | None = None) -> int:
    if device is None:
        import torch
        device = torch.cuda.current_device()
    h = ctypes.c_void_p()
    _check(lib().purlin_create(ctypes.byref(h), int(R), int(staging_bytes), int(device)),
           "purlin_create")
    return h.value


def purlin_destroy(h) -> None:
    _check(lib().purlin_destroy(h), "purlin_destroy")


# Marshalling of each collective's arguments into the C call's ctypes values.
def _m_reduce_scatter(h, ins, outs, recv_counts, in_displs=None, dtype="bf16", op="sum",
                      stream=None):
    return (h, _ptrs(ins), _ptrs(outs), _sizes(recv_counts), _sizes(in_displs), _dtype(dtype),
            _op(op), _stream(stream))


def _m_all_gather(h, ins, outs, counts, out_displs=None, dtype="bf16", stream=None):
    return (h, _ptrs(ins), _ptrs(outs), _sizes(counts), _sizes(out_displs), _dtype(dtype),
            _stream(stream))


def _m_all_reduce(h, ins, outs, count, dtype="bf16", op="sum", stream=None):
    return (h, _ptrs(ins), _ptrs(outs), int(count), _dtype(dtype), _op(op), _stream(stream))


def _m_all_to_all(h, ins, outs, count_per_pair, dtype="bf16", stream=None):
    return (h, _ptrs(ins), _ptrs(outs), int(count_per_pair), _dtype(dtype), _stream(stream))


def _m_all_to_all_v(h, ins, outs, send_counts, send_displs=None, recv_displs=None,
                    dtype="bf16", stream=None):
    return (h, _ptrs(ins), _ptrs(outs), _sizes(send_counts), _sizes(send_displs),
            _sizes(recv_displs), _dtype(dtype), _stream(stream))


def _call(name, cargs):
    _check(getattr(lib(), name)(*cargs), name)


def purlin_reduce_scatter(h, ins, outs, recv_counts, in_displs=None, dtype="bf16", op="sum",
                          stream=None) -> None:
    _call("purlin_reduce_scatter",
          _m_reduce_scatter(h, ins, outs, recv_counts, in_displs, dtype, op, stream))


def purlin_all_gather(h, ins, outs, counts, out_displs=None, dtype="bf16", stream=None) -> None:
    _call("purlin_all_gather", _m_all_gather(h, ins, outs, counts, out_displs, dtype, stream))


def purlin_all_reduce(h, ins, outs, count, dtype="bf16", op="sum", stream=None) -> None:
    _call("purlin_all_reduce", _m_all_reduce(h, ins, outs, count, dtype, op, stream))


def purlin_all_to_all(h, ins, outs, count_per_pair, dtype="bf16", stream=None) -> None:
    _call("purlin_all_to_all", _m_all_to_all(h, ins, outs, count_per_pair, dtype, stream))


def purlin_all_to_all_v(h, ins, outs, send_counts, send_displs=None, recv_displs=None,
                        dtype="bf16", stream=None) -> None:
    _call("purlin_all_to_all_v",
          _m_all_to_all_v(h, ins, outs, send_counts, send_displs, recv_displs, dtype, stream))


_MARSHAL = {
    "purlin_reduce_scatter": _m_reduce_scatter,
    "purlin_all_gather": _m_all_gather,
    "purlin_all_reduce": _m_all_reduce,
    "purlin_all_to_all": _m_all_to_all,
    "purlin_all_to_all_v": _m_all_to_all_v,
}


def prepare(fn, *args, **kwargs):
    """Marshal the arguments of one collective call once and return a callable
    that repeats exactly that C call (same handle, buffers, counts, dtype and
    stream).  For loops that re-issue a collective on the same buffers: each
    repeat costs only the C call.  The buffers must outlive the callable."""
    name = fn if isinstance(fn, str) else fn.__name__
    cargs = _MARSHAL[name](*args, **kwargs)
    cfn = getattr(lib(), name)

    def call() -> None:
        st = cfn(*cargs)
        if st != OK:
            raise PurlinError(st, name)

    call.c_args = cargs   # keeps the ctypes arrays alive with the callable
    return call


def purlin_plan_begin(h) -> None:
    _check(lib().purlin_plan_begin(h), "purlin_plan_begin")


def purlin_plan_end(h):
    plan = ctypes.c_void_p()
    _check(lib().purlin_plan_end(h, ctypes.byref(plan)), "purlin_plan_end")
    return plan.value


def purlin_plan_launch(plan, stream=None) -> None:
    _check(lib().purlin_plan_launch(plan, _stream(stream)), "purlin_plan_launch")


def purlin_plan_destroy(plan) -> None:
    _check(lib().purlin_plan_destroy(plan), "purlin_plan_destroy")


class Plan:
    """One collective call planned once (purlin_plan_begin / _end): calling the
    object launches that call again on the stream it was planned with (or on
    `stream`).  The buffers must outlive the plan; the handle's policy is the
    one in force when the plan was made."""

    def __init__(self, fn, h, *args, **kwargs):
        name = fn if isinstance(fn, str) else fn.__name__
        self._stream = _stream(kwargs.get("stream"))
        self._lib = lib()
        purlin_plan_begin(h)
        try:
            _call(name, _MARSHAL[name](h, *args, **kwargs))
        finally:
            plan = ctypes.c_void_p()
            st = self._lib.purlin_plan_end(h, ctypes.byref(plan))
        _check(st, "purlin_plan_end")
        self.handle = plan.value
        self._launch = self._lib.purlin_plan_launch

    def __call__(self, stream=None) -> None:
        st = self._launch(self.handle, self._stream if stream is None else _stream(stream))
        if st != OK:
            raise PurlinError(st, "purlin_plan_launch")

    def destroy(self) -> None:
        if self.handle:
            self._lib.purlin_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def plan(fn, h, *args, **kwargs) -> Plan:
    """Plan one collective call (same arguments as the call itself) for repeated
    launches: each launch is one C call of two arguments."""
    return Plan(fn, h, *args, **kwargs)


def purlin_set_policy(h, chunk_bytes=0, depth=0, ctas=0, variant=VARIANT_AUTO) -> None:
    _check(lib().purlin_set_policy(h, int(chunk_bytes), int(depth), int(ctas), int(variant)),
           "purlin_set_policy")


def purlin_set_reduce_order(h, order) -> None:
    _check(lib().purlin_set_reduce_order(h, int(order)), "purlin_set_reduce_order")


def purlin_set_atom(h, atom) -> None:
    _check(lib().purlin_set_atom(h, int(atom)), "purlin_set_atom")


def purlin_set_direction(h, direction) -> None:
    _check(lib().purlin_set_direction(h, int(direction)), "purlin_set_direction")


def purlin_set_small_tiles(h, tiles) -> None:
    _check(lib().purlin_set_small_tiles(h, int(tiles)), "purlin_set_small_tiles")


def purlin_set_timeout(h, timeout_ns) -> None:
    _check(lib().purlin_set_timeout(h, int(timeout_ns)), "purlin_set_timeout")


def purlin_query_status(h) -> int:
    """Device status word (read and cleared); returns the code, does not raise."""
    return int(lib().purlin_query_status(h))


def purlin_last_launch(h) -> dict:
    info = LaunchInfo()
    _check(lib().purlin_last_launch(h, ctypes.byref(info)), "purlin_last_launch")
    return info.as_dict()


def purlin_status_string(status) -> str:
    return lib().purlin_status_string(int(status)).decode()


def purlin_debug_inject(h, what: int) -> None:
    _check(lib().purlin_debug_inject(h, int(what)), "purlin_debug_inject")


def purlin_debug_checked() -> bool:
    return bool(lib().purlin_debug_checked())


def purlin_debug_violation(h) -> int:
    v = ctypes.c_uint64(0)
    _check(lib().purlin_debug_violation(h, ctypes.byref(v)), "purlin_debug_violation")
    return int(v.value)


def purlin_all_reduce_noalloc(ins, outs, count, dtype="bf16", chunk_bytes=0, depth=0,
                              device_status=None, stream=None) -> None:
    """AllReduce that allocates nothing (see purlin.h): for callers that may not
    call cudaMalloc.  Scratch is a fixed 8 MiB static device array."""
    _check(lib().purlin_all_reduce_noalloc(_ptrs(ins), _ptrs(outs), len(ins), int(count),
                                           _dtype(dtype), int(chunk_bytes), int(depth),
                                           _ptr(device_status), _stream(stream)),
           "purlin_all_reduce_noalloc")


def purlin_plan_segments(coll, R, in_addr, out_addr, counts=None, displs_a=None, displs_b=None,
                         count=0, dtype="bf16", max_unit=32, max_segs=256):
    """Host-only plan of one collective (no GPU needed); returns (segments, ntiles)."""
    segs = (Segment * max_segs)()
    n = ctypes.c_int(0)
    nt = ctypes.c_uint32(0)
    ia = (ctypes.c_uint64 * len(in_addr))(*[int(a) for a in in_addr])
    oa = (ctypes.c_uint64 * len(out_addr))(*[int(a) for a in out_addr])
    _check(lib().purlin_plan_segments(int(coll), int(R), ia, oa, _sizes(counts),
                                      _sizes(displs_a), _sizes(displs_b), int(count),
                                      _dtype(dtype), int(max_unit), segs, max_segs,
                                      ctypes.byref(n), ctypes.byref(nt)),
           "purlin_plan_segments")
    out = [{f: getattr(segs[i], f) for f, _ in Segment._fields_} for i in range(n.value)]
    return out, nt.value
