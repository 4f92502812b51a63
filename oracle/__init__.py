"""CPU oracle for the sharded relay collectives -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and
its ``--impl reference`` arm) may import this package.  The CUDA library never calls
it, and it shares no code with ``pack_virtual_rank_gb300``.

``build()`` compiles ``oracle.c`` with gcc into ``liboracle.so`` next to it; ``lib()``
loads it.  The wrappers below only marshal numpy arrays: every step of the arithmetic
is in ``oracle.c``.  bfloat16 arrays travel as their raw uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")

F32, BF16, I32 = 0, 1, 2
AR, RS, AG, A2A = 0, 1, 2, 3
KIND_RELAY, KIND_ZERO_CHUNK, KIND_DIRECT, KIND_LEGACY = 0, 1, 2, 3
FORCE_AUTO, FORCE_RELAY, FORCE_DIRECT, FORCE_LEGACY = 0, 1, 2, 3
ESIZE = {F32: 4, BF16: 2, I32: 4}
NP_DTYPE = {F32: np.float32, BF16: np.uint16, I32: np.int32}

GEOM_FIELDS = ("coll", "A", "R", "H", "esize", "count", "kind", "groups", "chunk",
               "dirA", "dirA_off", "dirB", "pD", "d1", "d2", "owner_slice",
               "owner_last")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (plain C, no fused multiply-add) into liboracle.so."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-Wextra",
                               "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        i64, i32, vp, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
        L.orc_bf16_rne.restype = ctypes.c_uint16
        L.orc_bf16_rne.argtypes = [f32]
        L.orc_bf16_to_f32.restype = f32
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_bf16_rne_array.argtypes = [vp, vp, i64]
        L.orc_allreduce.argtypes = [i32, i32, vp, i64, i64, f32, vp, vp, vp]
        L.orc_reduce_scatter.argtypes = [i32, i32, vp, i64, i32, i64, i64, f32, i64,
                                         vp, vp, vp]
        L.orc_reduce_scatter_wide.argtypes = [i32, i32, vp, i64, i32, i64, i64, f32, i64,
                                              vp, vp, vp]
        L.orc_all_gather.argtypes = [i32, i32, vp, i64, vp]
        L.orc_all_to_all.argtypes = [i32, i32, vp, i64, i32, vp]
        L.orc_align_down.restype = i64
        L.orc_align_down.argtypes = [i64]
        L.orc_plan.restype = i32
        L.orc_plan.argtypes = [i32, i32, i32, i64, i32, i32, i32, vp]
        L.orc_link_elems.restype = i32
        L.orc_link_elems.argtypes = [vp, vp, i64]
        L.orc_cost_elems.restype = ctypes.c_uint64
        L.orc_cost_elems.argtypes = [vp]
        L.orc_passthrough_helper_size.restype = i64
        L.orc_passthrough_helper_size.argtypes = [i64, i32, i32]
        L.orc_relay_helper_contract.restype = i64
        L.orc_relay_helper_contract.argtypes = [i32, i32, i32, i64]
        _lib = L
    return _lib


def _ptrs(xs):
    arr = (ctypes.c_void_p * len(xs))(*[x.ctypes.data for x in xs])
    return arr


def _check(xs, dtype):
    for x in xs:
        if x.dtype != NP_DTYPE[dtype] or not x.flags.c_contiguous:
            raise TypeError(f"oracle expects contiguous {NP_DTYPE[dtype]} arrays")


# ---- bfloat16 ---------------------------------------------------------------

def bf16_rne(values: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().orc_bf16_rne_array(v.ctypes.data, out.ctypes.data, v.size)
    return out


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widening is exact: the bf16 bits become the upper half of a binary32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ---- collectives -------------------------------------------------------------

def allreduce(dtype, xs, scale=1.0, i0=0, i1=None):
    _check(xs, dtype)
    i1 = xs[0].size if i1 is None else i1
    n = i1 - i0
    r64 = np.empty(n, np.float64)
    r32 = np.empty(n, np.float32)
    rq = np.empty(n, NP_DTYPE[dtype])
    lib().orc_allreduce(dtype, len(xs), _ptrs(xs), i0, i1, scale, r64.ctypes.data,
                        r32.ctypes.data, rq.ctypes.data)
    return r64, r32, rq


def reduce_scatter(dtype, xs, m, owner, scale=1.0, helper_span=0, i0=0, i1=None):
    _check(xs, dtype)
    i1 = m if i1 is None else i1
    n = i1 - i0
    r64 = np.empty(n, np.float64)
    r32 = np.empty(n, np.float32)
    rq = np.empty(n, NP_DTYPE[dtype])
    lib().orc_reduce_scatter(dtype, len(xs), _ptrs(xs), m, owner, i0, i1, scale,
                             helper_span, r64.ctypes.data, r32.ctypes.data,
                             rq.ctypes.data)
    return r64, r32, rq


def reduce_scatter_wide(dtype, xs, m, owner, scale=1.0, helper_span=0, i0=0, i1=None):
    """Flat reduce-at-helper with the helper partial carried in fp32 (not rounded)."""
    _check(xs, dtype)
    i1 = m if i1 is None else i1
    n = i1 - i0
    r64 = np.empty(n, np.float64)
    r32 = np.empty(n, np.float32)
    rq = np.empty(n, NP_DTYPE[dtype])
    lib().orc_reduce_scatter_wide(dtype, len(xs), _ptrs(xs), m, owner, i0, i1, scale,
                                  helper_span, r64.ctypes.data, r32.ctypes.data, rq.ctypes.data)
    return r64, r32, rq


def all_gather(xs, S):
    out = np.empty(len(xs) * S, xs[0].dtype)
    lib().orc_all_gather(xs[0].itemsize, len(xs), _ptrs(xs), S, out.ctypes.data)
    return out


def all_to_all(xs, seg, dst):
    out = np.empty(len(xs) * seg, xs[0].dtype)
    lib().orc_all_to_all(xs[0].itemsize, len(xs), _ptrs(xs), seg, dst, out.ctypes.data)
    return out


# ---- planner restatement -------------------------------------------------------

def plan(coll, A, R, count, esize, permille=500, force=FORCE_AUTO):
    g = np.zeros(len(GEOM_FIELDS), np.int64)
    rc = lib().orc_plan(coll, A, R, count, esize, permille, force, g.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle plan rejected coll={coll} A={A} R={R} count={count}")
    return dict(zip(GEOM_FIELDS, (int(v) for v in g))), g


def link_elems(gvec) -> np.ndarray:
    R = int(gvec[2])
    G = int(gvec[7])
    t = np.zeros(max(G, 1) * R * R, np.uint64)
    rc = lib().orc_link_elems(gvec.ctypes.data, t.ctypes.data, t.size)
    if rc < 0:
        raise ValueError("link table does not fit")
    return t[: G * R * R].reshape(G, R, R)


def cost_elems(gvec) -> int:
    return int(lib().orc_cost_elems(gvec.ctypes.data))


def passthrough_helper_size(count_g, A, num_chunks) -> int:
    return int(lib().orc_passthrough_helper_size(count_g, A, num_chunks))


def relay_helper_contract(coll, A, R, count) -> int:
    return int(lib().orc_relay_helper_contract(coll, A, R, count))


def align_down(x) -> int:
    return int(lib().orc_align_down(x))
