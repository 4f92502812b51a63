"""ctypes binding of ``librelay.so`` (the C ABI in ``include/relay.h``).

Argument marshalling only: every step of a collective runs in the library's CUDA
kernels. PyTorch is used for device memory and streams. There is no fallback: if the
library is not built the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librelay.so")

# enums (relay.h)
OK, ERR_INVALID_ARGUMENT, ERR_UNSUPPORTED, ERR_CUDA = 0, 1, 2, 3
F32, BF16, I32 = 0, 1, 2
ALLREDUCE, REDUCE_SCATTER, ALL_GATHER, ALL_TO_ALL = 0, 1, 2, 3
KIND_RELAY, KIND_ZERO_CHUNK, KIND_DIRECT, KIND_LEGACY = 0, 1, 2, 3
SCHEDULE_AUTO, SCHEDULE_RELAY, SCHEDULE_DIRECT, SCHEDULE_LEGACY = 0, 1, 2, 3
FLAG_CHECK_HAZARDS = 1
FLAG_DRY_RUN = 2
FLAG_SEPARATE_PASSES = 4
FLAG_FUSED_PASSES = 8
FLAG_PAYLOAD_PARTIAL = 16
FLAG_CHAINED = 32
FLAG_KEEP_SCRATCH = 64
ESIZE = {F32: 4, BF16: 2, I32: 4}
PASS_NAMES = ("group1", "group2", "group3", "active_reduce", "pack", "helper_forward", "unpack")


class RelayError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"relay status {status}: {message}")
        self.status = status


class RelayOpts(ctypes.Structure):
    _fields_ = [("offload_permille", ctypes.c_int32), ("schedule", ctypes.c_int32),
                ("relay_threshold_bytes", ctypes.c_int64), ("pass_events", ctypes.c_void_p),
                ("n_pass_events", ctypes.c_int32), ("flags", ctypes.c_int32)]


class RelayPlan(ctypes.Structure):
    _fields_ = ([(f, ctypes.c_int32) for f in ("coll", "dtype", "A", "R", "H", "esize", "kind",
                                               "num_groups", "offload_permille", "wide_partial")]
                + [(f, ctypes.c_int64) for f in ("count", "chunk", "relay_total", "dirA_offset",
                                                 "dirA_size", "dirB_size", "direct_total",
                                                 "direct_g1", "direct_g2", "owner_slice",
                                                 "owner_slice_last", "helper_elems",
                                                 "active_scratch_elems", "input_elems",
                                                 "output_elems")])

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class RelayPassInfo(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("num_segments", ctypes.c_int32),
                ("bytes_read", ctypes.c_int64), ("bytes_written", ctypes.c_int64)]


_lib = None


def lib():
    """Load librelay.so (build it first with ``pack_virtual_rank_gb300.build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built: call pack_virtual_rank_gb300.build.build() "
                           "(needs nvcc); there is no fallback implementation")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz, f32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                             ctypes.c_float)
    P = ctypes.POINTER
    L.relay_opts_init.argtypes = [P(RelayOpts)]
    L.relay_opts_init.restype = None
    L.relay_abi_version.restype = i32
    L.relay_last_error.restype = ctypes.c_char_p
    L.relay_last_launch.restype = ctypes.c_char_p
    L.relay_plan.argtypes = [i32, sz, i32, i32, i32, P(RelayOpts), P(RelayPlan)]
    L.relay_plan.restype = i32
    L.relay_plan_link_bytes.argtypes = [P(RelayPlan), P(ctypes.c_uint64), sz]
    L.relay_plan_link_bytes.restype = i32
    L.relay_plan_cost_bytes.argtypes = [P(RelayPlan)]
    L.relay_plan_cost_bytes.restype = ctypes.c_uint64
    L.relay_plan_passes.argtypes = [P(RelayPlan), i32, P(RelayPassInfo), i32]
    L.relay_plan_passes.restype = i32
    L.relay_pass_name.argtypes = [i32]
    L.relay_pass_name.restype = ctypes.c_char_p
    L.relay_passthrough_helper_size.argtypes = [i64, i32, i32]
    L.relay_passthrough_helper_size.restype = i64
    arr = P(vp)
    for name in ("relay_allreduce", "relay_reduce_scatter"):
        fn = getattr(L, name)
        fn.argtypes = [arr, arr, arr, sz, i32, i32, i32, f32, P(RelayOpts), vp]
        fn.restype = i32
    for name in ("relay_all_gather", "relay_all_to_all"):
        fn = getattr(L, name)
        fn.argtypes = [arr, arr, arr, sz, i32, i32, i32, P(RelayOpts), vp]
        fn.restype = i32
    L.relay_multi_group.argtypes = [i32, i32, P(sz), arr, arr, arr, i32, i32, f32, P(RelayOpts), vp]
    L.relay_multi_group.restype = i32
    L.relay_multi_group_link_bytes.argtypes = [i32, i32, P(sz), i32, i32, P(RelayOpts),
                                               P(ctypes.c_uint64), sz, P(ctypes.c_int)]
    L.relay_multi_group_link_bytes.restype = i32
    L.relay_helper_size.argtypes = [P(RelayPlan)]
    L.relay_helper_size.restype = i64
    L.relay_active_scratch_size.argtypes = [P(RelayPlan)]
    L.relay_active_scratch_size.restype = i64
    L.relay_helper_contract_size.argtypes = [i32, i64, i32, i32]
    L.relay_helper_contract_size.restype = i64
    L.relay_allreduce_noalloc.argtypes = [arr, arr, sz, i32, i32, i32, f32, P(RelayOpts), vp]
    L.relay_allreduce_noalloc.restype = i32
    L.relay_pack_flat.argtypes = [arr, P(sz), i32, vp, i32, vp]
    L.relay_pack_flat.restype = i32
    L.relay_unpack_flat.argtypes = [vp, arr, P(sz), i32, i32, vp]
    L.relay_unpack_flat.restype = i32
    L.relay_copy.argtypes = [vp, vp, sz, i32, i32, vp]
    L.relay_copy.restype = i32
    L.relay_device_status.argtypes = []
    L.relay_device_status.restype = i32
    L.relay_test_staged_wait.argtypes = [vp, vp, sz, i32, i32, vp]
    L.relay_test_staged_wait.restype = i32
    if L.relay_abi_version() != 1:
        raise RuntimeError("librelay.so ABI version mismatch")
    _lib = L
    return L


def _check(status: int):
    if status != OK:
        raise RelayError(status, lib().relay_last_error().decode(errors="replace"))


def device_status() -> None:
    """Raise if a bounded wait in a relay kernel gave up since the last check (reads and
    clears the device's fault word; synchronous)."""
    _check(lib().relay_device_status())


def last_launch() -> str:
    """How this thread's last collective call was launched: "chained", "cooperative" or
    "passes" ("dry run" for a dry run that would not run chained)."""
    return lib().relay_last_launch().decode()


def dtype_code(dtype) -> int:
    """Accept a relay dtype code, "f32"/"bf16"/"i32", or a torch dtype."""
    if isinstance(dtype, int):
        return dtype
    if isinstance(dtype, str):
        return {"f32": F32, "bf16": BF16, "i32": I32}[dtype]
    import torch
    return {torch.float32: F32, torch.bfloat16: BF16, torch.int32: I32}[dtype]


def make_opts(offload_permille: int = -1, schedule: int = SCHEDULE_AUTO,
              relay_threshold_bytes: int = -1, flags: int = 0, pass_events=None) -> RelayOpts:
    o = RelayOpts()
    lib().relay_opts_init(ctypes.byref(o))
    o.offload_permille = offload_permille
    o.schedule = schedule
    o.relay_threshold_bytes = relay_threshold_bytes
    o.flags = flags
    if pass_events is not None:
        for e in pass_events:
            # torch creates the CUDA event lazily, on its first record
            if hasattr(e, "cuda_event") and int(e.cuda_event) == 0:
                e.record()
        handles = (ctypes.c_void_p * len(pass_events))(*[int(e.cuda_event) if hasattr(e, "cuda_event")
                                                          else int(e) for e in pass_events])
        o._events_keepalive = handles
        o.pass_events = ctypes.cast(handles, ctypes.c_void_p)
        o.n_pass_events = len(pass_events)
    return o


# ------------------------------------------------------------------------ planning --

def relay_plan(coll: int, count: int, dtype, A: int, R: int,
               opts: Optional[RelayOpts] = None) -> RelayPlan:
    p = RelayPlan()
    _check(lib().relay_plan(coll, count, dtype_code(dtype), A, R,
                            ctypes.byref(opts) if opts is not None else None, ctypes.byref(p)))
    return p


def relay_plan_link_bytes(plan: RelayPlan) -> np.ndarray:
    G, R = plan.num_groups, plan.R
    out = np.zeros(max(G, 1) * R * R, np.uint64)
    _check(lib().relay_plan_link_bytes(ctypes.byref(plan),
                                       out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)),
                                       out.size))
    return out[: G * R * R].reshape(G, R, R)


def relay_plan_cost_bytes(plan: RelayPlan) -> int:
    return int(lib().relay_plan_cost_bytes(ctypes.byref(plan)))


def relay_plan_passes(plan: RelayPlan, in_place: bool = False) -> list:
    n = lib().relay_plan_passes(ctypes.byref(plan), int(in_place), None, 0)
    if n < 0:
        raise RelayError(ERR_INVALID_ARGUMENT, "not a plan")
    buf = (RelayPassInfo * max(n, 1))()
    lib().relay_plan_passes(ctypes.byref(plan), int(in_place), buf, n)
    return [{"kind": buf[i].kind, "name": PASS_NAMES[buf[i].kind],
             "num_segments": buf[i].num_segments, "bytes_read": buf[i].bytes_read,
             "bytes_written": buf[i].bytes_written} for i in range(n)]


def relay_passthrough_helper_size(count_g: int, A: int, num_chunks: int) -> int:
    return int(lib().relay_passthrough_helper_size(count_g, A, num_chunks))


def relay_helper_size(plan: RelayPlan) -> int:
    return int(lib().relay_helper_size(ctypes.byref(plan)))


def relay_active_scratch_size(plan: RelayPlan) -> int:
    return int(lib().relay_active_scratch_size(ctypes.byref(plan)))


def relay_helper_contract_size(coll: int, count: int, A: int, R: int) -> int:
    return int(lib().relay_helper_contract_size(coll, count, A, R))


def relay_pass_name(kind: int) -> str:
    return lib().relay_pass_name(kind).decode()


# --------------------------------------------------------------------- collectives --

def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("relay buffers must be CUDA tensors (device memory)")
    if not x.is_contiguous():
        raise ValueError("relay buffers must be contiguous")
    return x.data_ptr()


def _ptr_array(xs: Sequence, R: int):
    if len(xs) != R:
        raise ValueError(f"expected {R} entries (one per virtual rank), got {len(xs)}")
    return (ctypes.c_void_p * R)(*[_ptr(x) for x in xs])


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _pad(xs, R):
    xs = list(xs) if xs is not None else []
    return xs + [None] * (R - len(xs))


def relay_allreduce(send, recv, scratch, count: int, dtype, A: int, R: int, scale: float = 1.0,
                    opts: Optional[RelayOpts] = None, stream=None) -> None:
    _check(lib().relay_allreduce(_ptr_array(_pad(send, R), R), _ptr_array(_pad(recv, R), R),
                                 _ptr_array(_pad(scratch, R), R), count, dtype_code(dtype), A, R,
                                 scale, ctypes.byref(opts) if opts is not None else None,
                                 _stream(stream)))


def relay_reduce_scatter(send, recv, scratch, recv_count: int, dtype, A: int, R: int,
                         scale: float = 1.0, opts: Optional[RelayOpts] = None, stream=None) -> None:
    _check(lib().relay_reduce_scatter(_ptr_array(_pad(send, R), R), _ptr_array(_pad(recv, R), R),
                                      _ptr_array(_pad(scratch, R), R), recv_count,
                                      dtype_code(dtype), A, R, scale,
                                      ctypes.byref(opts) if opts is not None else None,
                                      _stream(stream)))


def relay_all_gather(send, recv, scratch, send_count: int, dtype, A: int, R: int,
                     opts: Optional[RelayOpts] = None, stream=None) -> None:
    _check(lib().relay_all_gather(_ptr_array(_pad(send, R), R), _ptr_array(_pad(recv, R), R),
                                  _ptr_array(_pad(scratch, R), R), send_count, dtype_code(dtype),
                                  A, R, ctypes.byref(opts) if opts is not None else None,
                                  _stream(stream)))


def relay_all_to_all(send, recv, scratch, segment_count: int, dtype, A: int, R: int,
                     opts: Optional[RelayOpts] = None, stream=None) -> None:
    _check(lib().relay_all_to_all(_ptr_array(_pad(send, R), R), _ptr_array(_pad(recv, R), R),
                                  _ptr_array(_pad(scratch, R), R), segment_count,
                                  dtype_code(dtype), A, R,
                                  ctypes.byref(opts) if opts is not None else None,
                                  _stream(stream)))


def relay_allreduce_noalloc(send, recv, count: int, dtype, A: int, R: int, scale: float = 1.0,
                            opts: Optional[RelayOpts] = None, stream=None) -> None:
    """Allreduce whose scratch is the library's built-in device array (see relay.h)."""
    _check(lib().relay_allreduce_noalloc(_ptr_array(_pad(send, R), R), _ptr_array(_pad(recv, R), R),
                                         count, dtype_code(dtype), A, R, scale,
                                         ctypes.byref(opts) if opts is not None else None,
                                         _stream(stream)))


COLLECTIVES = {ALLREDUCE: relay_allreduce, REDUCE_SCATTER: relay_reduce_scatter,
               ALL_GATHER: relay_all_gather, ALL_TO_ALL: relay_all_to_all}


def alloc_scratch(plan: RelayPlan, device, torch_dtype=None):
    """R scratch buffers sized by the plan (None where a rank needs none)."""
    import torch
    td = torch_dtype or {F32: torch.float32, BF16: torch.bfloat16, I32: torch.int32}[plan.dtype]
    out = []
    for r in range(plan.R):
        n = plan.active_scratch_elems if r < plan.A else plan.helper_elems
        out.append(torch.empty(n, dtype=td, device=device) if n > 0 else None)
    return out


# -------------------------------------------------------------- fused multi-group --

def group_ranks(g: int, A: int, R: int) -> list:
    """Global ranks of group g's local ranks: its A actives, then its helpers."""
    return [g * A + a for a in range(A)] + [r for r in range(R) if r // A != g]


def relay_multi_group(coll: int, counts: Sequence[int], send, recv, scratch, dtype, A: int,
                      scale: float = 1.0, opts: Optional[RelayOpts] = None, stream=None) -> None:
    """Fused call over len(counts) groups of A consecutive ranks (R = groups * A).
    send/recv: R entries (rank r's buffers for its own group); scratch: one list of R
    entries per group (rank r's scratch for that group)."""
    G = len(counts)
    R = G * A
    flat = [x for per_group in scratch for x in _pad(per_group, R)]
    if len(flat) != G * R:
        raise ValueError("scratch needs one list of R entries per group")
    c = (ctypes.c_size_t * G)(*counts)
    _check(lib().relay_multi_group(coll, G, c, _ptr_array(send, R), _ptr_array(recv, R),
                                   (ctypes.c_void_p * (G * R))(*[_ptr(x) for x in flat]),
                                   dtype_code(dtype), A, scale,
                                   ctypes.byref(opts) if opts is not None else None,
                                   _stream(stream)))


def relay_multi_group_link_bytes(coll: int, counts: Sequence[int], dtype, A: int,
                                 opts: Optional[RelayOpts] = None) -> np.ndarray:
    G = len(counts)
    R = G * A
    out = np.zeros(3 * R * R, np.uint64)
    phases = ctypes.c_int(0)
    c = (ctypes.c_size_t * G)(*counts)
    _check(lib().relay_multi_group_link_bytes(
        coll, G, c, dtype_code(dtype), A, ctypes.byref(opts) if opts is not None else None,
        out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), out.size, ctypes.byref(phases)))
    return out[: phases.value * R * R].reshape(phases.value, R, R)


def alloc_multi_scratch(coll: int, counts: Sequence[int], dtype, A: int, device,
                        opts: Optional[RelayOpts] = None):
    """Per group, R scratch buffers sized by that group's plan (None where not needed)."""
    import torch
    G = len(counts)
    R = G * A
    td = {F32: torch.float32, BF16: torch.bfloat16, I32: torch.int32}[dtype_code(dtype)]
    out = []
    for g in range(G):
        p = relay_plan(coll, counts[g], dtype, A, R, opts)
        row = [None] * R
        for l, r in enumerate(group_ranks(g, A, R)):
            n = p.active_scratch_elems if l < A else p.helper_elems
            if n > 0:
                row[r] = torch.empty(n, dtype=td, device=device)
        out.append(row)
    return out


# ------------------------------------------------------------ flat pack / unpack --

def relay_pack_flat(tensors: Sequence, flat, dtype=None, stream=None) -> None:
    """Copy `tensors` end to end into `flat` (one launch)."""
    n = len(tensors)
    dt = dtype_code(dtype if dtype is not None else flat.dtype)
    counts = (ctypes.c_size_t * max(n, 1))(*[t.numel() for t in tensors])
    _check(lib().relay_pack_flat((ctypes.c_void_p * max(n, 1))(*[_ptr(t) for t in tensors]),
                                 counts, n, _ptr(flat), dt, _stream(stream)))


def relay_unpack_flat(flat, tensors: Sequence, dtype=None, stream=None) -> None:
    """Copy consecutive pieces of `flat` back into `tensors` (one launch)."""
    n = len(tensors)
    dt = dtype_code(dtype if dtype is not None else flat.dtype)
    counts = (ctypes.c_size_t * max(n, 1))(*[t.numel() for t in tensors])
    _check(lib().relay_unpack_flat(_ptr(flat), (ctypes.c_void_p * max(n, 1))(*[_ptr(t) for t in tensors]),
                                   counts, n, dt, _stream(stream)))


# ---------------------------------------------------------------------- host link --

def _any_ptr(x) -> int:
    """Address of a contiguous tensor in device memory or host memory (pinned or not)."""
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("relay_copy tensors must be contiguous")
    return x.data_ptr()


def relay_copy(dst, src, max_ctas: int = 0, stream=None) -> None:
    """Copy `src` into `dst` (same dtype and numel) with the library's streaming kernel.
    Either may be a CUDA tensor or a host tensor (pinned, or pageable where the device
    reads host page tables); max_ctas caps the launch's CTAs (0: one per 16 KiB tile)."""
    if dst.dtype != src.dtype or dst.numel() != src.numel():
        raise ValueError("relay_copy: dst and src must have the same dtype and size")
    _check(lib().relay_copy(_any_ptr(dst), _any_ptr(src), src.numel(), dtype_code(src.dtype),
                            max_ctas, _stream(stream)))
