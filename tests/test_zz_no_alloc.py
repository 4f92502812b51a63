"""relay_allreduce_noalloc: the allreduce entry point for callers that cannot allocate
device memory when they call it (an allocator or memory-pool hook, a process whose HBM
is fully reserved, a path that cannot afford an allocation's synchronisation). It takes
no scratch argument; its scratch is the library's built-in device array.

Checked through the C ABI against relay_allreduce with caller-allocated scratch and
against the oracle, on two calls in a row (the array keeps the first call's contents),
for the tolerances of the other parity tests (bit-exact here: same kernels, same order).
The largest call the array admits runs with canary bands around every buffer, and the
device's free memory and torch's reserved memory must not change across calls. This file
runs last so a stop-at-first-failure run has already run every other test; it also
passes alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import harness as hz
import oracle as orc
import pack_virtual_rank_gb300 as rv
import synth

pytestmark = pytest.mark.gpu

LIMIT = 64 << 20          # RELAY_NOALLOC_SCRATCH_BYTES in include/relay.h

TORCH = {rv.F32: torch.float32, rv.BF16: torch.bfloat16}


def _arr(xs, R):
    xs = list(xs) + [None] * (R - len(xs))
    return (ctypes.c_void_p * R)(*[x.data_ptr() if x is not None else None for x in xs])


@pytest.mark.parametrize("dtype,A,count,sched", [
    (rv.BF16, 2, 3 << 20, rv.SCHEDULE_AUTO),        # relay, numChunks 8
    (rv.F32, 2, 65536, rv.SCHEDULE_RELAY),
    (rv.BF16, 2, 100_000, rv.SCHEDULE_AUTO),        # below 2 MB: one full exchange
    (rv.BF16, 4, (1 << 20) + 77, rv.SCHEDULE_AUTO),
])
def test_noalloc_matches_allreduce_twice(dtype, A, count, sched):
    R = 8
    L = rv.lib()
    opts = rv.make_opts(schedule=sched)
    plan = rv.relay_plan(rv.ALLREDUCE, count, dtype, A, R, opts)
    scale = 1.0 / A
    scratch = rv.alloc_scratch(plan, "cuda")
    for call in range(2):
        name = "f32" if dtype == rv.F32 else "bf16"
        xs = [synth.rank_input(30 + call, r, count, name).cuda() for r in range(A)]
        ref = [torch.empty_like(x) for x in xs]
        got = [torch.full_like(x, 7) for x in xs]
        st = L.relay_allreduce(_arr(xs, R), _arr(ref, R),
                               (ctypes.c_void_p * R)(*[s.data_ptr() if s is not None else None
                                                       for s in scratch]),
                               count, dtype, A, R, scale, ctypes.byref(opts), None)
        assert st == rv.OK
        st = L.relay_allreduce_noalloc(_arr(xs, R), _arr(got, R), count, dtype, A, R, scale,
                                       ctypes.byref(opts), None)
        assert st == rv.OK, L.relay_last_error()
        torch.cuda.synchronize()
        q = orc.allreduce(dtype, [synth.to_numpy(x) for x in xs], scale)[2]
        for a in range(A):
            g, r = synth.to_numpy(got[a]), synth.to_numpy(ref[a])
            assert np.array_equal(g, r)
            assert np.array_equal(g, q)


def _need(count, dtype, A, R):
    """Bytes of the built-in array a call needs, as the header states it: every active's
    and every helper's scratch, each rounded up to 256 bytes."""
    p = rv.relay_plan(rv.ALLREDUCE, count, dtype, A, R)
    r256 = lambda b: (b + 255) // 256 * 256
    return A * r256(p.active_scratch_elems * p.esize) + p.H * r256(p.helper_elems * p.esize)


@pytest.mark.parametrize("dtype,count", [(rv.BF16, 16 << 20), (rv.F32, 8 << 20)])
def test_noalloc_largest_call(dtype, count):
    """The largest 2-active relay allreduce the array holds: its scratch fills the 64 MiB
    exactly, one more element is refused. Two calls in a row match the oracle with every
    canary intact, and allocate nothing."""
    A, R = 2, 8
    L = rv.lib()
    assert _need(count, dtype, A, R) == LIMIT
    assert _need(count + 1, dtype, A, R) > LIMIT
    name = "f32" if dtype == rv.F32 else "bf16"
    inputs = [[synth.rank_input(50 + call, r, count, name) for r in range(A)] for call in range(3)]
    send = [hz.Guarded(count, dtype, "cuda") for _ in range(A)]
    recv = [hz.Guarded(count, dtype, "cuda") for _ in range(A)]
    scale = 1.0 / A
    opts = rv.make_opts()

    def call(k):
        for a in range(A):
            send[a].view.copy_(inputs[k][a])
        return L.relay_allreduce_noalloc(_arr([b.view for b in send], R), _arr([b.view for b in recv], R),
                                         count, dtype, A, R, scale, ctypes.byref(opts), None)

    # one call first: the library's device code (and its array) is loaded, and the
    # array's address looked up, by the first call on the device at the latest
    assert call(2) == rv.OK, L.relay_last_error()
    torch.cuda.synchronize()
    free0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_reserved()
    for k in range(2):
        assert call(k) == rv.OK, L.relay_last_error()
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, "device memory was allocated"
        assert torch.cuda.memory_reserved() == reserved0
        q = orc.allreduce(dtype, [synth.to_numpy(x) for x in inputs[k]], scale)[2]
        for a in range(A):
            assert np.array_equal(synth.to_numpy(recv[a].view), q)
        assert all(b.guards_intact() for b in send + recv)
    st = L.relay_allreduce_noalloc(_arr([b.view for b in send], R), _arr([b.view for b in recv], R),
                                   count + 1, dtype, A, R, scale, ctypes.byref(opts), None)
    assert st == rv.ERR_INVALID_ARGUMENT and b"scratch" in L.relay_last_error()


def test_noalloc_rejects_what_does_not_fit():
    R, A, count = 8, 2, 64 << 20                   # 64 Mi bf16 elements: needs ~256 MiB
    L = rv.lib()
    x = [torch.zeros(1, dtype=torch.bfloat16, device="cuda") for _ in range(2 * A)]
    # the size check comes before any access, so 1-element stand-ins are enough
    st = L.relay_allreduce_noalloc(_arr(x[:A], R), _arr(x[A:], R), count, rv.BF16, A, R, 0.5,
                                   None, None)
    assert st == rv.ERR_INVALID_ARGUMENT
    assert b"scratch" in L.relay_last_error()
