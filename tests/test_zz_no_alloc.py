"""relay_allreduce_noalloc: the allreduce entry point for callers that cannot allocate
device memory when they call it (an allocator or memory-pool hook, a process whose HBM
is fully reserved, a path that cannot afford an allocation's synchronisation). It takes
no scratch argument; its scratch is the library's built-in device array.

Checked through the C ABI against relay_allreduce with caller-allocated scratch, on two
calls in a row (the array keeps the first call's contents), for the tolerances of the
other parity tests (bit-exact here: same kernels, same order). This file runs last so a
stop-at-first-failure run has already run every other test; it also passes alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import pack_virtual_rank_gb300 as rv
import synth

pytestmark = pytest.mark.gpu

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
        for a in range(A):
            g, r = synth.to_numpy(got[a]), synth.to_numpy(ref[a])
            assert np.array_equal(g, r)


def test_noalloc_rejects_what_does_not_fit():
    R, A, count = 8, 2, 64 << 20                   # 64 Mi bf16 elements: needs ~256 MiB
    L = rv.lib()
    x = [torch.zeros(1, dtype=torch.bfloat16, device="cuda") for _ in range(2 * A)]
    # the size check comes before any access, so 1-element stand-ins are enough
    st = L.relay_allreduce_noalloc(_arr(x[:A], R), _arr(x[A:], R), count, rv.BF16, A, R, 0.5,
                                   None, None)
    assert st == rv.ERR_INVALID_ARGUMENT
    assert b"scratch" in L.relay_last_error()
