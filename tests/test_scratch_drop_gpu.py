"""The chained launch drops dead scratch lines from L2 without a write-back (the
RELAY_FLAG_KEEP_SCRATCH note in relay.h). These tests check that no live byte is ever
lost to a drop:

- every buffer of a call is packed back to back in one arena, at offsets off the 128-byte
  line grid, so that scratch shares its end lines with inputs, outputs and guard bytes;
- every byte of the arena is written once, pushed out to memory by a large write, then
  written again just before the call: memory holds a stale value, L2 the live one, and a
  line dropped by mistake reads back stale;
- after the call, the outputs equal the oracle's, the inputs and guard bytes are
  unchanged, and the same call with RELAY_FLAG_KEEP_SCRATCH gives bit-identical outputs.
"""
import re

import numpy as np
import pytest
import torch

import harness as hz
import pack_virtual_rank_gb300 as rv

pytestmark = pytest.mark.gpu

STALE = 0x11
LIVE = 0x5A
NAMES = {rv.ALLREDUCE: "allreduce", rv.REDUCE_SCATTER: "reduce_scatter",
         rv.ALL_GATHER: "all_gather", rv.ALL_TO_ALL: "all_to_all"}

CASES = [
    # coll, A, R, dtype, count
    (rv.ALLREDUCE, 2, 8, rv.BF16, 200_003),
    (rv.ALLREDUCE, 4, 8, rv.F32, 100_001),
    (rv.ALLREDUCE, 2, 5, rv.I32, 65_537),
    (rv.REDUCE_SCATTER, 2, 8, rv.F32, 70_001),
    (rv.REDUCE_SCATTER, 4, 8, rv.BF16, 50_001),     # fp32 helper partials
    (rv.ALL_GATHER, 2, 8, rv.BF16, 90_001),
    (rv.ALL_GATHER, 4, 8, rv.F32, 40_003),
    (rv.ALL_TO_ALL, 4, 8, rv.BF16, 50_001),
    (rv.ALL_TO_ALL, 2, 8, rv.F32, 30_001),
]


@pytest.fixture(scope="module")
def flush():
    """A buffer well past the 126 MiB L2: writing it evicts (and writes back) every line."""
    return torch.empty(512 << 20, dtype=torch.uint8, device="cuda")


def _dropped(how):
    m = re.fullmatch(r"chained: (\d+) groups, (\d+) pieces, (\d+) dropped", how)
    assert m, how
    return int(m.group(3))


def _arena_call(flush, coll, A, R, dtype, count, skew, flags):
    E = rv.ESIZE[dtype]
    opts = rv.make_opts(schedule=rv.SCHEDULE_RELAY, flags=flags | rv.FLAG_CHECK_HAZARDS)
    plan = rv.relay_plan(coll, count, dtype, A, R, opts)
    c = hz.Call()
    c.plan, c.coll, c.A, c.R, c.count, c.dtype = plan, coll, A, R, count, dtype
    c.scale = 1.0 if dtype == rv.I32 else 1.0 / A
    c.in_place = False
    hz.read_request(c, rv.SCHEDULE_RELAY, -1, flags)
    hz.assert_plan_agrees(c)

    # layout: send a, a helper's scratch, recv a, active a's scratch, ...; then the rest of
    # the helpers. Gaps of 0, 1 and 3 elements and 128 - E bytes cycle between buffers.
    order = []
    helpers = list(range(A, R))
    for a in range(A):
        order.append(("send", a, plan.input_elems))
        if helpers:
            h = helpers.pop(0)
            order.append(("scratch", h, plan.helper_elems))
        order.append(("recv", a, plan.output_elems))
        order.append(("scratch", a, plan.active_scratch_elems))
    order += [("scratch", h, plan.helper_elems) for h in helpers]
    gaps = [0, E, 3 * E, 128 - E]
    off = skew
    place = {}
    for i, (kind, r, n) in enumerate(order):
        if n <= 0:
            continue
        off += gaps[i % len(gaps)]
        place[(kind, r)] = (off, n)
        off += n * E
    total = off + 256
    arena = torch.empty(total, dtype=torch.uint8, device="cuda")
    view = lambda o, n: arena[o:o + n * E].view(hz.TORCH[dtype])

    xs = hz.make_inputs(7, A, plan.input_elems, dtype, "cuda")
    arena.fill_(STALE)
    flush.fill_(1)
    arena.fill_(LIVE)
    send = [view(*place[("send", a)]) for a in range(A)]
    recv = [view(*place[("recv", a)]) for a in range(A)]
    for a in range(A):
        send[a].copy_(xs[a])
    scratch = [view(*place[("scratch", r)]) if ("scratch", r) in place else None
               for r in range(R)]
    fn = rv.COLLECTIVES[coll]
    pad = [None] * (R - A)
    if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER):
        fn(send + pad, recv + pad, scratch, count, dtype, A, R, c.scale, opts)
    else:
        fn(send + pad, recv + pad, scratch, count, dtype, A, R, opts)
    c.launch = rv.last_launch()
    torch.cuda.synchronize()
    rv.device_status()

    # bytes outside every buffer: still the live fill
    mask = torch.ones(total, dtype=torch.bool, device="cuda")
    for (kind, r), (o, n) in place.items():
        mask[o:o + n * E] = False
    outside = arena[mask]
    assert bool((outside == LIVE).all().item()), "a byte outside the call's buffers changed"
    c.inputs, c.send, c.recv, c.scratch = xs, send, recv, scratch
    return c


@pytest.mark.parametrize("skew_units", [0, 1, 63])
@pytest.mark.parametrize("case", CASES,
                         ids=[f"{NAMES[t[0]]}-A{t[1]}-R{t[2]}-{hz.NAME[t[3]]}" for t in CASES])
def test_dropped_lines_keep_every_live_byte(flush, case, skew_units):
    coll, A, R, dtype, count = case
    skew = skew_units * rv.ESIZE[dtype]
    c = _arena_call(flush, coll, A, R, dtype, count, skew, 0)
    assert _dropped(c.launch) > 0, c.launch
    xs_host = [hz.host(x) for x in c.inputs]
    for a in range(A):
        hz.check_window(c, a, 0, hz.out_elems(c), xs_host)
        assert np.array_equal(hz.host(c.send[a]), xs_host[a]), "input changed"
    got = [hz.host(y) for y in c.recv]

    k = _arena_call(flush, coll, A, R, dtype, count, skew, rv.FLAG_KEEP_SCRATCH)
    assert _dropped(k.launch) == 0, k.launch
    for a in range(A):
        assert np.array_equal(hz.host(k.recv[a]), got[a]), "kept and dropped scratch disagree"


TIER_CASES = [
    # one program per size of the chained kernel's parameter table (up to 32, 128 and 384
    # pieces): coll, A, R, dtype, count, smallest and largest piece count of the tier
    (rv.ALLREDUCE, 2, 8, rv.BF16, 1 << 20, 1, 32),
    (rv.REDUCE_SCATTER, 4, 8, rv.BF16, 1 << 18, 33, 128),
    (rv.ALL_GATHER, 4, 8, rv.BF16, 1 << 20, 33, 128),
    (rv.ALL_TO_ALL, 4, 8, rv.BF16, 1 << 18, 129, 384),
    (rv.ALL_TO_ALL, 4, 8, rv.BF16, (1 << 18) + 1, 129, 384),
    (rv.REDUCE_SCATTER, 4, 21, rv.BF16, 16391, 129, 384),   # 372 pieces: the table's top
]


@pytest.mark.parametrize("case", TIER_CASES,
                         ids=[f"{NAMES[t[0]]}-A{t[1]}-R{t[2]}-{t[4]}" for t in TIER_CASES])
def test_dropped_lines_leave_l2_unwritten(flush, case):
    """Dropped lines really leave L2 without a write-back, whatever the size of the
    kernel's parameter table: the scratch (a few MiB, well inside L2) holds a stale value in
    memory under a live one in L2 before the call; afterwards nearly every scratch byte
    reads back stale (what memory held), and with RELAY_FLAG_KEEP_SCRATCH nearly none does
    (only data bytes that happen to equal the stale byte)."""
    coll, A, R, dtype, count, lo, hi = case
    fractions = []
    for flags in (0, rv.FLAG_KEEP_SCRATCH):
        opts = rv.make_opts(schedule=rv.SCHEDULE_RELAY, flags=flags)
        plan = rv.relay_plan(coll, count, dtype, A, R, opts)
        xs = hz.make_inputs(11, A, plan.input_elems, dtype, "cuda")
        ys = [torch.empty(plan.output_elems, dtype=xs[0].dtype, device="cuda") for _ in range(A)]
        scratch = rv.alloc_scratch(plan, "cuda")
        live = [s for s in scratch if s is not None]
        for s in live:
            s.view(torch.uint8).fill_(STALE)
        flush.fill_(1)
        for s in live:
            s.view(torch.uint8).fill_(LIVE)
        fn = rv.COLLECTIVES[coll]
        pad = [None] * (R - A)
        if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER):
            fn(xs + pad, ys + pad, scratch, count, dtype, A, R, 1.0 / A, opts)
        else:
            fn(xs + pad, ys + pad, scratch, count, dtype, A, R, opts)
        how = rv.last_launch()
        torch.cuda.synchronize()
        m = re.fullmatch(r"chained: (\d+) groups, (\d+) pieces, (\d+) dropped", how)
        assert m and lo <= int(m.group(2)) <= hi, how
        total = sum(s.numel() * s.element_size() for s in live)
        stale = sum(int((s.view(torch.uint8) == STALE).sum().item()) for s in live)
        fractions.append(stale / total)
    assert fractions[0] >= 0.9, fractions
    assert fractions[1] <= 0.02, fractions
