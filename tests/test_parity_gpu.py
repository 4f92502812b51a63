"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Every output element is compared bit for bit with the oracle (the kernels sum in the
oracle's order, so fp32 and bf16 results are bit-identical, and the stated
tolerances -- fp32 relative error 1e-6 against the fp64 sum, bf16 within one ulp of
the fp32 sum -- are checked on top); int32, all-gather and all-to-all are bit-exact.
Canary bands around every buffer must stay untouched, inputs must be unchanged
out-of-place, and no launch may hold two segments that race (checked on the host).

Page: "Link-balance the sharded relay schedules (up to 3.2x vs NCCL)".
"""
import re

import numpy as np
import pytest
import torch

import harness as hz
import oracle as orc
import pack_virtual_rank_gb300 as rv

pytestmark = pytest.mark.gpu

SMALL_COUNTS = [1, 2, 127, 128, 129, 1000, 1023, 1024, 1025, 1792, 2047, 2048, 4109, 9000,
                65536 + 77]
SCHEDULES = [rv.SCHEDULE_AUTO, rv.SCHEDULE_RELAY, rv.SCHEDULE_DIRECT, rv.SCHEDULE_LEGACY]


def _scale(coll, A, dtype):
    if coll not in (rv.ALLREDUCE, rv.REDUCE_SCATTER) or dtype == rv.I32:
        return 1.0
    return 1.0 / A


@pytest.mark.parametrize("dtype", [rv.F32, rv.BF16, rv.I32])
@pytest.mark.parametrize("A", [2, 4])
@pytest.mark.parametrize("coll", [rv.ALLREDUCE, rv.REDUCE_SCATTER, rv.ALL_GATHER, rv.ALL_TO_ALL])
@pytest.mark.parametrize("launch", [0, rv.FLAG_SEPARATE_PASSES, rv.FLAG_FUSED_PASSES])
def test_small_sizes_every_schedule(coll, A, dtype, launch):
    """Every count around the 128-element alignment and chunk boundaries, every
    schedule, R = A+1 (one helper) and R = 8, in-place and out-of-place; small calls run
    as one chained launch by default, pass by pass or as one cooperative launch when
    asked."""
    n = 0
    for R in (A + 1, 8):
        for count in SMALL_COUNTS:
            for sched in SCHEDULES:
                if sched == rv.SCHEDULE_LEGACY and A != 2:
                    continue
                for in_place in (False, True):
                    if in_place and coll == rv.ALL_TO_ALL:
                        continue
                    try:
                        rv.relay_plan(coll, count, dtype, A, R, rv.make_opts(schedule=sched))
                    except rv.RelayError:
                        assert sched == rv.SCHEDULE_LEGACY   # chunk aligns down to 0
                        continue
                    c = hz.run(coll, A, R, count, dtype, _scale(coll, A, dtype), config=7,
                               schedule=sched, in_place=in_place, flags=launch)
                    hz.check_all(c)
                    n += 1
    assert n > 50


@pytest.mark.parametrize("coll", [rv.ALLREDUCE, rv.REDUCE_SCATTER, rv.ALL_GATHER, rv.ALL_TO_ALL])
@pytest.mark.parametrize("dtype", [rv.F32, rv.BF16])
@pytest.mark.parametrize("shift", [1, 3])
@pytest.mark.parametrize("launch", [0, rv.FLAG_SEPARATE_PASSES, rv.FLAG_FUSED_PASSES])
def test_unaligned_buffers(coll, dtype, shift, launch):
    """Buffers that are element- but not 16-byte-aligned: all sharing one offset
    (vector path after a peeled prologue) and with mixed offsets (per-element path), in the
    one-launch kernel and pass by pass (where misaligned copy passes run in one launch of
    the realign-all mode)."""
    for A in (2, 4):
        count = 5000 + 3
        sched = rv.SCHEDULE_RELAY
        opts = rv.make_opts(schedule=sched, flags=rv.FLAG_CHECK_HAZARDS | launch)
        plan = rv.relay_plan(coll, count, dtype, A, 8, opts)
        xs = hz.make_inputs(11, A, plan.input_elems, dtype, "cuda")
        td = hz.TORCH[dtype]

        def buf(n, s):
            full = torch.zeros(n + 64, dtype=td, device="cuda")
            return full[s:s + n]
        mixed = shift == 3
        send = [buf(plan.input_elems, 1) for _ in range(A)]
        for a in range(A):
            send[a].copy_(xs[a])
        recv = [buf(plan.output_elems, 3 if mixed else 1) for _ in range(A)]
        scratch = [buf(plan.active_scratch_elems, 1) if plan.active_scratch_elems else None
                   for _ in range(A)]
        scratch += [buf(plan.helper_elems, 5 if mixed else 1) for _ in range(8 - A)]
        fn = rv.COLLECTIVES[coll]
        args = (send + [None] * (8 - A), recv + [None] * (8 - A), scratch, count, dtype, A, 8)
        if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER):
            fn(*args, _scale(coll, A, dtype), opts)
        else:
            fn(*args, opts)
        torch.cuda.synchronize()
        c = hz.Call()
        c.plan, c.coll, c.A, c.R, c.count, c.dtype = plan, coll, A, 8, count, dtype
        c.scale, c.inputs, c.recv = _scale(coll, A, dtype), xs, recv
        hz.read_request(c, sched, -1, launch)
        hz.assert_plan_agrees(c)
        xs_host = [hz.host(x) for x in xs]
        for a in range(A):
            hz.check_window(c, a, 0, hz.out_elems(c), xs_host)


def test_many_helpers_split_launches():
    """R large enough that one group's segment table spans several launches."""
    for coll in (rv.REDUCE_SCATTER, rv.ALL_TO_ALL):
        c = hz.run(coll, 4, 40, 36 * 1024 + 5, rv.BF16, _scale(coll, 4, rv.BF16),
                   schedule=rv.SCHEDULE_RELAY)
        hz.check_all(c)


def test_repeat_calls_reuse_scratch():
    """Scratch keeps the previous call's contents; results must not depend on them."""
    c = hz.run(rv.ALLREDUCE, 4, 8, 300_000, rv.BF16, 0.25, schedule=rv.SCHEDULE_RELAY)
    hz.check_all(c)
    xs2 = hz.make_inputs(99, 4, c.plan.input_elems, rv.BF16, "cuda")
    for a in range(4):
        c.send[a].copy_(xs2[a])
    rv.relay_allreduce(c.send + [None] * 4, c.recv + [None] * 4, c.scratch, c.count, rv.BF16, 4,
                       8, 0.25, rv.make_opts(schedule=rv.SCHEDULE_RELAY))
    torch.cuda.synchronize()
    c.inputs = xs2
    hz.check_all(c)


def test_special_values():
    """Signed zeros, infinities and values whose sums round to ties survive the path
    exactly as the oracle computes them."""
    n = 4096
    vals = torch.tensor([0.0, -0.0, 1.0, -1.0, float("inf"), 2.0 ** -130, 3.0e38, -3.0e38,
                         1.0 + 2.0 ** -8, 2.0 ** -8], dtype=torch.float32)
    g = torch.Generator().manual_seed(3)
    for dtype in (rv.F32, rv.BF16):
        xs = []
        for a in range(4):
            idx = torch.randint(0, len(vals), (n,), generator=g)
            x = vals[idx]
            xs.append((x if dtype == rv.F32 else x.to(torch.bfloat16)).cuda())
        for coll, A in ((rv.ALLREDUCE, 2), (rv.ALLREDUCE, 4), (rv.REDUCE_SCATTER, 4)):
            ins = [x[: n if coll == rv.ALLREDUCE else n] for x in xs[:A]]
            count = n if coll == rv.ALLREDUCE else n // A
            c = hz.run(coll, A, 8, count, dtype, 0.5, schedule=rv.SCHEDULE_RELAY, inputs=ins)
            xs_host = [hz.host(x) for x in ins]
            for a in range(A):
                got = hz.host(c.recv[a])
                q = hz.expected(c, xs_host, a, 0, hz.out_elems(c))[0]
                # overflowing pairs make -inf too, so 4-term sums can be NaN: any NaN
                # matches any NaN (the encoding of a NaN is not part of the contract);
                # every other value must match bit for bit
                if dtype == rv.BF16:
                    gf, qf = orc.bf16_to_f32(got), orc.bf16_to_f32(q)
                else:
                    gf, qf = got, q
                nan = np.isnan(qf)
                assert np.array_equal(np.isnan(gf), nan)
                assert np.array_equal(gf[~nan].view(np.uint32), qf[~nan].view(np.uint32))


def test_pass_events_time_every_pass():
    plan = rv.relay_plan(rv.ALLREDUCE, 1 << 22, rv.BF16, 2, 8)
    npass = len(rv.relay_plan_passes(plan))
    events = [torch.cuda.Event(enable_timing=True) for _ in range(npass + 1)]
    opts = rv.make_opts(pass_events=events)
    c = hz.run(rv.ALLREDUCE, 2, 8, 1 << 22, rv.BF16, 0.5, config=2)
    rv.relay_allreduce(c.send + [None] * 6, c.recv + [None] * 6, c.scratch, 1 << 22, rv.BF16, 2, 8,
                       0.5, opts)
    torch.cuda.synchronize()
    ms = [events[i].elapsed_time(events[i + 1]) for i in range(npass)]
    assert all(t > 0 for t in ms)
    with pytest.raises(rv.RelayError):
        rv.relay_allreduce(c.send + [None] * 6, c.recv + [None] * 6, c.scratch, 1 << 22, rv.BF16,
                           2, 8, 0.5, rv.make_opts(pass_events=events[:npass]))


def test_flat_pack_unpack_round_trip():
    """Caller tensor lists packed into one flat buffer and unpacked again, one launch
    each (commit D115998366); odd sizes and offsets take the unaligned paths."""
    g = torch.Generator().manual_seed(5)
    sizes = [1, 7, 128, 1000, 4097, 65536 + 3, 0, 300_001]
    for dtype in (rv.F32, rv.BF16, rv.I32):
        td = hz.TORCH[dtype]
        ts = [torch.randint(-1000, 1000, (n,), generator=g).to(td).cuda() for n in sizes]
        flat = hz.Guarded(sum(sizes), dtype, "cuda")
        rv.relay_pack_flat(ts, flat.view)
        torch.cuda.synchronize()
        exp = torch.cat([t.cpu() for t in ts])
        assert torch.equal(flat.view.cpu(), exp)
        outs = [hz.Guarded(n, dtype, "cuda") for n in sizes]
        rv.relay_unpack_flat(flat.view, [o.view for o in outs])
        torch.cuda.synchronize()
        for t, o in zip(ts, outs):
            assert torch.equal(o.view.cpu(), t.cpu()) and o.guards_intact()
        assert flat.guards_intact()


def test_cuda_graph_capture_and_replay():
    """A whole collective captured into a CUDA graph (kernel parameters are captured by
    value) replays to the same bits as a direct call, for small launch-bound sizes."""
    for coll, A, count in ((rv.ALLREDUCE, 2, 32 * 1024), (rv.REDUCE_SCATTER, 4, 40_000),
                           (rv.ALL_TO_ALL, 4, 30_000)):
        scale = 0.5 if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER) else 1.0
        c = hz.run(coll, A, 8, count, rv.BF16, scale, schedule=rv.SCHEDULE_RELAY)
        hz.check_all(c)
        ref = [hz.host(y).copy() for y in c.recv]
        for y in c.recv:
            y.zero_()
        opts = rv.make_opts(schedule=rv.SCHEDULE_RELAY)
        s = torch.cuda.Stream()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        fn = rv.COLLECTIVES[coll]
        args = (c.send + [None] * (8 - A), c.recv + [None] * (8 - A), c.scratch, count, rv.BF16, A, 8)
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER):
                    fn(*args, scale, opts, stream=s)
                else:
                    fn(*args, opts, stream=s)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        for y, r in zip(c.recv, ref):
            assert np.array_equal(hz.host(y), r)


@pytest.mark.parametrize("policy", [0, rv.FLAG_SEPARATE_PASSES, rv.FLAG_FUSED_PASSES])
@pytest.mark.parametrize("dtype", [rv.F32, rv.BF16, rv.I32])
def test_realigned_sources_span_whole_tiles(dtype, policy):
    """Odd counts put sources at different offsets modulo 16 bytes from their
    destinations over many whole tiles: the register-realigned vector path of the per-pass
    kernel, and the two-block path of the one-launch kernel (forced, and as the default
    policy picks it)."""
    cases = [(rv.ALL_TO_ALL, 4, 200_003), (rv.ALL_TO_ALL, 2, 300_001),
             (rv.REDUCE_SCATTER, 2, 300_001), (rv.REDUCE_SCATTER, 4, 250_001),
             (rv.ALL_GATHER, 4, 500_001), (rv.ALLREDUCE, 4, 1_000_001)]
    for coll, A, count in cases:
        scale = _scale(coll, A, dtype)
        for in_place in (False, True):
            if in_place and coll == rv.ALL_TO_ALL:
                continue
            c = hz.run(coll, A, 8, count, dtype, scale, config=13, schedule=rv.SCHEDULE_RELAY,
                       in_place=in_place, flags=policy)
            hz.check_all(c)


def test_pass_events_inside_a_cuda_graph():
    """Pass events recorded during stream capture time the passes of every replay."""
    c = hz.run(rv.ALLREDUCE, 2, 8, 1 << 20, rv.BF16, 0.5, schedule=rv.SCHEDULE_RELAY)
    npass = len(rv.relay_plan_passes(c.plan))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(npass + 1)]
    opts = rv.make_opts(schedule=rv.SCHEDULE_RELAY, pass_events=ev)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        rv.relay_allreduce(c.send + [None] * 6, c.recv + [None] * 6, c.scratch, 1 << 20, rv.BF16,
                           2, 8, 0.5, opts, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert all(ev[i].elapsed_time(ev[i + 1]) > 0 for i in range(npass))
    hz.check_all(c)


@pytest.mark.parametrize("coll", [rv.ALLREDUCE, rv.REDUCE_SCATTER, rv.ALL_GATHER, rv.ALL_TO_ALL])
@pytest.mark.parametrize("form", [rv.FLAG_FUSED_PASSES, rv.FLAG_CHAINED])
def test_one_launch_at_sizes_past_its_default(coll, form):
    """The one-launch forms forced on calls of many tiles per pass (cooperative: grid
    barriers between passes; chained: every dependency inside one CTA; both load
    through L2 what the launch wrote) match the oracle like the per-pass path."""
    # the cooperative kernel has no mixed-width path: the fp32 partial only chained
    partials = (rv.FLAG_PAYLOAD_PARTIAL, 0) if form == rv.FLAG_CHAINED else (rv.FLAG_PAYLOAD_PARTIAL,)
    for A in (2, 4):
        for count in (3 << 20, (1 << 21) + 129):
            scale = _scale(coll, A, rv.BF16)
            for in_place in (False, True):
                if in_place and coll == rv.ALL_TO_ALL:
                    continue
                for partial in partials:
                    if partial == 0 and not (coll == rv.REDUCE_SCATTER and A == 4):
                        continue
                    c = hz.run(coll, A, 8, count, rv.BF16, scale, config=17, in_place=in_place,
                               schedule=rv.SCHEDULE_RELAY, flags=form | partial)
                    want = "chained" if form == rv.FLAG_CHAINED else "cooperative"
                    assert c.launch.startswith(want), c.launch
                    hz.check_all(c)


@pytest.mark.parametrize("coll,R,dtype,count", [
    (rv.REDUCE_SCATTER, 21, rv.BF16, 16391),   # 372 pieces, fp32 partials
    (rv.REDUCE_SCATTER, 21, rv.F32, 65613),    # 372 pieces
    (rv.ALL_TO_ALL, 13, rv.BF16, 16391),       # 352 pieces
])
def test_largest_chained_programs(coll, R, dtype, count):
    """Programs near the chained launch's 384-piece limit (the last entries of the largest
    parameter table) match the oracle element by element under the default launch."""
    scale = 0.25 if coll == rv.REDUCE_SCATTER else 1.0
    c = hz.run(coll, 4, R, count, dtype, scale, config=23, schedule=rv.SCHEDULE_RELAY)
    m = re.fullmatch(r"chained: (\d+) groups, (\d+) pieces, (\d+) dropped", c.launch)
    assert m and int(m.group(2)) >= 350, c.launch
    hz.check_all(c)


def test_default_launch_forms():
    """Small calls run chained by default, mixed-width programs (a bf16 4-active
    reduce-scatter's fp32 partial) included; pass events and RELAY_FLAG_SEPARATE_PASSES run
    pass by pass; RELAY_FLAG_FUSED_PASSES runs the cooperative launch; large calls run
    chained too, the coalesced all-to-all's three-pass chains of copies included."""
    c = hz.run(rv.ALLREDUCE, 2, 8, 65536, rv.F32, 0.5, config=1, schedule=rv.SCHEDULE_RELAY)
    assert c.launch == "chained: 10 groups, 26 pieces, 16 dropped"
    hz.check_all(c)
    c = hz.run(rv.ALLREDUCE, 2, 8, 65536, rv.F32, 0.5, config=1, schedule=rv.SCHEDULE_RELAY,
               in_place=True)
    assert c.launch == "chained: 8 groups, 26 pieces, 16 dropped"
    hz.check_all(c)
    c = hz.run(rv.ALLREDUCE, 2, 8, 65536, rv.F32, 0.5, schedule=rv.SCHEDULE_RELAY,
               flags=rv.FLAG_SEPARATE_PASSES)
    assert c.launch == "passes"
    c = hz.run(rv.ALLREDUCE, 2, 8, 65536, rv.F32, 0.5, schedule=rv.SCHEDULE_RELAY,
               flags=rv.FLAG_FUSED_PASSES)
    assert c.launch == "cooperative"
    c = hz.run(rv.REDUCE_SCATTER, 4, 8, 40_000, rv.BF16, 0.25, schedule=rv.SCHEDULE_RELAY)
    assert c.wide and c.launch.startswith("chained")
    hz.check_all(c)
    c = hz.run(rv.REDUCE_SCATTER, 4, 8, 40_000, rv.BF16, 0.25, schedule=rv.SCHEDULE_RELAY,
               flags=rv.FLAG_FUSED_PASSES)
    assert c.wide and c.launch == "passes"          # no mixed-width path in that kernel
    hz.check_all(c)
    c = hz.run(rv.ALLREDUCE, 4, 8, 1 << 27, rv.BF16, 0.25)      # 1.9 GiB of pass traffic
    assert c.launch.startswith("chained")
    c = hz.run(rv.ALL_TO_ALL, 4, 8, (1 << 29) // 12, rv.BF16, schedule=rv.SCHEDULE_RELAY,
               gpu_generator=True)                              # 3-pass chains, 1.5 GB
    assert c.launch.startswith("chained")


@pytest.mark.parametrize("case", ["ar2", "a2a_odd"])
def test_chained_at_scale_full(case):
    """The chained launch forced on calls of 64-128 MiB per rank, every output element
    compared with the oracle: many tiles per group, L2 holding what each CTA just wrote."""
    if case == "ar2":
        c = hz.run(rv.ALLREDUCE, 2, 8, (1 << 26) + 3, rv.BF16, 0.5, config=2,
                   flags=rv.FLAG_CHAINED, gpu_generator=True)
    else:
        c = hz.run(rv.ALL_TO_ALL, 4, 8, (1 << 24) // 3, rv.I32, config=5,
                   schedule=rv.SCHEDULE_RELAY, flags=rv.FLAG_CHAINED, gpu_generator=True)
    assert c.launch.startswith("chained")
    assert case == "ar2" or c.count % 2 == 1
    hz.check_full(c)


def test_reduce_scatter_partial_precision():
    """4-active bf16 reduce-scatter. By default the helper partial crosses in fp32: results
    match the oracle's wide reading bit for bit and sit within one bf16 ulp of the fp64
    sum (the fp32 partial is exact unless a tiny term needs more than 24 bits next to
    large ones). With RELAY_FLAG_PAYLOAD_PARTIAL the partial crosses as bf16: results
    match the oracle's payload-typed reading bit for bit."""
    for m, in_place in ((300_000, False), (250_001, True), (1 << 20, False)):
        for flags in (0, rv.FLAG_SEPARATE_PASSES, rv.FLAG_PAYLOAD_PARTIAL):
            c = hz.run(rv.REDUCE_SCATTER, 4, 8, m, rv.BF16, 0.25, config=19,
                       schedule=rv.SCHEDULE_RELAY, in_place=in_place, flags=flags)
            assert c.wide == (not flags & rv.FLAG_PAYLOAD_PARTIAL)
            hz.check_all(c)
            if c.wide:
                xs = [hz.host(x) for x in c.inputs]
                for o in range(4):
                    r64 = orc.reduce_scatter(rv.BF16, xs, m, o, 0.25, 0)[0]
                    got = orc.bf16_to_f32(hz.host(c.recv[o])).astype(np.float64)
                    assert np.all(np.abs(got - r64) <= hz.bf16_ulp(r64.astype(np.float32)))
