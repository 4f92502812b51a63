"""Host-side checks of the C-ABI library (no GPU): every declared symbol is exported,
the planner and the link-byte accountant agree with the oracle's independent
restatement, pass byte counts follow the schedules' closed forms, and invalid calls
are rejected before anything is launched.

Page: "Link-balance the sharded relay schedules (up to 3.2x vs NCCL)" -- "item k" of
its summary, "Dnnnnnnnnn" a commit of its stack.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import pack_virtual_rank_gb300 as rv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def test_every_declared_symbol_is_exported(relay_lib):
    header = open(os.path.join(ROOT, "include", "relay.h")).read()
    declared = set(re.findall(r"\b(relay_[a-z0-9_]+)\s*\(", header))
    assert {"relay_plan", "relay_allreduce", "relay_reduce_scatter", "relay_all_gather",
            "relay_all_to_all"} <= declared
    for name in sorted(declared):
        assert hasattr(relay_lib, name), name
    assert relay_lib.relay_abi_version() == 1


def test_struct_sizes_match_header():
    # the ctypes mirrors must have the C layouts (all fields 4- or 8-byte, no padding)
    assert ctypes.sizeof(rv.RelayPlan) == 10 * 4 + 15 * 8
    assert ctypes.sizeof(rv.RelayOpts) == 4 + 4 + 8 + 8 + 4 + 4
    assert ctypes.sizeof(rv.RelayPassInfo) == 24


# ---------------------------------------------------------------- planner parity --

def _grid():
    counts = [0, 1, 2, 127, 128, 1023, 1024, 1025, 1792, 2047, 4109, 65536, (1 << 20) + 13,
              5120 * 1024, 50 << 20]
    for coll in range(4):
        for A in (2, 4):
            for R in (A + 1, 8, 12):
                for dt in (rv.F32, rv.BF16):
                    for count in counts:
                        for sched in (0, 1, 2, 3):
                            if sched == 3 and A == 4:
                                continue
                            yield coll, A, R, dt, count, sched


@pytest.mark.parametrize("coll", range(4))
def test_planner_and_accountant_match_oracle(orc, coll):
    n = 0
    for c, A, R, dt, count, sched in _grid():
        if c != coll:
            continue
        E = rv.ESIZE[dt]
        for pm in (500, 780):
            # the oracle's cost model carries the 4-active reduce-scatter partial as one
            # payload-typed chunk (item 6); the library's default fp32 partial doubles
            # that hop and is checked separately
            opts = rv.make_opts(offload_permille=pm, schedule=sched, flags=rv.FLAG_PAYLOAD_PARTIAL)
            try:
                g, gv = orc.plan(coll, A, R, count, E, permille=pm, force=sched)
            except ValueError:
                with pytest.raises(rv.RelayError):
                    rv.relay_plan(coll, count, dt, A, R, opts)
                continue
            p = rv.relay_plan(coll, count, dt, A, R, opts)
            assert (p.kind, p.num_groups, p.chunk) == (g["kind"], g["groups"], g["chunk"])
            if A == 2:
                assert (p.dirA_offset, p.dirA_size, p.dirB_size) == (g["dirA_off"], g["dirA"],
                                                                      g["dirB"])
            else:
                assert (p.direct_total, p.direct_g1, p.direct_g2) == (g["pD"], g["d1"], g["d2"])
                assert (p.owner_slice, p.owner_slice_last) == (g["owner_slice"],
                                                               g["owner_last"])
            lib_t = rv.relay_plan_link_bytes(p)
            orc_t = orc.link_elems(gv).astype(np.uint64) * np.uint64(E)
            assert lib_t.shape == orc_t.shape and np.array_equal(lib_t, orc_t)
            assert rv.relay_plan_cost_bytes(p) == orc.cost_elems(gv) * E
            n += 1
    assert n > 300


def test_reference_workload_geometry():
    # allreduce, A=2 of R=8, 65536 fp32, relay forced: numChunks = 8, chunk 8192, direct
    # share d = count/4 = 16384 riding the two groups; cost 0.25*count per link direction
    p = rv.relay_plan(rv.ALLREDUCE, 65536, rv.F32, 2, 8, rv.make_opts(schedule=rv.SCHEDULE_RELAY))
    assert (p.chunk, p.dirA_offset, p.dirA_size, p.dirB_size) == (8192, 49152, 8192, 8192)
    assert p.dirA_size + p.dirB_size == 65536 // 4
    t = rv.relay_plan_link_bytes(p)
    assert t[:, 0, 1].sum() == t[:, 1, 0].sum() == 65536 // 4 * 4
    assert rv.relay_plan_cost_bytes(p) == 65536 // 4 * 4
    for g in range(2):   # every used link carries exactly one chunk per direction
        nz = t[g][t[g] > 0]
        assert np.all(nz == 8192 * 4)


# ---------------------------------------------------------- pass byte closed forms --

def _passes(coll, count, dt, A, R, sched=rv.SCHEDULE_RELAY, in_place=False, **kw):
    p = rv.relay_plan(coll, count, dt, A, R, rv.make_opts(schedule=sched, **kw))
    return p, rv.relay_plan_passes(p, in_place)


def test_pass_bytes_a2_allreduce():
    n, E = 1 << 20, 2
    p, ps = _passes(rv.ALLREDUCE, n, rv.BF16, 2, 8)
    cs = p.chunk
    assert [q["name"] for q in ps] == ["group1", "group2", "active_reduce"]
    # group 1: 12 relay chunks to helpers + 2 dirA chunks, each read once, written once
    assert ps[0]["bytes_read"] == ps[0]["bytes_written"] == 14 * cs * E
    # group 2: 6 helpers read 2 slots and write 2 returned chunks; 2 dirB copies
    assert ps[1]["bytes_read"] == ps[1]["bytes_written"] == (12 + 2) * cs * E
    # actives: own + received over dirA+dirB (2 chunks), 2 actives
    assert ps[2]["bytes_read"] == 8 * cs * E and ps[2]["bytes_written"] == 4 * cs * E


def test_pass_bytes_a2_reduce_scatter_and_a4():
    m, E = 1 << 20, 4
    p, ps = _passes(rv.REDUCE_SCATTER, m, rv.F32, 2, 8)
    cs = p.chunk
    assert ps[0]["bytes_read"] == 14 * cs * E
    assert ps[1]["bytes_read"] == 14 * cs * E     # 12 forwarded slots + 2 dirB
    assert ps[2]["bytes_read"] == 2 * 2 * m * E and ps[2]["bytes_written"] == 2 * m * E
    n = 1 << 22
    p, ps = _passes(rv.ALLREDUCE, n, rv.BF16, 4, 8)
    oc, ds, E = p.chunk, p.owner_slice, 2
    assert ps[0]["bytes_read"] == (16 * oc + 12 * ds) * E
    # helpers and owners: 4 sources in, 4 destinations out
    assert ps[1]["bytes_read"] == ps[1]["bytes_written"] == (4 * 4 * oc + 4 * 4 * ds) * E
    p, ps = _passes(rv.REDUCE_SCATTER, n, rv.BF16, 4, 8)
    oc = p.chunk
    assert ps[0]["bytes_read"] - 12 * p.direct_g1 * E == 48 * oc * E   # pack 4x4x3 chunks
    helper = ps[1]["bytes_read"] - 12 * p.direct_g2 * E
    assert helper == 4 * 4 * 3 * oc * E     # 16 reductions of 3 chunks


def test_pass_bytes_all_to_all_pack_unpack():
    seg, E = 120000 * 8, 2
    p, ps = _passes(rv.ALL_TO_ALL, seg, rv.BF16, 4, 8)
    oc = p.chunk
    assert [q["name"] for q in ps] == ["pack", "helper_forward", "unpack"]
    assert ps[2]["bytes_read"] == ps[2]["bytes_written"] == 4 * 4 * 3 * oc * E
    assert ps[0]["bytes_read"] == (4 * 4 * 3 * oc + 12 * p.direct_g1 + 4 * seg) * E


def test_in_place_drops_self_copies():
    p, out_of_place = _passes(rv.ALL_GATHER, 1 << 20, rv.BF16, 4, 8)
    _, in_place = _passes(rv.ALL_GATHER, 1 << 20, rv.BF16, 4, 8, in_place=True)
    assert out_of_place[0]["bytes_read"] - in_place[0]["bytes_read"] == 4 * (1 << 20) * 2


# ----------------------------------------------------------------- size contracts --

def _golden_rows(name):
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if line:
            yield line.split()


def test_passthrough_helper_size_literals():
    # D115998394 / D115998388 hand-computed literals
    for row in _golden_rows("helper_sizes.txt"):
        if row[0] == "total":
            groups, count, A, nc, total = (int(v) for v in row[1:])
            assert groups * rv.relay_passthrough_helper_size(count, A, nc) == total
        else:
            count, A, nc, exp = (int(v) for v in row)
            assert rv.relay_passthrough_helper_size(count, A, nc) == exp


@pytest.mark.parametrize("count", [1024, 65536, 1 << 20, 12_002_982_488 // 64, 777_777])
def test_helper_need_fits_page_contract(orc, count):
    for coll in range(4):
        for A in (2, 4):
            p = rv.relay_plan(coll, count, rv.BF16, A, 8, rv.make_opts(schedule=rv.SCHEDULE_RELAY))
            contract = orc.relay_helper_contract(coll, A, 8, count)
            if A == 4 and coll == rv.ALL_TO_ALL:
                continue   # the page's A=4 all-to-all never relays (size-1 placeholder)
            assert p.helper_elems <= contract, (coll, A, count)
    # item 6: the 4-active reduce-scatter helper needs A*(A-1)*chunk = 1.5x recvCount
    m = 1 << 20
    p = rv.relay_plan(rv.REDUCE_SCATTER, m, rv.BF16, 4, 8, rv.make_opts(schedule=rv.SCHEDULE_RELAY))
    assert p.helper_elems * 2 == 3 * m


# -------------------------------------------------------------------- validation --

def _call(coll, send, recv, scratch, count, dt=rv.F32, A=2, R=8, scale=1.0):
    fn = rv.lib()
    arr = lambda xs: (ctypes.c_void_p * R)(*(xs + [None] * (R - len(xs))))
    if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER):
        f = fn.relay_allreduce if coll == rv.ALLREDUCE else fn.relay_reduce_scatter
        return f(arr(send), arr(recv), arr(scratch), count, dt, A, R, scale, None, None)
    f = fn.relay_all_gather if coll == rv.ALL_GATHER else fn.relay_all_to_all
    return f(arr(send), arr(recv), arr(scratch), count, dt, A, R, None, None)


GB = 1 << 30


def _fake(i):
    return (i + 1) * 64 * GB   # widely spaced, never dereferenced


def test_validation_rejects_before_launch():
    inval = rv.ERR_INVALID_ARGUMENT
    ok_scratch = [_fake(10 + r) for r in range(8)]
    # A and R (D115998382)
    for A, R in [(3, 8), (1, 8), (2, 2), (4, 4), (2, 65)]:
        p = rv.RelayPlan()
        assert rv.lib().relay_plan(0, 1024, 0, A, R, None, ctypes.byref(p)) == inval
    # int32 reductions are SUM only
    assert _call(rv.ALLREDUCE, [_fake(0), _fake(1)], [_fake(2), _fake(3)], ok_scratch, 4096,
                 rv.I32, scale=0.5) == inval
    # NULL active buffers
    assert _call(rv.ALLREDUCE, [_fake(0), None], [_fake(2), _fake(3)], ok_scratch, 4096) == inval
    # overlapping outputs
    assert _call(rv.ALLREDUCE, [_fake(0), _fake(1)], [_fake(2), _fake(2) + 64], ok_scratch,
                 4096) == inval
    # element alignment
    assert _call(rv.ALLREDUCE, [_fake(0) + 2, _fake(1)], [_fake(2), _fake(3)], ok_scratch,
                 4096) == inval
    # all-to-all is out-of-place only (D115998370)
    assert _call(rv.ALL_TO_ALL, [_fake(0), _fake(1)], [_fake(0), _fake(3)], ok_scratch,
                 4096) == inval
    # reduce-scatter in-place must be at the own block offset (D115998376)
    assert _call(rv.REDUCE_SCATTER, [_fake(0), _fake(1)], [_fake(0) + 4, _fake(3)],
                 ok_scratch, 4096) == inval
    # every rejection leaves a message
    assert b"overlap" in rv.lib().relay_last_error() or rv.lib().relay_last_error()


def test_count_zero_is_a_noop():
    for coll in range(4):
        assert _call(coll, [None, None], [None, None], [None] * 8, 0) == rv.OK


def test_missing_scratch_is_rejected():
    opts = rv.make_opts(schedule=rv.SCHEDULE_RELAY)
    arr = lambda xs: (ctypes.c_void_p * 8)(*(xs + [None] * (8 - len(xs))))
    st = rv.lib().relay_allreduce(arr([_fake(0), _fake(1)]), arr([_fake(2), _fake(3)]),
                                  arr([_fake(4), _fake(5)]), 1 << 20, rv.F32, 2, 8, 1.0,
                                  ctypes.byref(opts), None)
    assert st == rv.ERR_INVALID_ARGUMENT
    assert b"helper" in rv.lib().relay_last_error()


def test_legacy_only_at_two_actives():
    with pytest.raises(rv.RelayError):
        rv.relay_plan(rv.ALLREDUCE, 1 << 20, rv.F32, 4, 8, rv.make_opts(schedule=rv.SCHEDULE_LEGACY))
    p = rv.relay_plan(rv.ALLREDUCE, 1 << 20, rv.F32, 2, 8, rv.make_opts(schedule=rv.SCHEDULE_LEGACY))
    assert p.kind == rv.KIND_LEGACY and p.num_groups == 3


def test_pass_names():
    assert [rv.relay_pass_name(k) for k in range(7)] == list(rv.PASS_NAMES)


# ------------------------------------------- bounds and races of every program (dry) --

def _dry(coll, count, dt, A, R, sched, in_place, skew=0):
    """Run a collective in dry-run mode over fake, disjoint buffers of exactly the
    declared sizes: the library builds every pass and checks that each segment stays
    inside a declared buffer and that no launch races with itself; nothing launches."""
    opts = rv.make_opts(schedule=sched, flags=rv.FLAG_CHECK_HAZARDS | rv.FLAG_DRY_RUN)
    p = rv.relay_plan(coll, count, dt, A, R, opts)
    E = rv.ESIZE[dt]
    base = lambda r, k: ((4 * r + k + 1) << 40) + 256 * (r % 3) + skew * ((r + k) % 2)
    send, recv, scratch = [], [], []
    for a in range(A):
        s, r = base(a, 0), base(a, 1)
        if in_place and coll == rv.ALLREDUCE:
            r = s
        elif in_place and coll == rv.REDUCE_SCATTER:
            r = s + a * count * E
        elif in_place and coll == rv.ALL_GATHER:
            s = r + a * count * E
        send.append(s)
        recv.append(r)
    for r_ in range(R):
        scratch.append(base(r_, 2))
    arr = lambda xs: (ctypes.c_void_p * R)(*(xs + [None] * (R - len(xs))))
    L = rv.lib()
    if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER):
        f = L.relay_allreduce if coll == rv.ALLREDUCE else L.relay_reduce_scatter
        scale = 1.0 if dt == rv.I32 else 0.5
        st = f(arr(send), arr(recv), arr(scratch), count, dt, A, R, scale, ctypes.byref(opts), None)
    else:
        f = L.relay_all_gather if coll == rv.ALL_GATHER else L.relay_all_to_all
        st = f(arr(send), arr(recv), arr(scratch), count, dt, A, R, ctypes.byref(opts), None)
    return st


@pytest.mark.parametrize("coll", range(4))
def test_every_program_stays_in_bounds_and_race_free(coll):
    n = 0
    for A in (2, 4):
        for R in (A + 1, 8, 40):
            for dt in (rv.F32, rv.BF16, rv.I32):
                for count in (1, 127, 1024, 1025, 4109, 65536 + 77, 1 << 22, (3 << 20) + 5):
                    for sched in (0, 1, 2, 3):
                        if sched == 3 and A == 4:
                            continue
                        for in_place in (False, True):
                            if in_place and coll == rv.ALL_TO_ALL:
                                continue
                            try:
                                rv.relay_plan(coll, count, dt, A, R, rv.make_opts(schedule=sched))
                            except rv.RelayError:
                                continue
                            for skew in (0, rv.ESIZE[dt]):
                                st = _dry(coll, count, dt, A, R, sched, in_place, skew)
                                assert st == rv.OK, rv.lib().relay_last_error()
                            n += 1
    assert n > 200


# ------------------------------------------------------------ fused multi-group call --

def _dry_multi(coll, counts, dt, A, sched, in_place=False):
    G = len(counts)
    R = G * A
    opts = rv.make_opts(schedule=sched, flags=rv.FLAG_CHECK_HAZARDS | rv.FLAG_DRY_RUN)
    E = rv.ESIZE[dt]
    send, recv = [], []
    for r in range(R):
        s, rr = (r + 1) << 40, ((r + 1) << 40) + (1 << 38)
        if in_place and coll == rv.ALLREDUCE:
            rr = s
        elif in_place and coll == rv.REDUCE_SCATTER:
            rr = s + (r % A) * counts[r // A] * E
        elif in_place and coll == rv.ALL_GATHER:
            s = rr + (r % A) * counts[r // A] * E
        send.append(s)
        recv.append(rr)
    scratch = [((100 + g * R + r) << 40) for g in range(G) for r in range(R)]
    c = (ctypes.c_size_t * G)(*counts)
    arr = lambda xs: (ctypes.c_void_p * len(xs))(*xs)
    scale = 1.0 if dt == rv.I32 else 0.5
    return rv.lib().relay_multi_group(coll, G, c, arr(send), arr(recv), arr(scratch), dt, A, scale,
                                      ctypes.byref(opts), None)


@pytest.mark.parametrize("coll", range(4))
def test_fused_programs_stay_in_bounds_and_race_free(coll):
    mixes = {2: [[65536, 1000, 300_000, 4097], [1 << 20] * 4, [0, 5, 1024, 129]],
             4: [[65536, 3000], [1 << 20, 1 << 20], [0, 70_000]]}
    n = 0
    for A, lists in mixes.items():
        for counts in lists:
            for dt in (rv.F32, rv.BF16, rv.I32):
                for sched in (0, 1, 2):
                    for in_place in (False, True):
                        if in_place and coll == rv.ALL_TO_ALL:
                            continue
                        st = _dry_multi(coll, counts, dt, A, sched, in_place)
                        assert st == rv.OK, rv.lib().relay_last_error()
                        n += 1
    assert n > 50


def test_fused_uniform_relay_puts_one_chunk_on_every_link():
    # 4 groups of 2 on 8 ranks: each rank is active once and a helper 3 times; with the
    # same count everywhere every directed link carries exactly one chunk per phase, so
    # all four allreduces finish in the time of one (cost model, item 1)
    n = 1 << 20
    t = rv.relay_multi_group_link_bytes(rv.ALLREDUCE, [n] * 4, rv.BF16, 2,
                                        rv.make_opts(schedule=rv.SCHEDULE_RELAY))
    cs = n // 8
    assert t.shape == (2, 8, 8)
    for ph in range(2):
        off = t[ph][~np.eye(8, dtype=bool)]
        assert np.all(off == cs * 2)
        assert np.all(np.diag(t[ph]) == 0)


@pytest.mark.parametrize("coll", range(4))
def test_fused_table_is_sum_of_group_tables(orc, coll):
    # the fused table equals each group's oracle table, local ranks renamed to global
    counts, A = [65536, 1000, 300_000, 4097], 2
    if coll in (rv.REDUCE_SCATTER, rv.ALL_TO_ALL):
        counts = [c // 2 for c in counts]
    opts = rv.make_opts(schedule=rv.SCHEDULE_RELAY)
    got = rv.relay_multi_group_link_bytes(coll, counts, rv.F32, A, opts)
    R = len(counts) * A
    exp = np.zeros((3, R, R), np.uint64)
    for g, c in enumerate(counts):
        _, gv = orc.plan(coll, A, R, c, 4, force=rv.SCHEDULE_RELAY)
        t = orc.link_elems(gv).astype(np.uint64) * np.uint64(4)
        m = rv.group_ranks(g, A, R)
        for ph in range(t.shape[0]):
            for s in range(R):
                for d in range(R):
                    exp[ph, m[s], m[d]] += t[ph, s, d]
    assert np.array_equal(got, exp[: got.shape[0]])
    assert not exp[got.shape[0]:].any()


def test_fused_validation():
    arr = lambda xs: (ctypes.c_void_p * len(xs))(*xs)
    c = (ctypes.c_size_t * 1)(1024)
    # a single group is not a fused call
    assert rv.lib().relay_multi_group(0, 1, c, arr([1 << 40, 2 << 40]), arr([3 << 40, 4 << 40]),
                                      arr([None] * 2), 0, 2, 1.0, None, None) == rv.ERR_INVALID_ARGUMENT


def test_flat_pack_validation():
    arr = lambda xs: (ctypes.c_void_p * len(xs))(*xs)
    c = (ctypes.c_size_t * 2)(100, 100)
    # the flat buffer overlaps a tensor
    assert rv.lib().relay_pack_flat(arr([1 << 40, 2 << 40]), c, 2, (1 << 40) + 8, 0, None) \
        == rv.ERR_INVALID_ARGUMENT
    # empty list: nothing to do
    assert rv.lib().relay_pack_flat(arr([None]), c, 0, None, 0, None) == rv.OK


def test_copy_validation():
    L = rv.lib()
    # nothing to copy: no launch, no pointer check
    assert L.relay_copy(None, None, 0, rv.BF16, 0, None) == rv.OK
    assert L.relay_copy(None, 1 << 40, 16, rv.BF16, 0, None) == rv.ERR_INVALID_ARGUMENT
    # a negative CTA cap, an unknown dtype, a misaligned pointer
    assert L.relay_copy(2 << 40, 1 << 40, 16, rv.BF16, -1, None) == rv.ERR_INVALID_ARGUMENT
    assert L.relay_copy(2 << 40, 1 << 40, 16, 7, 0, None) == rv.ERR_INVALID_ARGUMENT
    assert L.relay_copy((2 << 40) + 2, 1 << 40, 16, rv.F32, 0, None) == rv.ERR_INVALID_ARGUMENT
    # overlapping ranges (either way round)
    assert L.relay_copy((1 << 40) + 30, 1 << 40, 16, rv.BF16, 0, None) == rv.ERR_INVALID_ARGUMENT
    assert L.relay_copy(1 << 40, (1 << 40) + 30, 16, rv.BF16, 0, None) == rv.ERR_INVALID_ARGUMENT
    assert "overlap" in L.relay_last_error().decode()


def test_size_queries_and_page_contract(orc):
    for coll in range(4):
        for A in (2, 4):
            for R in (A + 1, 8, 12):
                for count in (0, 100, 1024, 896_000, 12_002_982_488 // 1024, 12_002_982_488):
                    assert rv.relay_helper_contract_size(coll, count, A, R) == \
                        orc.relay_helper_contract(coll, A, R, count)
                    if count < (1 << 31):
                        p = rv.relay_plan(coll, count, rv.BF16, A, R)
                        assert rv.relay_helper_size(p) == p.helper_elems
                        assert rv.relay_active_scratch_size(p) == p.active_scratch_elems
    assert rv.relay_helper_contract_size(0, 10, 3, 8) == -1


def test_oversized_counts_are_rejected():
    p = rv.RelayPlan()
    for coll in range(4):
        assert rv.lib().relay_plan(coll, 1 << 62, 0, 2, 8, None, ctypes.byref(p)) == \
            rv.ERR_INVALID_ARGUMENT
    arr = lambda xs: (ctypes.c_void_p * 8)(*(xs + [None] * (8 - len(xs))))
    st = rv.lib().relay_allreduce(arr([1 << 40, 2 << 40]), arr([3 << 40, 4 << 40]), arr([]),
                                  (1 << 64) - 1, 0, 2, 8, 1.0, None, None)
    assert st == rv.ERR_INVALID_ARGUMENT


def test_wide_partial_plan_links_and_bounds(orc):
    """By default a bf16 4-active reduce-scatter carries each helper partial in fp32: that
    doubles the bytes of each helper -> owner hop and nothing else, and the owner scratch
    grows by H*chunk. RELAY_FLAG_PAYLOAD_PARTIAL restores the one payload-sized chunk.
    Every program stays in bounds and race-free either way."""
    for m in (1 << 20, 250_001, 4096 + 77):
        p = rv.relay_plan(rv.REDUCE_SCATTER, m, rv.BF16, 4, 8, rv.make_opts(schedule=rv.SCHEDULE_RELAY))
        narrow = rv.relay_plan(rv.REDUCE_SCATTER, m, rv.BF16, 4, 8,
                               rv.make_opts(schedule=rv.SCHEDULE_RELAY, flags=rv.FLAG_PAYLOAD_PARTIAL))
        assert p.wide_partial == 1 and narrow.wide_partial == 0
        # fp32 partials take H*chunk more elements plus 128 of slack that lets them start
        # on a 16-byte boundary and keeps the direct slots line-aligned
        assert p.active_scratch_elems == narrow.active_scratch_elems + 4 * p.chunk + 128
        _, gv = orc.plan(rv.REDUCE_SCATTER, 4, 8, m, 2, force=rv.SCHEDULE_RELAY)
        exp = orc.link_elems(gv).astype(np.uint64) * np.uint64(2)
        assert np.array_equal(rv.relay_plan_link_bytes(narrow), exp)
        exp[1, 4:, :4] *= np.uint64(2)            # helpers -> owners in group 2
        assert np.array_equal(rv.relay_plan_link_bytes(p), exp)
        for in_place in (False, True):
            for extra in (0, rv.FLAG_PAYLOAD_PARTIAL):
                for skew in (0, 2, 6, 14):      # bf16 scratch is only 2-byte aligned
                    st = _dry_wide(m, in_place, extra, skew)
                    assert st == rv.OK, rv.lib().relay_last_error()
    # fp32 payloads have nothing to widen
    p = rv.relay_plan(rv.REDUCE_SCATTER, 1 << 20, rv.F32, 4, 8, rv.make_opts(schedule=rv.SCHEDULE_RELAY))
    assert p.wide_partial == 0


def _dry_wide(m, in_place, extra=0, skew=0):
    """Dry run with every buffer `skew` bytes past a 16-byte boundary: the host checks
    (bounds, races, operand alignment: fp32 partials need 4 bytes) must all pass."""
    A, R, E = 4, 8, 2
    opts = rv.make_opts(schedule=rv.SCHEDULE_RELAY,
                        flags=extra | rv.FLAG_CHECK_HAZARDS | rv.FLAG_DRY_RUN)
    send = [((r + 1) << 40) + skew for r in range(A)]
    recv = [s + r * m * E for r, s in enumerate(send)] if in_place else \
        [((r + 10) << 40) + skew for r in range(A)]
    scratch = [((r + 20) << 40) + skew for r in range(R)]
    arr = lambda xs: (ctypes.c_void_p * R)(*(xs + [None] * (R - len(xs))))
    return rv.lib().relay_reduce_scatter(arr(send), arr(recv), arr(scratch), m, rv.BF16, A, R,
                                         0.25, ctypes.byref(opts), None)


# ------------------------------------------------------------- the chained launch --

def _dry_call(coll, count, dt, A, R, sched, in_place, skew, flags=0):
    """A dry run with the host checks on fake, widely spaced buffers `skew` bytes past a
    16-byte boundary; returns (status, launch form)."""
    L = rv.lib()
    E = rv.ESIZE[dt]
    opts = rv.make_opts(schedule=sched, flags=flags | rv.FLAG_CHECK_HAZARDS | rv.FLAG_DRY_RUN)
    send = [((r + 1) << 40) + skew for r in range(A)]
    recv = [((r + 10) << 40) + skew for r in range(A)]
    if in_place and coll == rv.ALLREDUCE:
        recv = send
    elif in_place and coll == rv.REDUCE_SCATTER:
        recv = [s + r * count * E for r, s in enumerate(send)]
    elif in_place and coll == rv.ALL_GATHER:
        send = [y + r * count * E for r, y in enumerate(recv)]
    scratch = [((r + 20) << 40) + skew for r in range(R)]
    arr = lambda xs: (ctypes.c_void_p * R)(*(xs + [None] * (R - len(xs))))
    if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER):
        fn = L.relay_allreduce if coll == rv.ALLREDUCE else L.relay_reduce_scatter
        st = fn(arr(send), arr(recv), arr(scratch), count, dt, A, R,
                1.0 if dt == rv.I32 else 0.5, ctypes.byref(opts), None)
    else:
        fn = L.relay_all_gather if coll == rv.ALL_GATHER else L.relay_all_to_all
        st = fn(arr(send), arr(recv), arr(scratch), count, dt, A, R, ctypes.byref(opts), None)
    return st, rv.last_launch()


def _dropped(how):
    """D of a "chained: G groups, P pieces, D dropped" launch description."""
    m = re.fullmatch(r"chained: (\d+) groups, (\d+) pieces, (\d+) dropped", how)
    assert m, how
    return int(m.group(3))


@pytest.mark.parametrize("coll", range(4))
def test_chained_programs_are_race_free(coll):
    """Every small call, on every schedule, in-place form and buffer skew: the chained
    launch's analysis takes the program (mixed-width fp32 partials included), and its independent
    re-check finds no two CTAs touching the same bytes with one writing, no race inside
    one pass of a group, and no dropped scratch line that anything reads after the drop.
    Relay programs drop their helpers' consumed scratch; RELAY_FLAG_KEEP_SCRATCH drops
    nothing."""
    n = 0
    for A in (2, 4):
        for R in (A + 1, 8):
            for dt in (rv.F32, rv.BF16):
                for count in (1, 127, 1000, 1025, 4109, 65536 + 77, (1 << 20) + 13):
                    for sched in (0, 1, 2, 3):
                        if sched == 3 and A == 4:
                            continue
                        for in_place in (False, True):
                            if in_place and coll == rv.ALL_TO_ALL:
                                continue
                            for skew in (0, rv.ESIZE[dt], 3 * rv.ESIZE[dt]):
                                try:
                                    p = rv.relay_plan(coll, count, dt, A, R, rv.make_opts(schedule=sched))
                                except rv.RelayError:
                                    continue
                                st, how = _dry_call(coll, count, dt, A, R, sched, in_place, skew)
                                assert st == rv.OK, rv.lib().relay_last_error()
                                single = len(rv.relay_plan_passes(p, in_place)) < 2
                                if single:
                                    assert how == "dry run"
                                else:
                                    assert how.startswith("chained"), (coll, A, R, count, sched)
                                    # helpers' scratch is always consumed by a later pass
                                    if p.helper_elems > 0 and count >= 1000:
                                        assert _dropped(how) > 0, how
                                    st, kept = _dry_call(coll, count, dt, A, R, sched, in_place,
                                                         skew, rv.FLAG_KEEP_SCRATCH)
                                    assert st == rv.OK and _dropped(kept) == 0, kept
                                n += 1
    assert n > 500


def test_repeated_calls_reuse_nothing_stale():
    """A call repeated on the same arguments reuses its prepared program; every argument
    that shapes the program keys it. The scale check still runs on a repeat, a call that
    failed validation is never reused, and more distinct calls than the memo holds,
    interleaved, each keep their own program."""
    L = rv.lib()
    R = 8

    def call(A, count, dt, sched, scale, send_base=1, recv_base=10, overlap=False):
        opts = rv.make_opts(schedule=sched, flags=rv.FLAG_DRY_RUN)
        send = [((r + send_base) << 40) for r in range(A)]
        recv = [((r + recv_base) << 40) for r in range(A)]
        if overlap:
            recv[1] = send[0] + 64
        scratch = [((r + 20) << 40) for r in range(R)]
        arr = lambda xs: (ctypes.c_void_p * R)(*(xs + [None] * (R - len(xs))))
        st = L.relay_allreduce(arr(send), arr(recv), arr(scratch), count, dt, A, R, scale,
                               ctypes.byref(opts), None)
        return st, rv.last_launch()

    # int32 takes scale 1 only, on the first call and on a repeat alike
    assert call(2, 65536, rv.I32, rv.SCHEDULE_RELAY, 1.0)[0] == rv.OK
    assert call(2, 65536, rv.I32, rv.SCHEDULE_RELAY, 0.5)[0] == rv.ERR_INVALID_ARGUMENT
    assert call(2, 65536, rv.I32, rv.SCHEDULE_RELAY, 1.0)[0] == rv.OK
    # overlapping buffers fail every time
    for _ in range(3):
        assert call(2, 65536, rv.F32, rv.SCHEDULE_RELAY, 0.5, overlap=True)[0] == rv.ERR_INVALID_ARGUMENT
    # distinct calls, more than the memo holds, interleaved: each gives its own program
    cases = [(A, count, sched) for A in (2, 4) for count in (65536, 4109, 1 << 20)
             for sched in (rv.SCHEDULE_RELAY, rv.SCHEDULE_DIRECT)]
    first = {}
    for rep in range(3):
        for i, (A, count, sched) in enumerate(cases):
            st, how = call(A, count, rv.F32, sched, 1.0 / A, send_base=40 + 4 * i,
                           recv_base=100 + 4 * i)
            assert st == rv.OK, rv.lib().relay_last_error()
            key = (A, count, sched)
            if rep == 0:
                first[key] = how
            assert how == first[key], (key, how, first[key])
    assert len(set(first.values())) > 2


def test_chained_all_gather_shares_its_loads():
    """The 4-active all-gather's chained program merges each active's own copy with the
    copies that scatter the same input bytes to helpers and peers (one load, several
    stores), the second direct part included (it runs in the first one-launch phase):
    24 groups of 40 pieces at R=8, where separate copies would make 28 groups of 44. The
    2-active all-gather's program (18 groups of 30 pieces) is pinned beside it."""
    st, how = _dry_call(rv.ALL_GATHER, 1 << 20, rv.BF16, 4, 8, rv.SCHEDULE_RELAY, False, 0)
    assert st == rv.OK and how.startswith("chained: 24 groups, 40 pieces"), how
    st, how = _dry_call(rv.ALL_GATHER, 1 << 20, rv.BF16, 2, 8, rv.SCHEDULE_RELAY, False, 0)
    assert st == rv.OK and how.startswith("chained: 18 groups, 30 pieces"), how
