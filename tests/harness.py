"""Shared pieces of the GPU parity tests: seeded inputs, guarded device buffers, one
call through the C ABI, and the oracle's expected values for any output window.

The oracle is the CPU restatement in ``oracle/``; nothing here computes a result
itself beyond slicing.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle as orc
import pack_virtual_rank_gb300 as rv
import synth

TORCH = {rv.F32: torch.float32, rv.BF16: torch.bfloat16, rv.I32: torch.int32}
NAME = {rv.F32: "f32", rv.BF16: "bf16", rv.I32: "i32"}
GUARD = 256          # elements of canary on each side of every buffer
POISON = 0xA5
CANARY = 0x5A


def host(t: torch.Tensor) -> np.ndarray:
    return synth.to_numpy(t)


class Guarded:
    """A device buffer with canary bands on both sides (stand-in for a sanitizer)."""

    def __init__(self, n: int, dtype: int, device, fill=POISON):
        self.n = n
        self.full = torch.empty(n + 2 * GUARD, dtype=TORCH[dtype], device=device)
        self.full.view(torch.uint8).fill_(CANARY)
        self.view = self.full[GUARD:GUARD + n]
        if n:
            self.view.view(torch.uint8).fill_(fill)

    def guards_intact(self) -> bool:
        b = self.full.view(torch.uint8)
        e = self.full.element_size()
        lo = b[: GUARD * e]
        hi = b[(GUARD + self.n) * e:]
        return bool((lo == CANARY).all().item() and (hi == CANARY).all().item())


def make_inputs(config: int, A: int, numel: int, dtype: int, device, gpu_generator=False):
    """Active inputs: seeded synthetic draws (recipe in synth.py)."""
    if gpu_generator:
        return [synth.rank_input(config, r, numel, NAME[dtype], device=device) for r in range(A)]
    return [synth.rank_input(config, r, numel, NAME[dtype]).to(device) for r in range(A)]


class Call:
    """Everything one collective call touched, kept for checking."""


def run(coll, A, R, count, dtype, scale=1.0, config=0, schedule=rv.SCHEDULE_AUTO,
        in_place=False, permille=-1, device="cuda", gpu_generator=False, check_hazards=True,
        inputs=None, flags=0):
    opts = rv.make_opts(offload_permille=permille, schedule=schedule,
                        flags=flags | (rv.FLAG_CHECK_HAZARDS if check_hazards else 0))
    plan = rv.relay_plan(coll, count, dtype, A, R, opts)
    c = Call()
    c.plan, c.coll, c.A, c.R, c.count, c.dtype, c.scale = plan, coll, A, R, count, dtype, scale
    c.in_place = in_place
    read_request(c, schedule, permille, flags)
    assert_plan_agrees(c)
    xs = inputs if inputs is not None else make_inputs(config, A, plan.input_elems, dtype, device,
                                                       gpu_generator)
    c.inputs = xs
    c.bufs = []
    send, recv = [], []
    for a in range(A):
        if in_place and coll == rv.ALLREDUCE:
            g = Guarded(plan.input_elems, dtype, device)
            g.view.copy_(xs[a])
            send.append(g.view)
            recv.append(g.view)
            c.bufs.append(g)
        elif in_place and coll == rv.REDUCE_SCATTER:
            g = Guarded(plan.input_elems, dtype, device)
            g.view.copy_(xs[a])
            send.append(g.view)
            recv.append(g.view[a * count:(a + 1) * count])
            c.bufs.append(g)
        elif in_place and coll == rv.ALL_GATHER:
            g = Guarded(plan.output_elems, dtype, device)
            g.view[a * count:(a + 1) * count].copy_(xs[a])
            send.append(g.view[a * count:(a + 1) * count])
            recv.append(g.view)
            c.bufs.append(g)
        else:
            gs = Guarded(plan.input_elems, dtype, device)
            gs.view.copy_(xs[a])
            gr = Guarded(plan.output_elems, dtype, device)
            send.append(gs.view)
            recv.append(gr.view)
            c.bufs += [gs, gr]
    scratch = []
    for r in range(R):
        n = plan.active_scratch_elems if r < A else plan.helper_elems
        if n > 0:
            g = Guarded(n, dtype, device)
            c.bufs.append(g)
            scratch.append(g.view)
        else:
            scratch.append(None)
    c.send, c.recv, c.scratch = send, recv, scratch
    fn = rv.COLLECTIVES[coll]
    if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER):
        fn(send + [None] * (R - A), recv + [None] * (R - A), scratch, count, dtype, A, R, scale,
           opts)
    else:
        fn(send + [None] * (R - A), recv + [None] * (R - A), scratch, count, dtype, A, R, opts)
    c.launch = rv.last_launch()
    torch.cuda.synchronize()
    rv.device_status()          # no bounded wait in any kernel gave up
    return c


OCOLL = {rv.ALLREDUCE: orc.AR, rv.REDUCE_SCATTER: orc.RS, rv.ALL_GATHER: orc.AG,
         rv.ALL_TO_ALL: orc.A2A}
OFORCE = {rv.SCHEDULE_AUTO: orc.FORCE_AUTO, rv.SCHEDULE_RELAY: orc.FORCE_RELAY,
          rv.SCHEDULE_DIRECT: orc.FORCE_DIRECT, rv.SCHEDULE_LEGACY: orc.FORCE_LEGACY}


def read_request(c, schedule=rv.SCHEDULE_AUTO, permille=-1, flags=0):
    """What the oracle needs to know about a call, taken from the request and the oracle's
    own plan only (never from the library under test):
      c.oplan -- the oracle's planner restatement of the request;
      c.span  -- positions of each reduce-scatter block reduced at a helper: H * chunk of
                 the 4-active relay reduce-scatter (item 6), 0 otherwise;
      c.wide  -- the 4-active bf16 relay reduce-scatter carries its helper partial in fp32
                 unless the request sets FLAG_PAYLOAD_PARTIAL (the library's documented
                 default); every other call has no partial."""
    pm = 500 if permille < 0 else permille
    c.oplan, _ = orc.plan(OCOLL[c.coll], c.A, c.R, c.count, rv.ESIZE[c.dtype], permille=pm,
                          force=OFORCE[schedule])
    relay_rs4 = (c.coll == rv.REDUCE_SCATTER and c.A > 2 and c.oplan["kind"] == orc.KIND_RELAY)
    c.span = c.oplan["H"] * c.oplan["chunk"] if relay_rs4 else 0
    c.wide = relay_rs4 and c.dtype == rv.BF16 and not (flags & rv.FLAG_PAYLOAD_PARTIAL)
    return c


def assert_plan_agrees(c):
    """The library's plan of the call equals the oracle's restatement (checked on its own,
    apart from the results)."""
    p, g = c.plan, c.oplan
    assert (p.kind, p.num_groups, p.chunk) == (g["kind"], g["groups"], g["chunk"])
    if c.A == 2:
        assert (p.dirA_offset, p.dirA_size, p.dirB_size) == (g["dirA_off"], g["dirA"], g["dirB"])
    else:
        assert (p.direct_total, p.direct_g1, p.direct_g2) == (g["pD"], g["d1"], g["d2"])
        assert (p.owner_slice, p.owner_slice_last) == (g["owner_slice"], g["owner_last"])
    assert p.wide_partial == int(c.wide)


def out_elems(c) -> int:
    """Output elements per active, from the request: A blocks for all-gather and
    all-to-all, one for allreduce and reduce-scatter (D115998376, D115998385, D115998370)."""
    return c.A * c.count if c.coll in (rv.ALL_GATHER, rv.ALL_TO_ALL) else c.count


def helper_span(c) -> int:
    """Positions of each reduce-scatter block reduced at a helper (4-active relay), from
    the oracle's plan."""
    return c.span


def expected(c, xs_host, rank, i0, i1):
    """Oracle values of output window [i0, i1) of active `rank`: (q, ref32, ref64)."""
    d, A, n = c.dtype, c.A, c.count
    if c.coll == rv.ALLREDUCE:
        r64, r32, rq = orc.allreduce(d, xs_host, c.scale, i0, i1)
        return rq, r32, r64
    if c.coll == rv.REDUCE_SCATTER:
        rs = orc.reduce_scatter_wide if c.wide else orc.reduce_scatter
        r64, r32, rq = rs(d, xs_host, n, rank, c.scale, helper_span(c), i0, i1)
        return rq, r32, r64
    if c.coll == rv.ALL_GATHER:
        return orc.all_gather(xs_host, n)[i0:i1], None, None
    return orc.all_to_all(xs_host, n, rank)[i0:i1], None, None


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """One bf16 ulp at the magnitude of fp32 values x (8 significant bits); subnormal
    magnitudes use the smallest normal exponent."""
    ax = np.abs(x.astype(np.float64))
    e = np.floor(np.log2(np.maximum(ax, np.finfo(np.float32).tiny)))
    e = np.maximum(e, -126)
    return np.exp2(e - 7)


def check_window(c, rank, i0, i1, xs_host):
    """Compare output window [i0, i1) of active `rank` with the oracle."""
    _compare_window(c, rank, i0, i1, xs_host, host(c.recv[rank][i0:i1]))


def _compare_window(c, rank, i0, i1, xs_host, got):
    q, r32, r64 = expected(c, xs_host, rank, i0, i1)
    if c.dtype == rv.I32 or r32 is None:
        assert np.array_equal(got, q), _first_diff(got, q, i0)
        return
    # identical arithmetic order as the oracle: bit-exact
    assert np.array_equal(got, q), _first_diff(got, q, i0)
    if c.dtype == rv.F32:
        # fp32 criterion: relative error <= 1e-6 against the fp64-accumulated sum. Two
        # terms round once, so this holds for every element at A=2. With more terms a
        # cancelling sum can defeat any fixed relative bound, so there the bound also
        # admits the recursive-summation error (A-1) * 2^-24 * sum|x|.
        err = np.abs(got.astype(np.float64) - r64)
        if c.A == 2:
            assert np.all(err <= 1e-6 * np.abs(r64)), "fp32 relative error above 1e-6"
        else:
            mag = np.zeros_like(r64)
            for x in xs_host:
                mag += np.abs(_window_terms(c, x, rank, i0, i1).astype(np.float64))
            mag *= abs(c.scale)
            bound = np.maximum(1e-6 * np.abs(r64), (c.A - 1) * 2.0 ** -24 * mag)
            assert np.all(err <= bound), "fp32 tolerance"
    else:
        g = orc.bf16_to_f32(got).astype(np.float64)
        assert np.all(np.abs(g - r32.astype(np.float64)) <= bf16_ulp(r32)), "bf16 1-ulp bound"


def _window_terms(c, x, rank, i0, i1):
    if c.coll == rv.REDUCE_SCATTER:
        base = rank * c.count
        x = x[base + i0: base + i1]
    else:
        x = x[i0:i1]
    return orc.bf16_to_f32(x) if c.dtype == rv.BF16 else x


def _first_diff(got, exp, i0):
    bad = np.nonzero(got != exp)[0]
    if bad.size == 0:
        return "equal"
    k = bad[0]
    return f"{bad.size} mismatches; first at {i0 + k}: got {got[k]!r} expected {exp[k]!r}"


def check_all(c):
    """Full comparison of every active output, inputs unchanged, canaries intact."""
    xs_host = [host(x) for x in c.inputs]
    for a in range(c.A):
        check_window(c, a, 0, out_elems(c), xs_host)
    check_common(c, xs_host)


def check_common(c, xs_host):
    for g in c.bufs:
        assert g.guards_intact(), "a canary band changed: write outside a declared buffer"
    if not c.in_place:
        for a in range(c.A):
            assert np.array_equal(host(c.send[a]), xs_host[a]), "input changed (out-of-place)"


def boundaries(c):
    """Output positions where the schedule switches region: chunk, slice and direct
    boundaries and the ends, for sampled checks of large outputs."""
    g = c.oplan
    total = out_elems(c)
    pts = {0, total}
    n = c.count
    if c.A == 2:
        cs = g["chunk"]
        for h in range(g["H"] + 2):
            pts.add(h * cs)
        pts.update({g["dirA_off"], g["dirA_off"] + g["dirA"], g["dirA_off"] + g["dirA"] + g["dirB"]})
    else:
        oc = g["chunk"]
        for h in range(g["H"] + 1):
            pts.add(h * oc)
        P = g["H"] * oc
        pts.update({P, P + g["d1"], P + g["owner_slice"], P + 2 * g["owner_slice"],
                    P + 3 * g["owner_slice"], n})
    blocks = total // max(n, 1)
    out = set()
    for b in range(max(blocks, 1)):
        for q in pts:
            v = b * n + q if blocks > 1 else q
            if 0 <= v <= total:
                out.add(v)
    return sorted(out)


def check_sampled(c, width=512, seed=0, n_random=8):
    """Windows of `width` around every region boundary plus random windows, split at
    block boundaries. For each window only the input ranges it depends on are fetched,
    laid out as a tiny input whose oracle result is exactly that window."""
    rng = np.random.default_rng(seed)
    total, n = out_elems(c), c.count
    centres = boundaries(c) + [int(v) for v in rng.integers(0, max(total, 1), n_random)]
    for a in range(c.A):
        for ctr in centres:
            i0, i1 = max(0, ctr - width // 2), min(total, ctr + width // 2)
            while i0 < i1:
                k = i0 // n
                j1 = min(i1, (k + 1) * n)
                _check_block_window(c, a, k, i0 - k * n, j1 - k * n)
                i0 = j1


def _check_block_window(c, rank, k, lo, hi):
    """Output positions [k*n + lo, k*n + hi) of active `rank` (block k)."""
    A, n, w, d = c.A, c.count, hi - lo, c.dtype
    got = host(c.recv[rank][k * n + lo: k * n + hi])
    if c.coll == rv.ALLREDUCE:
        tiny = [host(x[lo:hi]) for x in c.inputs]
        exp = orc.allreduce(d, tiny, c.scale)[2]
    elif c.coll == rv.REDUCE_SCATTER:
        tiny = []
        for x in c.inputs:
            t = np.zeros(A * w, dtype=NP[d])
            t[rank * w:(rank + 1) * w] = host(x[rank * n + lo: rank * n + hi])
            tiny.append(t)
        span = max(0, min(helper_span(c) - lo, w))
        rs = orc.reduce_scatter_wide if c.wide else orc.reduce_scatter
        exp = rs(d, tiny, w, rank, c.scale, span)[2]
    elif c.coll == rv.ALL_GATHER:
        tiny = [np.zeros(w, dtype=NP[d]) for _ in range(A)]
        tiny[k] = host(c.inputs[k][lo:hi])
        exp = orc.all_gather(tiny, w)[k * w:(k + 1) * w]
    else:
        tiny = []
        for s in range(A):
            t = np.zeros(A * w, dtype=NP[d])
            if s == k:
                for dd in range(A):
                    t[dd * w:(dd + 1) * w] = host(c.inputs[s][dd * n + lo: dd * n + hi])
            tiny.append(t)
        exp = orc.all_to_all(tiny, w, rank)[k * w:(k + 1) * w]
    assert np.array_equal(got, exp), _first_diff(got, exp, k * n + lo)


NP = {rv.F32: np.float32, rv.BF16: np.uint16, rv.I32: np.int32}


FULL_WINDOW = 1 << 22     # output elements per oracle window of check_full


def _threads():
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:
        return max(1, min(16, os.cpu_count() or 1))


def check_full(c):
    """Every output element of every active compared with the oracle, at any size.

    The outputs and inputs are copied to the host once; the output is cut into windows of
    FULL_WINDOW elements (split at block boundaries) and each window is compared with the
    oracle's result for that window on a pool of host threads (the oracle's C calls release
    the GIL). Allreduce and reduce-scatter windows go through check_window (bit-exact plus
    the stated tolerances); all-gather and all-to-all windows feed the oracle the input
    ranges the window depends on, laid out as a small input whose whole result is that
    window. Canaries and untouched inputs are checked as in check_all."""
    xs_host = [host(x) for x in c.inputs]
    total, n = out_elems(c), c.count
    got = [host(c.recv[a]) for a in range(c.A)]
    windows = []
    i0 = 0
    while i0 < total:
        k = i0 // n if n else 0
        i1 = min(total, i0 + FULL_WINDOW, (k + 1) * n)
        windows.append((k, i0, i1))
        i0 = i1

    def one(w):
        k, lo, hi = w
        if c.coll == rv.ALLREDUCE:
            # every active holds the same result: the oracle's window once, then the
            # other actives bit for bit against the first
            _compare_window(c, 0, lo, hi, xs_host, got[0][lo:hi])
            for a in range(1, c.A):
                assert np.array_equal(got[a][lo:hi], got[0][lo:hi]), _first_diff(
                    got[a][lo:hi], got[0][lo:hi], lo)
            return
        if c.coll == rv.REDUCE_SCATTER:
            for a in range(c.A):
                _compare_window(c, a, lo, hi, xs_host, got[a][lo:hi])
            return
        bl, bh = lo - k * n, hi - k * n
        for a in range(c.A):
            if c.coll == rv.ALL_GATHER:
                exp = orc.all_gather([x[bl:bh] for x in xs_host], bh - bl)[k * (bh - bl):(k + 1) * (bh - bl)]
            else:
                tiny = [np.concatenate([x[dd * n + bl: dd * n + bh] for dd in range(c.A)])
                        for x in xs_host]
                exp = orc.all_to_all(tiny, bh - bl, a)[k * (bh - bl):(k + 1) * (bh - bl)]
            assert np.array_equal(got[a][lo:hi], exp), _first_diff(got[a][lo:hi], exp, lo)

    with cf.ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, windows))
    check_common(c, xs_host)
