"""Every count from 0 to 4096 for the 2-active collectives on the relay schedule (the
zero-chunk fallback below 1024, the relay geometry above), bit-exact against the oracle,
with a poisoned band past each output that must stay untouched. Small calls run as one
chained launch; every 5th count also runs pass by pass, every 7th as one cooperative
launch."""
import numpy as np
import pytest
import torch

import oracle as orc
import pack_virtual_rank_gb300 as rv
import synth

pytestmark = pytest.mark.gpu

A, R, MAXN, BAND = 2, 8, 4096, 64
DT = {rv.F32: torch.float32, rv.BF16: torch.bfloat16, rv.I32: torch.int32}
ODT = {rv.F32: orc.F32, rv.BF16: orc.BF16, rv.I32: orc.I32}
CASES = [(rv.ALLREDUCE, rv.BF16, 0.5), (rv.REDUCE_SCATTER, rv.F32, 0.5),
         (rv.ALL_GATHER, rv.I32, 1.0), (rv.ALL_TO_ALL, rv.BF16, 1.0)]


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).cpu().numpy()


def _expected(coll, d, xs, n, rank, scale):
    if coll == rv.ALLREDUCE:
        return orc.allreduce(ODT[d], xs, scale)[2]
    if coll == rv.REDUCE_SCATTER:
        return orc.reduce_scatter(ODT[d], xs, n, rank, scale)[2]
    if coll == rv.ALL_GATHER:
        return orc.all_gather(xs, n)
    return orc.all_to_all(xs, n, rank)


@pytest.mark.parametrize("coll,dtype,scale", CASES)
def test_every_count_up_to_4096(coll, dtype, scale):
    dev = torch.device("cuda")
    opts = {0: rv.make_opts(schedule=rv.SCHEDULE_RELAY, flags=rv.FLAG_CHECK_HAZARDS),
            1: rv.make_opts(schedule=rv.SCHEDULE_RELAY,
                            flags=rv.FLAG_CHECK_HAZARDS | rv.FLAG_SEPARATE_PASSES),
            2: rv.make_opts(schedule=rv.SCHEDULE_RELAY,
                            flags=rv.FLAG_CHECK_HAZARDS | rv.FLAG_FUSED_PASSES)}
    plans = [rv.relay_plan(coll, n, dtype, A, R, opts[0]) for n in range(MAXN + 1)]
    # every buffer sized for the largest need over all counts (the zero-chunk fallback
    # needs more active scratch than the relay geometry above it)
    cap_in = max(p.input_elems for p in plans)
    cap_out = max(p.output_elems for p in plans)
    cap_act = max(p.active_scratch_elems for p in plans)
    cap_help = max(p.helper_elems for p in plans)
    xs_full = [synth.rank_input(31, r, cap_in, {rv.F32: "f32", rv.BF16: "bf16", rv.I32: "i32"}[dtype])
               for r in range(A)]
    send = [x.to(dev) for x in xs_full]
    recv = [torch.empty(cap_out + BAND, dtype=DT[dtype], device=dev) for _ in range(A)]
    scratch = [torch.empty(max(cap_act if r < A else cap_help, 1), dtype=DT[dtype], device=dev)
               for r in range(R)]
    xs_host = [synth.to_numpy(x) for x in xs_full]
    fn = rv.COLLECTIVES[coll]
    checked = 0
    for n in range(0, MAXN + 1):
        # input and output sizes from the request (D115998376, D115998385, D115998370)
        n_in = A * n if coll in (rv.REDUCE_SCATTER, rv.ALL_TO_ALL) else n
        n_out = A * n if coll in (rv.ALL_GATHER, rv.ALL_TO_ALL) else n
        for policy in (0,) + ((1,) if n % 5 == 0 else ()) + ((2,) if n % 7 == 0 else ()):
            for y in recv:
                y.view(torch.uint8).fill_(0xA5)
            args = ([s[:n_in] for s in send] + [None] * (R - A),
                    [y[:n_out] for y in recv] + [None] * (R - A),
                    scratch, n, dtype, A, R)
            if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER):
                fn(*args, scale, opts[policy])
            else:
                fn(*args, opts[policy])
            torch.cuda.synchronize()
            xs = [x[:n_in] for x in xs_host]
            for a in range(A):
                got = synth.to_numpy(recv[a][:n_out])
                want = _expected(coll, dtype, xs, n, a, scale)
                assert np.array_equal(got.view(np.uint8), want.view(np.uint8)), \
                    f"count {n}, active {a}, policy {policy}"
                tail = _bits(recv[a][n_out:n_out + BAND]).view(np.uint8)
                assert np.all(tail == 0xA5), f"count {n}: bytes past the output were written"
            checked += 1
    assert checked == (MAXN + 1) + (MAXN // 5 + 1) + (MAXN // 7 + 1)
