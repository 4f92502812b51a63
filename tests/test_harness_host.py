"""The parity harness itself, on the CPU: the full-output checker accepts the oracle's own
results laid out as a call's outputs and rejects a single changed element in any
collective, in any window, including windows that end on a block boundary."""
import numpy as np
import pytest
import torch

import harness as hz
import oracle as orc
import pack_virtual_rank_gb300 as rv
import synth


def _fake_call(coll, A, R, count, dtype, scale):
    c = hz.Call()
    c.coll, c.A, c.R, c.count, c.dtype, c.scale = coll, A, R, count, dtype, scale
    c.in_place, c.bufs = False, []
    hz.read_request(c, rv.SCHEDULE_RELAY, -1, 0)
    n_in = A * count if coll in (rv.REDUCE_SCATTER, rv.ALL_TO_ALL) else count
    c.inputs = [synth.rank_input(41, r, n_in, hz.NAME[dtype]) for r in range(A)]
    c.send = c.inputs
    xs = [hz.host(x) for x in c.inputs]
    outs = []
    for a in range(A):
        if coll == rv.ALLREDUCE:
            q = orc.allreduce(dtype, xs, scale)[2]
        elif coll == rv.REDUCE_SCATTER:
            rs = orc.reduce_scatter_wide if c.wide else orc.reduce_scatter
            q = rs(dtype, xs, count, a, scale, c.span)[2]
        elif coll == rv.ALL_GATHER:
            q = orc.all_gather(xs, count)
        else:
            q = orc.all_to_all(xs, count, a)
        t = torch.from_numpy(q.copy())
        outs.append(t.view(torch.bfloat16) if dtype == rv.BF16 else t)
    c.recv = outs
    return c


CASES = [(rv.ALLREDUCE, 2, rv.BF16, 0.5), (rv.REDUCE_SCATTER, 4, rv.BF16, 0.25),
         (rv.REDUCE_SCATTER, 2, rv.I32, 1.0), (rv.ALL_GATHER, 4, rv.I32, 1.0),
         (rv.ALL_TO_ALL, 4, rv.BF16, 1.0), (rv.ALLREDUCE, 4, rv.F32, 0.25)]


@pytest.mark.parametrize("coll,A,dtype,scale", CASES)
def test_check_full_accepts_oracle_and_rejects_one_flip(monkeypatch, coll, A, dtype, scale):
    monkeypatch.setattr(hz, "FULL_WINDOW", 1000)       # many windows, some ragged
    count = 2 * 1000 + 77
    c = _fake_call(coll, A, 8, count, dtype, scale)
    hz.check_full(c)
    total = hz.out_elems(c)
    for pos in sorted({p for p in (0, 999, 1000, count - 1, count, total - 1) if p < total}):
        for a in (0, A - 1):
            d = _fake_call(coll, A, 8, count, dtype, scale)
            v = d.recv[a].view(torch.int16 if dtype == rv.BF16 else torch.int32)
            v[pos] ^= 1
            with pytest.raises(AssertionError):
                hz.check_full(d)
