"""GPU parity of the fused multi-group call: R/A groups of A consecutive ranks run in
one phase-synchronized call, each rank active in its own group and a helper in the
others, each group on its own schedule. Every group's outputs must equal the oracle's
collective of that group's inputs, bit for bit; canaries must stay intact.

Page: "Link-balance the sharded relay schedules (up to 3.2x vs NCCL)", commits
D115998367 (per-group schedules) and D115998376 (fused multi-group reduce-scatter).
"""
import numpy as np
import pytest
import torch

import harness as hz
import oracle as orc
import pack_virtual_rank_gb300 as rv

pytestmark = pytest.mark.gpu

MIXES = {2: [65536, 1000, 300_000, 4097], 4: [262_144 + 77, 3000]}


@pytest.mark.parametrize("dtype", [rv.F32, rv.BF16, rv.I32])
@pytest.mark.parametrize("A", [2, 4])
@pytest.mark.parametrize("coll", [rv.ALLREDUCE, rv.REDUCE_SCATTER, rv.ALL_GATHER, rv.ALL_TO_ALL])
def test_fused_groups_match_oracle(coll, A, dtype):
    counts = MIXES[A]
    G, R = len(counts), len(counts) * A
    scale = 1.0 if (dtype == rv.I32 or coll in (rv.ALL_GATHER, rv.ALL_TO_ALL)) else 1.0 / A
    for sched in (rv.SCHEDULE_AUTO, rv.SCHEDULE_RELAY):
        opts = rv.make_opts(schedule=sched, flags=rv.FLAG_CHECK_HAZARDS)
        plans = [rv.relay_plan(coll, c, dtype, A, R, opts) for c in counts]
        guards, send, recv, xs = [], [], [], []
        for r in range(R):
            p = plans[r // A]
            x = hz.make_inputs(20 + r, 1, p.input_elems, dtype, "cuda")[0]
            gs, gr = hz.Guarded(p.input_elems, dtype, "cuda"), hz.Guarded(p.output_elems, dtype, "cuda")
            gs.view.copy_(x)
            guards += [gs, gr]
            send.append(gs.view)
            recv.append(gr.view)
            xs.append(hz.host(x))
        scratch = []
        for g in range(G):
            row = [None] * R
            for l, r in enumerate(rv.group_ranks(g, A, R)):
                n = plans[g].active_scratch_elems if l < A else plans[g].helper_elems
                if n > 0:
                    gw = hz.Guarded(n, dtype, "cuda")
                    guards.append(gw)
                    row[r] = gw.view
            scratch.append(row)
        rv.relay_multi_group(coll, counts, send, recv, scratch, dtype, A, scale, opts)
        torch.cuda.synchronize()
        for g in range(G):
            c = hz.Call()
            c.plan, c.coll, c.A, c.R, c.count, c.dtype, c.scale = (plans[g], coll, A, R, counts[g],
                                                                    dtype, scale)
            hz.read_request(c, sched, -1, 0)
            hz.assert_plan_agrees(c)
            gx = [xs[g * A + a] for a in range(A)]
            c.recv = recv[g * A:(g + 1) * A]
            for a in range(A):
                hz.check_window(c, a, 0, hz.out_elems(c), gx)
        for gd in guards:
            assert gd.guards_intact()
        for r in range(R):
            assert np.array_equal(hz.host(send[r]), xs[r])
