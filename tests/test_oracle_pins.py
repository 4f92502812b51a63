"""Pins for the CPU oracle: what the page and mathematics fix, independent of the oracle.

Each check is chosen so that a plausible slip inside the oracle (a dropped term, a
wrong index, a transposed operand, a missed rounding, an off-by-one in the geometry)
fails at least one of them.  Page: "Link-balance the sharded relay schedules (up to
3.2x vs NCCL)" -- "item k" of its summary, "Dnnnnnnnnn" a commit of its stack.
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                yield line.split()


def _torch_bf16_bits(f32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- bfloat16 ----

def test_bf16_hand_cases(orc):
    for f_bits, b_bits, *_ in _rows("bf16_rne_cases.txt"):
        f = np.array([int(f_bits, 16)], np.uint32).view(np.float32)
        assert int(orc.bf16_rne(f)[0]) == int(b_bits, 16), f_bits


def test_bf16_matches_library_conversion(orc):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=400_000, dtype=np.uint64).astype(np.uint32)
    # force many exact ties and near-ties
    bits[::3] = (bits[::3] & 0xFFFF0000) | 0x8000
    bits[1::7] = (bits[1::7] & 0xFFFF0000) | 0x7FFF
    f = bits.view(np.float32)
    finite = np.isfinite(f) | np.isinf(f)
    mine = orc.bf16_rne(f)
    lib = _torch_bf16_bits(f.copy())
    assert np.array_equal(mine[finite], lib[finite])
    nan = ~finite
    back = orc.bf16_to_f32(mine[nan])
    assert np.all(np.isnan(back))


# ------------------------------------------------------------- collectives ----

def _inputs(dtype, A, n, seed):
    g = torch.Generator().manual_seed(seed)
    if dtype == 2:
        return [torch.randint(-2 ** 20, 2 ** 20 + 1, (n,), generator=g, dtype=torch.int32)
                for _ in range(A)]
    xs = [torch.randn(n, generator=g) for _ in range(A)]
    return xs if dtype == 0 else [x.to(torch.bfloat16) for x in xs]


def _np(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


@pytest.mark.parametrize("A", [2, 4])
@pytest.mark.parametrize("dtype", [0, 1, 2])
def test_allreduce_matches_library_sum(orc, A, dtype):
    n = 5003
    xs = _inputs(dtype, A, n, 11 + A)
    scale = 1.0 if dtype == 2 else 1.0 / A
    r64, r32, rq = orc.allreduce(dtype, [_np(x) for x in xs], scale)
    if dtype == 2:
        exact = torch.stack([x.long() for x in xs]).sum(0)
        wrapped = ((exact + 2 ** 31) % 2 ** 32 - 2 ** 31).to(torch.int32)
        assert np.array_equal(rq, wrapped.numpy())
        return
    wide = torch.stack([x.double() for x in xs]).sum(0) * scale
    np.testing.assert_allclose(r64, wide.numpy(), rtol=1e-15, atol=0)
    acc = xs[0].float()
    for x in xs[1:]:
        acc = acc + x.float()        # torch elementwise fp32, ascending rank order
    acc = acc * scale
    assert np.array_equal(r32, acc.numpy())
    lib_q = _np(acc.to(torch.bfloat16)) if dtype == 1 else acc.numpy()
    assert np.array_equal(rq, lib_q)


def test_sum_of_negative_zeros_stays_negative(orc):
    # IEEE: -0 + -0 = -0 (round to nearest); a sum seeded with +0 would lose the sign
    nz = [np.array([-0.0, 0.0, -0.0], np.float32) for _ in range(3)]
    nz[1][2] = 0.0
    _, r32, _ = orc.allreduce(0, nz, 1.0)
    assert np.signbit(r32).tolist() == [True, False, False]
    blocks = [np.full(4, -0.0, np.float32) for _ in range(4)]   # A blocks of m = 1
    _, r32, _ = orc.reduce_scatter(0, blocks, 1, 2, 1.0, 1)
    assert np.signbit(r32).tolist() == [True]


def test_allreduce_window_and_int_wrap(orc):
    big = np.array([2 ** 31 - 1, -2 ** 31, 5], np.int32)
    one = np.array([1, -1, 7], np.int32)
    _, _, rq = orc.allreduce(2, [big, one], 1.0)
    assert rq.tolist() == [-2 ** 31, 2 ** 31 - 1, 12]
    xs = [np.arange(10, dtype=np.float32), np.ones(10, np.float32)]
    _, _, rq = orc.allreduce(0, xs, 0.5, 3, 7)
    assert rq.tolist() == [2.0, 2.5, 3.0, 3.5]


@pytest.mark.parametrize("A", [2, 4])
@pytest.mark.parametrize("dtype", [0, 1, 2])
def test_reduce_scatter_is_sliced_allreduce(orc, A, dtype):
    m = 777
    xs = [_np(x) for x in _inputs(dtype, A, A * m, 3 * A + dtype)]
    scale = 1.0 if dtype == 2 else 0.5
    full64, _, fullq = orc.allreduce(dtype, xs, scale)
    for o in range(A):
        r64, _, rq = orc.reduce_scatter(dtype, xs, m, o, scale)
        assert np.array_equal(rq, fullq[o * m:(o + 1) * m])
        if dtype != 2:
            np.testing.assert_array_equal(r64, full64[o * m:(o + 1) * m])


def test_rs4_partial_rounding_hand_case(orc):
    for *xb, scale, relayed, direct in _rows("rs4_partial_rounding.txt"):
        xs = [np.array([int(b, 16)], np.uint16) for b in xb]
        # blocks of m = 1: owner 0 reads position 0 of every input
        _, _, rq_relay = orc.reduce_scatter(1, xs, 1, 0, float(scale), helper_span=1)
        _, _, rq_direct = orc.reduce_scatter(1, xs, 1, 0, float(scale), helper_span=0)
        assert int(rq_relay[0]) == int(relayed, 16)
        assert int(rq_direct[0]) == int(direct, 16)


def test_rs4_wide_partial_hand_case(orc):
    # the fp32 partial 1 + 2^-8 is exact, so the owner's result is the single-rounding
    # one: the golden file's "direct" column
    for *xb, scale, relayed, direct in _rows("rs4_partial_rounding.txt"):
        xs = [np.array([int(b, 16)], np.uint16) for b in xb]
        _, _, rq = orc.reduce_scatter_wide(1, xs, 1, 0, float(scale), helper_span=1)
        assert int(rq[0]) == int(direct, 16)


def test_rs4_wide_partial_is_one_reassociation(orc):
    # fp32: carrying the partial unrounded changes only the association (own + others)
    rng = np.random.default_rng(9)
    m = 500
    xs = [rng.standard_normal(4 * m).astype(np.float32) for _ in range(4)]
    for o in range(4):
        _, r32, _ = orc.reduce_scatter_wide(0, xs, m, o, 0.5, helper_span=m)
        others = [x[o * m:(o + 1) * m] for s, x in enumerate(xs) if s != o]
        part = others[0] + others[1]
        part = part + others[2]
        exp = (xs[o][o * m:(o + 1) * m] + part) * np.float32(0.5)
        assert np.array_equal(r32, exp)
    # bf16, integer-valued inputs: every partial is exact, all three forms agree
    xs = [orc.bf16_rne(rng.integers(-8, 9, 4 * m).astype(np.float32)) for _ in range(4)]
    for o in range(4):
        a = orc.reduce_scatter_wide(1, xs, m, o, 0.25, helper_span=m)[2]
        b = orc.reduce_scatter(1, xs, m, o, 0.25, helper_span=0)[2]
        assert np.array_equal(a, b)


def test_rs4_partial_rounding_is_noop_on_exact_sums(orc):
    # small integers: every partial sum is exact in bf16, so the relayed and the
    # direct reading must agree bit for bit
    rng = np.random.default_rng(5)
    m = 300
    xs = [orc.bf16_rne(rng.integers(-8, 9, 4 * m).astype(np.float32)) for _ in range(4)]
    for o in range(4):
        a = orc.reduce_scatter(1, xs, m, o, 0.25, helper_span=m)[2]
        b = orc.reduce_scatter(1, xs, m, o, 0.25, helper_span=0)[2]
        assert np.array_equal(a, b)


@pytest.mark.parametrize("A", [2, 4])
def test_all_gather_is_concatenation(orc, A):
    S = 301
    xs = [np.random.default_rng(k).standard_normal(S).astype(np.float32) for k in range(A)]
    assert np.array_equal(orc.all_gather(xs, S), np.concatenate(xs))


@pytest.mark.parametrize("A", [2, 4])
@pytest.mark.parametrize("esize", [2, 4])
def test_all_to_all_is_block_transpose_and_involution(orc, A, esize):
    seg = 129
    dt = np.uint16 if esize == 2 else np.int32
    rng = np.random.default_rng(A * esize)
    xs = [rng.integers(0, 2 ** 15, A * seg).astype(dt) for _ in range(A)]
    cube = np.stack(xs).reshape(A, A, seg)            # [src][dst][i]
    outs = [orc.all_to_all(xs, seg, d) for d in range(A)]
    for d in range(A):
        assert np.array_equal(outs[d], cube[:, d, :].reshape(-1))
    back = [orc.all_to_all(outs, seg, d) for d in range(A)]
    for d in range(A):
        assert np.array_equal(back[d], xs[d])


# ---------------------------------------------------------------- planner ----

def _closed(kind):
    for row in _rows("closed_forms.txt"):
        if row[0] == kind:
            yield int(row[1]), dict(kv.split("=") for kv in row[2:])


def test_config_geometry_a2_relay(orc):
    for n, exp in _closed("a2_relay"):
        g, gv = orc.plan(orc.AR, 2, 8, n, 4, force=orc.FORCE_RELAY)
        assert g["kind"] == orc.KIND_RELAY and g["groups"] == 2
        assert g["chunk"] == int(exp["chunk"])
        assert g["dirA"] == int(exp["dirA"]) and g["dirA_off"] == int(exp["dirA_off"])
        assert g["dirB"] == int(exp["dirB"])
        assert orc.cost_elems(gv) == int(exp["cost"])


@pytest.mark.parametrize("n", [1024, 65536, 1 << 20, 7 * 1024 * 13, (1 << 29)])
def test_a2_cost_is_quarter_count(orc, n):
    # item 1: 0.43*count -> 0.25*count, exact whenever numChunks*128 = 1024 divides n
    for coll in range(4):
        g, gv = orc.plan(coll, 2, 8, n, 2, force=orc.FORCE_RELAY)
        assert orc.cost_elems(gv) * 4 == n


def test_a2_every_link_one_chunk_per_direction_per_group(orc):
    n = 1 << 20
    g, gv = orc.plan(orc.AR, 2, 8, n, 2, force=orc.FORCE_RELAY)
    t = orc.link_elems(gv)
    cs = g["chunk"]
    assert t.shape == (2, 8, 8)
    for grp in range(2):
        nz = t[grp][t[grp] > 0]
        assert np.all(nz == cs)            # exactly one chunk on every used link
        for s in range(8):
            for d in range(8):
                if s == d:
                    assert t[grp, s, d] == 0
    # actives -> helpers in G1 only; helpers -> actives in G2 only; direct both
    assert np.all(t[0, :2, 2:] == cs) and np.all(t[1, 2:, :2] == cs)
    assert np.all(t[1, :2, 2:] == 0) and np.all(t[0, 2:, :2] == 0)
    assert t[0, 0, 1] == t[0, 1, 0] == t[1, 0, 1] == t[1, 1, 0] == cs
    # per link direction totals: direct link 0.25*count, relay links count/8
    assert t[:, 0, 1].sum() == n // 4 and t[:, 0, 2].sum() == n // 8


def test_a2_direct_share_is_brute_force_optimum(orc):
    # item 1: balancing egress (2*count - d over 7 links) against the direct link (d)
    n = 65536
    ds = np.arange(0, n + 1, 128)
    cost = np.maximum((2 * n - ds) / 7.0, ds)
    d_star = int(ds[np.argmin(cost)])
    g, _ = orc.plan(orc.AR, 2, 8, n, 4, force=orc.FORCE_RELAY)
    assert g["dirA"] + g["dirB"] == d_star == n // 4


def test_legacy_three_group_cost(orc):
    for n, exp in _closed("a2_legacy"):
        g, gv = orc.plan(orc.AR, 2, 8, n, 4, force=orc.FORCE_LEGACY)
        assert g["groups"] == 3 and orc.cost_elems(gv) == int(exp["cost"])
    # ceilings vs a full exchange (count per link): 2.33x -> 4.0x
    n = 7168 * 64
    _, legacy = orc.plan(orc.AR, 2, 8, n, 4, force=orc.FORCE_LEGACY)
    _, new = orc.plan(orc.AR, 2, 8, n, 4, force=orc.FORCE_RELAY)
    assert n * 3 == orc.cost_elems(legacy) * 7
    assert n == orc.cost_elems(new) * 4


def test_a4_allreduce_critical_path_and_ceilings(orc):
    for n, exp in _closed("a4_ar"):
        g, gv = orc.plan(orc.AR, 4, 8, n, 2, permille=int(exp["permille"]))
        pO = g["H"] * g["chunk"]
        pD = g["pD"]
        assert orc.cost_elems(gv) == int(exp["cost"]) == 2 * max(pD, pO) // 4
        _, direct = orc.plan(orc.AR, 4, 8, n, 2, force=orc.FORCE_DIRECT)
        assert orc.cost_elems(direct) == int(exp["direct_cost"]) == 2 * n // 4
    # 780 permille: 1.28x ceiling; 500: 2.0x
    r780 = 13107200 / 10223616
    assert abs(r780 - 1.28) < 0.005


@pytest.mark.parametrize("permille", range(0, 1001, 100))
def test_a4_allreduce_cost_formula_over_offload(orc, permille):
    n = 5120 * 1024
    g, gv = orc.plan(orc.AR, 4, 8, n, 2, permille=permille, force=orc.FORCE_RELAY)
    pO, pD = g["H"] * g["chunk"], g["pD"]
    assert pO == permille * n // 1000
    assert orc.cost_elems(gv) == 2 * max(pD, pO) // 4


def test_a4_all_gather_split_and_ceiling(orc):
    for S, exp in _closed("a4_ag"):
        g, gv = orc.plan(orc.AG, 4, 8, S, 2, force=orc.FORCE_RELAY)
        assert g["kind"] == orc.KIND_RELAY
        assert g["d1"] == int(exp["d1"]) and g["d2"] == int(exp["d2"])
        assert g["d2"] == 3 * g["d1"]                     # split 1:(A-1)
        assert orc.cost_elems(gv) == int(exp["cost"])
        _, direct = orc.plan(orc.AG, 4, 8, S, 2, force=orc.FORCE_DIRECT)
        assert orc.cost_elems(direct) == int(exp["direct_cost"])


def test_a4_reduce_scatter_helper_need(orc):
    for m, exp in _closed("a4_rs"):
        g, gv = orc.plan(orc.RS, 4, 8, m, 2, force=orc.FORCE_RELAY)
        need = 4 * 3 * g["chunk"]
        assert g["chunk"] == int(exp["chunk"])
        assert need == int(exp["helper_need"]) == 3 * m // 2      # 1.5x recvCount
        assert orc.relay_helper_contract(orc.RS, 4, 8, m) == int(exp["contract"]) == 2 * m
        _, direct = orc.plan(orc.RS, 4, 8, m, 2, force=orc.FORCE_DIRECT)
        assert orc.cost_elems(gv) * 2 == orc.cost_elems(direct) == m


def test_a4_all_to_all_link_model_promise(orc):
    for seg, exp in _closed("a4_a2a"):
        g, gv = orc.plan(orc.A2A, 4, 8, seg, 2, force=orc.FORCE_RELAY)
        assert g["chunk"] == int(exp["chunk"])
        assert orc.cost_elems(gv) == int(exp["cost"])
        _, direct = orc.plan(orc.A2A, 4, 8, seg, 2, force=orc.FORCE_DIRECT)
        assert orc.cost_elems(direct) == int(exp["direct_cost"])
        assert abs(int(exp["direct_cost"]) / int(exp["cost"]) - 1.67) < 0.005


def test_helper_size_literals(orc):
    for row in _rows("helper_sizes.txt"):
        if row[0] == "total":
            groups, count, A, nc, total = (int(v) for v in row[1:])
            assert groups * orc.passthrough_helper_size(count, A, nc) == total
        else:
            count, A, nc, exp = (int(v) for v in row)
            assert orc.passthrough_helper_size(count, A, nc) == exp


def test_helper_size_clamp_and_whole_chunks(orc):
    # min() binds only when A >= num_chunks (D115998388)
    assert orc.passthrough_helper_size(1000, 4, 3) == 1000
    for count in [10 ** 6 + 17, 123_456_789, 12_002_982_488]:
        for A, nc in [(2, 7), (4, 5)]:
            s = orc.passthrough_helper_size(count, A, nc)
            assert s % A == 0 and (s // A) % 128 == 0


def test_minimum_sizes(orc):
    # the old A=2 relay (numChunks = 7) needs recvCount >= 896, i.e. 1792 input
    # elements for the 2-block reduce-scatter; the new geometry needs n >= 1024
    assert orc.align_down(895 // 7) == 0 and orc.align_down(896 // 7) == 128
    g, _ = orc.plan(orc.RS, 2, 8, 1023, 4, force=orc.FORCE_RELAY)
    assert g["kind"] == orc.KIND_ZERO_CHUNK
    g, _ = orc.plan(orc.RS, 2, 8, 1024, 4, force=orc.FORCE_RELAY)
    assert g["kind"] == orc.KIND_RELAY and g["chunk"] == 128


@pytest.mark.parametrize("n", [1, 2, 3, 511, 1023])
def test_zero_chunk_fallback(orc, n):
    # D115998367: dirA takes half, dirB absorbs the remainder; no helper traffic
    for coll in range(4):
        g, gv = orc.plan(coll, 2, 8, n, 2, force=orc.FORCE_RELAY)
        assert g["kind"] == orc.KIND_ZERO_CHUNK
        assert g["dirA"] == n // 2 and g["dirB"] == n - n // 2 and g["dirA_off"] == 0
        t = orc.link_elems(gv)
        assert t[:, 2:, :].sum() == 0 and t[:, :, 2:].sum() == 0
        assert orc.cost_elems(gv) == n


def test_default_crossovers(orc):
    MB = 1 << 20
    # item 7: reduce-scatter A=2 fused relays from 2 MB (fp32 input = 2*m*4 bytes)
    assert orc.plan(orc.RS, 2, 8, MB // 4, 4)[0]["kind"] == orc.KIND_RELAY
    assert orc.plan(orc.RS, 2, 8, MB // 8, 4)[0]["kind"] == orc.KIND_DIRECT
    # item 7: A=4 reduce-scatter offload only past 48 MB (bf16, input = 4*m*2)
    assert orc.plan(orc.RS, 4, 8, 48 * MB // 8, 2)[0]["kind"] == orc.KIND_DIRECT
    assert orc.plan(orc.RS, 4, 8, 64 * MB // 8, 2)[0]["kind"] == orc.KIND_RELAY
    # item 7: A=4 all-gather past 12 MB
    assert orc.plan(orc.AG, 4, 8, 12 * MB // 2, 2)[0]["kind"] == orc.KIND_DIRECT
    assert orc.plan(orc.AG, 4, 8, 27 * MB // 4, 2)[0]["kind"] == orc.KIND_RELAY
    # item 4: A=4 allreduce 2 MB pure-direct floor
    assert orc.plan(orc.AR, 4, 8, MB // 2, 2)[0]["kind"] == orc.KIND_DIRECT
    assert orc.plan(orc.AR, 4, 8, MB, 2)[0]["kind"] == orc.KIND_RELAY
    # item 3: A=2 allreduce small messages take one full exchange (one group)
    g = orc.plan(orc.AR, 2, 8, 32 * 1024, 2)[0]
    assert g["kind"] == orc.KIND_DIRECT and g["groups"] == 1


# ----------------------------------------------- per-entry tables and contracts ----

_COLL = {"ar": 0, "rs": 1, "ag": 2, "a2a": 3}


def _expand(rows, A, R, G):
    """The golden link table: every (group, sender, receiver) entry the rows name."""
    t = np.zeros((G, R, R), np.uint64)

    def ranks(spec):
        if spec == "A":
            return range(A)
        if spec == "H":
            return range(A, R)
        return [int(spec)]
    for grp, src, dst, v in rows:
        for s in ranks(src):
            for d in ranks(dst):
                if s != d:
                    t[int(grp) - 1, s, d] = int(v)
    return t


@pytest.mark.parametrize("coll", ["ar", "rs", "ag", "a2a"])
def test_a4_link_table_every_entry(orc, coll):
    # items 4-7: every entry of each group's table, including those below the group's
    # maximum, worked by hand at one count on a 7-rank node (3 helpers)
    rows = [r[1:] for r in _rows("link_tables.txt") if r[0] == coll]
    _, gv = orc.plan(_COLL[coll], 4, 7, 3_000_000, 2, permille=500, force=orc.FORCE_RELAY)
    got = orc.link_elems(gv)
    exp = _expand(rows, 4, 7, 2)
    assert got.shape == exp.shape
    assert np.array_equal(got, exp), np.argwhere(got != exp)[:5]


def test_helper_contract_literals(orc):
    # every branch of the contract: A=2 with num_chunks = (R-A)+1, and the four 4-active
    # collectives, against values worked by hand
    n = 0
    for coll, A, R, count, exp in _rows("helper_contracts.txt"):
        assert orc.relay_helper_contract(_COLL[coll], int(A), int(R), int(count)) == int(exp), \
            (coll, A, R, count)
        n += 1
    assert n == 11
