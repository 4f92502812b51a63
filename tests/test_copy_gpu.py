"""relay_copy on the GPU: device and host memory on either side, aligned and realigned
offsets, capped and uncapped grids. Every copy must be bit-exact and touch nothing outside
its destination (canary bands around device destinations)."""
import pytest
import torch

import harness as hz
import pack_virtual_rank_gb300 as rv

pytestmark = pytest.mark.gpu

DT = {rv.F32: torch.float32, rv.BF16: torch.bfloat16, rv.I32: torch.int32}


def _src(n, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    if dtype == rv.I32:
        return torch.randint(-2**31, 2**31 - 1, (n,), generator=g, dtype=torch.int64).to(torch.int32)
    return torch.randn(n, generator=g).to(DT[dtype])


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32).cpu()


@pytest.mark.parametrize("dtype", [rv.F32, rv.BF16, rv.I32])
@pytest.mark.parametrize("n", [1, 7, 4096, 8192 + 5, (1 << 20) + 3])
@pytest.mark.parametrize("offs", [(0, 0), (1, 1), (0, 3), (5, 2)])
@pytest.mark.parametrize("max_ctas", [0, 1, 152])
def test_device_to_device(dtype, n, offs, max_ctas):
    so, do = offs
    src_full = _src(n + 16, dtype, seed=n + so).cuda()
    src = src_full[so:so + n]
    g = hz.Guarded(n + 16, dtype, "cuda")
    dst = g.view[do:do + n]
    before = g.view.clone()
    rv.relay_copy(dst, src, max_ctas=max_ctas)
    torch.cuda.synchronize()
    assert torch.equal(_bits(dst), _bits(src))
    # the rest of the guarded buffer and its canaries are untouched
    rest = torch.ones(n + 16, dtype=torch.bool)
    rest[do:do + n] = False
    assert torch.equal(_bits(g.view)[rest], _bits(before)[rest])
    assert g.guards_intact()


@pytest.mark.parametrize("dtype", [rv.BF16, rv.I32])
@pytest.mark.parametrize("n", [3, (1 << 22) + 9])
@pytest.mark.parametrize("offs", [(0, 0), (3, 1)])
@pytest.mark.parametrize("max_ctas", [0, 152])
def test_pinned_host_both_ways(dtype, n, offs, max_ctas):
    so, do = offs
    host = _src(n + 8, dtype, seed=7 * n).pin_memory()
    g = hz.Guarded(n + 8, dtype, "cuda")
    rv.relay_copy(g.view[do:do + n], host[so:so + n], max_ctas=max_ctas)
    back = torch.zeros(n + 8, dtype=DT[dtype]).pin_memory()
    rv.relay_copy(back[so:so + n], g.view[do:do + n], max_ctas=max_ctas)
    torch.cuda.synchronize()
    assert torch.equal(_bits(g.view[do:do + n]), _bits(host[so:so + n]))
    assert torch.equal(_bits(back[so:so + n]), _bits(host[so:so + n]))
    assert not _bits(back[:so]).any() and not _bits(back[so + n:]).any()
    assert g.guards_intact()


def test_pageable_host_where_addressable():
    n = (1 << 20) + 1
    host = _src(n, rv.BF16, seed=11)                # ordinary (pageable) host memory
    out = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    try:
        rv.relay_copy(out, host)
    except rv.RelayError as e:
        # a device that cannot read the host's page tables refuses before any launch
        assert e.status == rv.ERR_UNSUPPORTED
        return
    torch.cuda.synchronize()
    assert torch.equal(_bits(out), _bits(host))


def test_copy_count_zero_and_in_graph():
    src = _src(1 << 16, rv.F32, seed=3).cuda()
    dst = torch.zeros_like(src)
    rv.relay_copy(dst[:0], src[:0])                  # nothing happens
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        rv.relay_copy(dst, src, max_ctas=8, stream=s)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(dst, src)
