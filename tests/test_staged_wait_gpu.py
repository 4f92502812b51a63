"""The bounded wait of the TMA-staged kernel, made to run out on purpose without faulting
the GPU: one staged copy whose mbarrier expects more bytes than its bulk copy brings. The
kernel must record the fault, leave its tile unwritten and return; the host reads the
fault through relay_device_status(); the context stays usable for the next call."""
import ctypes

import pytest
import torch

import harness as hz
import pack_virtual_rank_gb300 as rv

pytestmark = pytest.mark.gpu


def test_staged_wait_runs_out_and_is_reported():
    L = rv.lib()
    rv.device_status()                                   # start from a clear fault word
    src = torch.arange(8192, dtype=torch.int32, device="cuda")
    dst = torch.full((4096,), -1, dtype=torch.int32, device="cuda")
    n = 4000
    # an ordinary staged copy from a source 4 bytes off the 16-byte grid
    st = L.relay_test_staged_wait(dst.data_ptr(), src[1:].data_ptr(), n, rv.I32, 0, None)
    assert st == rv.OK, L.relay_last_error()
    torch.cuda.synchronize()
    rv.device_status()
    assert torch.equal(dst[:n].cpu(), src[1:n + 1].cpu())
    # the same copy with 16 bytes more expected than arrive: the wait runs out (200 ms),
    # then once more while the copy is given time to finish, and the CTA leaves
    dst.fill_(-1)
    st = L.relay_test_staged_wait(dst.data_ptr(), src[1:].data_ptr(), n, rv.I32, 16, None)
    assert st == rv.OK, L.relay_last_error()
    torch.cuda.synchronize()
    assert L.relay_device_status() == rv.ERR_CUDA
    assert b"bounded wait" in L.relay_last_error()
    assert bool((dst == -1).all())                     # the tile was left unwritten
    assert L.relay_device_status() == rv.OK            # reading cleared the word
    # the context is still usable: a collective whose closing reduction realigns one of its
    # sources (odd recvCount) runs through the staged kernel
    c = hz.run(rv.REDUCE_SCATTER, 2, 8, 300_001, rv.F32, 0.5, schedule=rv.SCHEDULE_RELAY,
               flags=rv.FLAG_SEPARATE_PASSES)
    hz.check_all(c)


def test_staged_wait_hook_rejects_bad_arguments():
    L = rv.lib()
    x = torch.zeros(16384, dtype=torch.int32, device="cuda")
    assert L.relay_test_staged_wait(x.data_ptr(), x.data_ptr(), 1 << 20, rv.I32, 0, None) == \
        rv.ERR_INVALID_ARGUMENT                        # more than one tile
    assert L.relay_test_staged_wait(x[1:].data_ptr(), x.data_ptr(), 10, rv.I32, 0, None) == \
        rv.ERR_INVALID_ARGUMENT                        # destination off the 16-byte grid
    assert L.relay_test_staged_wait(x.data_ptr(), x.data_ptr(), 10, rv.I32, -1, None) == \
        rv.ERR_INVALID_ARGUMENT
