"""Device-side wait limits.  Every wait in the decode kernel is bounded: when
one runs out the kernel sets FD_DEV_TIMEOUT in the status word, lets its own
copies in flight land, and returns -- no trap, no hang -- so the context stays
usable.  The plan's test hook makes one side late on purpose (a bounded idle
of the producer warp before its first load, or of the consumer warps before
they release their first stage), longer than a short wait limit, so the other
side's waits run out.  The tests check the flag, that check() raises and
clears the workspace, and that a clean call on the same workspace then
matches the oracle."""
import pytest
import torch

import split_kv_decode_paged_gb300 as fd
from split_kv_decode_paged_gb300 import _lib
from split_kv_decode_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_close, oracle_full

pytestmark = pytest.mark.gpu

LIMIT_US = 200      # wait limit of the stalled call
STALL_US = 20000    # the late side idles 100x longer


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
@pytest.mark.parametrize("role", [1, 2], ids=["late-producer", "slow-consumers"])
def test_wait_timeout_is_flagged_and_recovers(fdlib, role, kv):
    # every item spans more tiles than the pipeline has stages, so the
    # producer fills the ring and then waits on a release that never comes
    spec = W.Spec("timeout", B=3, Hq=16, Hkv=4, D=128, page_size=16 if kv == "bf16" else 128, kv=kv, q="bf16",
                  lens=("list", [3000, 1500, 1100]))
    wl = W.make(spec, 61, "cpu")
    g = wl.to("cuda")
    dec = fd.PagedDecoder.for_pools(g.q, g.k_pages, g.v_pages, g.block_table, wl.seq_lens, num_splits=2,
                                    timeout_us=LIMIT_US, debug_stall_us=STALL_US, debug_stall_role=role)
    assert dec.plan.grid_ctas > 1
    dec(g.q, g.k_pages, g.v_pages, g.block_table, g.seq_lens, g.k_scale, g.v_scale)
    torch.cuda.synchronize()
    assert int(dec.status.item()) & _lib.FD_DEV_TIMEOUT
    with pytest.raises(fd.FdError) as ei:
        dec.check()
    assert ei.value.code == _lib.FD_ERR_TIMEOUT
    assert int(dec.status.item()) == 0 and int(dec.workspace.abs().sum()) == 0

    # a clean plan (same layout, a generous but short limit) on the same
    # workspace and status word
    clean = _lib.fd_plan(dec.problem, wl.seq_lens, num_splits=2, timeout_us=5000)
    assert (clean.workspace_bytes, clean.ws_counters) == (dec.plan.workspace_bytes, dec.plan.ws_counters)
    out = torch.empty_like(g.q)
    lse = torch.empty(g.q.shape[:2], dtype=torch.float32, device="cuda")
    for _ in range(2):
        _lib.fd_decode_paged(clean, g.q, g.k_pages, g.v_pages, g.k_scale, g.v_scale, g.block_table, g.seq_lens, out,
                             lse, dec.workspace, dec.status)
        torch.cuda.synchronize()
        assert int(dec.status.item()) == 0
    ref_o, ref_l = oracle_full(wl)
    assert_close(kv, out, lse, ref_o, ref_l, f"after timeout role={role}")
