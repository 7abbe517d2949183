"""fd_decode_paged_noalloc: the decode entry point that takes no workspace.

It is for callers that cannot allocate device memory where they call the
library (an engine or plugin interface that owns all device allocations,
loops that must not take cudaMalloc's synchronisation, C callers without an
allocator).  Its workspace is a fixed buffer inside libfd.  These tests call
it through the C ABI, twice in a row on the same buffer, and compare with the
workspace-taking fd_decode_paged on the same plan and inputs, within the
parity tolerance the other tests use.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import split_kv_decode_paged_gb300 as fd
from split_kv_decode_paged_gb300 import _lib
from split_kv_decode_paged_gb300 import workloads as W
from tests.gpu_helpers import TOL_OUT, TOL_LSE, half_ulp

pytestmark = pytest.mark.gpu

NOALLOC_MAX = 16 * 1024 * 1024  # FD_NOALLOC_SCRATCH_BYTES in include/fd_api.h


def _noalloc_fn(lib):
    f = lib.fd_decode_paged_noalloc
    P = ctypes.c_void_p
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(_lib.FdPlan), P, P, P, P, P, P, P, P, P, P, P]
    return f


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _close(kv, got, ref_out, got_lse, ref_lse):
    a = got.double().cpu().numpy()
    b = ref_out.double().cpu().numpy()
    assert np.isfinite(a).all()
    assert (np.abs(a - b) <= TOL_OUT[kv] + half_ulp(b, got.dtype)).all()
    la, lb = got_lse.double().cpu().numpy(), ref_lse.double().cpu().numpy()
    same_inf = np.isneginf(la) & np.isneginf(lb)
    assert (np.abs(np.where(same_inf, 0.0, la - np.where(same_inf, 0.0, lb))) <= TOL_LSE[kv]).all()


CASES = [
    ("single-sequence MHA, split", W.CONFIGS[2], {}),
    ("GQA bf16, forced 3 splits, ragged", W.Spec("gqa", B=3, Hq=16, Hkv=4, D=128, page_size=16, kv="bf16",
                                                 q="bf16", lens=("list", [0, 700, 2100])), {"num_splits": 3}),
    ("FP8 pages, 2 splits", W.Spec("fp8", B=2, Hq=16, Hkv=2, D=128, page_size=128, kv="e4m3", q="bf16",
                                   lens=("list", [130, 1500])), {"num_splits": 2}),
]


@pytest.mark.parametrize("name,spec,opts", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_workspace_entry_point(fdlib, name, spec, opts):
    wl = W.make(spec, 21, "cuda")
    dec = fd.PagedDecoder.for_pools(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens.cpu(), **opts)
    assert dec.plan.workspace_bytes <= NOALLOC_MAX
    ref_out, ref_lse = dec(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens, wl.k_scale, wl.v_scale)
    torch.cuda.synchronize()
    dec.check()

    f = _noalloc_fn(fdlib)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):  # the second call reuses the buffer the first one left behind
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        rc = f(ctypes.byref(dec.plan), _p(wl.q), _p(wl.k_pages), _p(wl.v_pages), _p(wl.k_scale),
               _p(wl.v_scale), _p(wl.block_table), _p(wl.seq_lens), _p(out), _p(lse), _p(status), stream)
        assert rc == _lib.FD_OK, _lib.fd_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _close(spec.kv, out, ref_out, lse, ref_lse)
        # same kernel on the same plan: the results are also bit-identical
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def _spec(B, Hq, Hkv, lens, kv="bf16", ps=16):
    return W.Spec("alt", B=B, Hq=Hq, Hkv=Hkv, D=128, page_size=ps, kv=kv, q=kv if kv != "e4m3" else "bf16",
                  lens=("list", lens))


def test_noalloc_alternating_plans_reuse_the_buffer(fdlib):
    """Two plans with different workspace layouts take turns on the shared
    buffer.  Plan A (fused merge, 3 splits) has its counters inside the bytes
    where plan B leaves the partial output of a split row, so an A call after
    a B call finds B's floats where its counters must read zero: each call
    has to clear them itself.  Plan B merges in a separate kernel
    (fuse_merge = 0), which reads its partial states back from the shared
    buffer after A's calls have overwritten the start of it.  Each call is
    checked bit for bit against fd_decode_paged with a workspace of its own
    on the same plan (same kernel, same plan: identical results)."""
    lens_b = [300, 1700, 0, 520, 1999, 999, 2048, 640]
    wa = W.make(_spec(3, 16, 4, [900, 2600, 77]), 41, "cuda")
    wb = W.make(_spec(8, 8, 2, lens_b), 42, "cuda")
    da = fd.PagedDecoder.for_pools(wa.q, wa.k_pages, wa.v_pages, wa.block_table, wa.seq_lens.cpu(), num_splits=3)
    db = fd.PagedDecoder.for_pools(wb.q, wb.k_pages, wb.v_pages, wb.block_table, wb.seq_lens.cpu(), num_splits=4,
                                   fuse_merge=0)
    pa, pb = da.plan, db.plan
    assert pa.num_splits == 3 and pb.num_splits == 4 and pb.fuse_merge == 0
    # A's counters lie inside B's partial outputs, in the row of a sequence
    # that B splits (so B writes those bytes on every call)
    row_bytes = pb.num_splits * 128 * 4
    assert pb.ws_partial_o <= pa.ws_counters and pa.workspace_bytes <= pb.ws_partial_md
    rows = range((pa.ws_counters - pb.ws_partial_o) // row_bytes,
                 (pa.workspace_bytes - pb.ws_partial_o + row_bytes - 1) // row_bytes)
    assert all(lens_b[r // 8] > pb.chunk_tokens for r in rows)
    assert max(pa.workspace_bytes, pb.workspace_bytes) <= NOALLOC_MAX
    refs = {}
    for key, dec, wl in (("a", da, wa), ("b", db, wb)):
        refs[key] = dec(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    da.check()
    db.check()
    f = _noalloc_fn(fdlib)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for key in ("a", "b", "a", "b", "b", "a"):
        dec, wl = (da, wa) if key == "a" else (db, wb)
        ref_out, ref_lse = refs[key]
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        rc = f(ctypes.byref(dec.plan), _p(wl.q), _p(wl.k_pages), _p(wl.v_pages), None, None, _p(wl.block_table),
               _p(wl.seq_lens), _p(out), _p(lse), _p(status), stream)
        assert rc == _lib.FD_OK, _lib.fd_status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), key


def test_noalloc_rejects_plans_beyond_its_buffer(fdlib):
    # 256 sequences x 64 heads of 32768-token capacity in 64 splits need far
    # more partial-state room than the built-in buffer holds.
    prob = _lib.make_problem(256, 64, 8, 128, 128, 256, 40000, torch.bfloat16, torch.float8_e4m3fn)
    plan = _lib.fd_plan(prob, [32768] * 256, num_splits=64, num_sms=148)
    assert plan.workspace_bytes > NOALLOC_MAX
    f = _noalloc_fn(fdlib)
    fake = ctypes.c_void_p(1 << 20)  # never touched: the size check comes first
    rc = f(ctypes.byref(plan), fake, fake, fake, fake, fake, fake, fake, fake, None, None, None)
    assert rc == _lib.FD_ERR_WORKSPACE_TOO_SMALL
