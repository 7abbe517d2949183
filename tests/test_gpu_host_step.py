"""fd_decode_paged_host: one decode step from and to host memory (one packed
input copy, the decode, one packed output copy) gives exactly the results of
fd_decode_paged on device buffers, and matches the oracle."""
import numpy as np
import pytest
import torch

import split_kv_decode_paged_gb300 as fd
from oracle import oracle as orc
from split_kv_decode_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_close, record_errors

pytestmark = pytest.mark.gpu

_CODE = {torch.float16: orc.F16, torch.bfloat16: orc.BF16, torch.float8_e4m3fn: orc.E4M3}

CASES = [
    W.Spec("gqa", B=5, Hq=16, Hkv=4, D=128, page_size=16, kv="bf16", q="bf16", lens=("list", [0, 700, 2100, 33, 4000])),
    W.Spec("fp8", B=3, Hq=16, Hkv=2, D=128, page_size=128, kv="e4m3", q="bf16", lens=("list", [130, 1500, 9000])),
    W.Spec("f16 D64", B=2, Hq=8, Hkv=8, D=64, page_size=64, kv="f16", q="f16", lens=("list", [5000, 64])),
]


@pytest.mark.parametrize("out32", [False, True], ids=["out-native", "out-f32"])
@pytest.mark.parametrize("spec", CASES, ids=[c.name for c in CASES])
def test_host_step_matches_device_call_and_oracle(fdlib, spec, out32):
    wl = W.make(spec, 31, "cpu")
    g = wl.to("cuda")
    dec = fd.PagedDecoder.for_pools(g.q, g.k_pages, g.v_pages, g.block_table, wl.seq_lens,
                                    out_dtype=torch.float32 if out32 else None)
    ref_out, ref_lse = dec(g.q, g.k_pages, g.v_pages, g.block_table, g.seq_lens, g.k_scale, g.v_scale)
    torch.cuda.synchronize()
    dec.check()
    io = dec.host_step()
    io.q.copy_(wl.q)
    io.block_table.copy_(wl.block_table)
    io.seq_lens.copy_(wl.seq_lens)
    io.out.fill_(float("nan"))
    io.lse.fill_(float("nan"))
    for _ in range(2):  # the second step reuses the blocks
        dec.step_host(io, g.k_pages, g.v_pages, g.k_scale, g.v_scale)
        torch.cuda.synchronize()
        dec.check()
        assert torch.equal(io.out.view(torch.uint8), ref_out.cpu().view(torch.uint8))
        assert torch.equal(io.lse.view(torch.int32), ref_lse.cpu().view(torch.int32))
    p = orc.problem(spec.B, spec.Hq, spec.Hkv, spec.D, spec.page_size, wl.max_blocks, wl.num_pages,
                    _CODE[wl.q.dtype], _CODE[wl.k_pages.dtype])
    ro, rl = orc.decode_paged(p, wl.q, wl.k_pages, wl.v_pages, wl.k_scale, wl.v_scale, wl.block_table,
                              wl.seq_lens)
    err_o, err_l = assert_close(spec.kv, io.out, io.lse, ro, rl, f"host step {spec.name}")
    record_errors(f"host step {spec.name}", out_dtype=str(io.out.dtype).replace("torch.", ""),
                  out_max_abs_err=err_o, lse_max_abs_err=err_l)


def test_host_step_pageable_output_block_is_copied(fdlib):
    """An output block in ordinary (pageable) host memory cannot be written by
    the kernel: the call falls back to the device block plus a copy."""
    from split_kv_decode_paged_gb300 import _lib
    spec = CASES[0]
    wl = W.make(spec, 32, "cpu")
    g = wl.to("cuda")
    dec = fd.PagedDecoder.for_pools(g.q, g.k_pages, g.v_pages, g.block_table, wl.seq_lens)
    ref_out, ref_lse = dec(g.q, g.k_pages, g.v_pages, g.block_table, g.seq_lens, g.k_scale, g.v_scale)
    io = dec.host_step()
    io.q.copy_(wl.q)
    io.block_table.copy_(wl.block_table)
    io.seq_lens.copy_(wl.seq_lens)
    pageable = torch.full((io.layout.out_bytes,), 0xFF, dtype=torch.uint8)  # not pinned
    assert not pageable.is_pinned()
    _lib.fd_decode_paged_host(dec.plan, io.host_in, io.dev_in, g.k_pages, g.v_pages, g.k_scale, g.v_scale,
                              io.dev_out, pageable, dec.workspace, dec.status)
    torch.cuda.synchronize()
    dec.check()
    lay = io.layout
    n_out = ref_out.numel() * ref_out.element_size()
    assert torch.equal(pageable[lay.out_offset:lay.out_offset + n_out], ref_out.cpu().view(torch.uint8).flatten())
    n_lse = ref_lse.numel() * 4
    assert torch.equal(pageable[lay.lse_offset:lay.lse_offset + n_lse], ref_lse.cpu().view(torch.uint8).flatten())


@pytest.mark.parametrize("direct_out", [True, False], ids=["mapped-out", "copied-out"])
@pytest.mark.parametrize("depth", [1, 2, 3])
def test_host_pipeline_steps_match_device_calls(fdlib, depth, direct_out):
    """HostPipeline (fd_host_copy_in on a copy stream, fd_decode_paged_staged
    on the caller's stream, fd_host_copy_out on another copy stream unless the
    kernel stores into the mapped block, blocks used in turn): six steps with
    different q rows each give exactly the results of fd_decode_paged on those
    rows."""
    spec = CASES[0]
    wl = W.make(spec, 33, "cpu")
    g = wl.to("cuda")
    dec = fd.PagedDecoder.for_pools(g.q, g.k_pages, g.v_pages, g.block_table, wl.seq_lens)
    gen = torch.Generator().manual_seed(7)
    qs = [torch.randn(wl.q.shape, generator=gen).to(wl.q.dtype) for _ in range(6)]
    refs = []
    for q in qs:
        o, l = dec(q.cuda(), g.k_pages, g.v_pages, g.block_table, g.seq_lens, g.k_scale, g.v_scale)
        refs.append((o.cpu(), l.cpu()))
    torch.cuda.synchronize()
    dec.check()
    pipe = dec.host_pipeline(depth, direct_out)
    for io in pipe.ios:
        io.block_table.copy_(wl.block_table)
        io.seq_lens.copy_(wl.seq_lens)
    pending = []
    for k, q in enumerate(qs):
        io = pipe.next_io()
        slot = k % depth
        if len(pending) == depth:  # the step that used these blocks: check it, then refill
            kk, ev = pending.pop(0)
            ev.synchronize()
            assert torch.equal(io.out.view(torch.uint8), refs[kk][0].view(torch.uint8)), f"step {kk}"
            assert torch.equal(io.lse.view(torch.int32), refs[kk][1].view(torch.int32)), f"step {kk}"
        io.q.copy_(q)
        io.out.fill_(float("nan"))
        pipe.submit(g.k_pages, g.v_pages, g.k_scale, g.v_scale)
        pending.append((k, pipe.done[slot]))
    torch.cuda.synchronize()
    dec.check()
    for kk, _ in pending:
        io = pipe.ios[kk % depth]
        assert torch.equal(io.out.view(torch.uint8), refs[kk][0].view(torch.uint8)), f"step {kk}"
        assert torch.equal(io.lse.view(torch.int32), refs[kk][1].view(torch.int32)), f"step {kk}"
