"""Paged, GQA-shared, split-KV decode attention for GB300 (sm_103a).

The compute lives in libfd.so (CUDA, C ABI in include/fd_api.h); this package
binds it with ctypes and uses PyTorch only for device memory and streams.

    from split_kv_decode_paged_gb300 import PagedDecoder
    dec = PagedDecoder.for_pools(q, k_pages, v_pages, block_table, seq_lens_host)
    out, lse = dec(q, k_pages, v_pages, block_table, seq_lens)
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import (FD_BF16, FD_E4M3, FD_F16, FD_F32, FdError, fd_append_kv, fd_decode_paged, fd_merge_states,
                   fd_plan, fd_status_from_device, fd_status_string, make_problem)

__all__ = ["PagedDecoder", "HostStep", "HostPipeline", "fd_plan", "fd_decode_paged", "fd_merge_states", "fd_append_kv", "fd_status_string",
           "fd_status_from_device", "make_problem", "FdError", "append_kv", "merge_states"]


class PagedDecoder:
    """A plan plus its workspace and device status word.

    The plan is made once from host lengths and reused while every device
    length stays within plan.capacity_tokens (pass max_seq_len to reserve
    room for growth).  Calls on one decoder must not overlap on the GPU."""

    def __init__(self, problem, seq_lens_host, device="cuda", **plan_opts):
        self.problem = problem
        self.plan = fd_plan(problem, seq_lens_host, **plan_opts)
        self.device = torch.device(device)
        nbytes = max(256, int(self.plan.workspace_bytes))
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    @classmethod
    def for_pools(cls, q, k_pages, v_pages, block_table, seq_lens_host, out_dtype=None, **plan_opts):
        """q [B, Hq, D], or [B, q_len, Hq, D] for q_len causal query tokens
        per sequence (the last q_len cached tokens of each)."""
        if q.dim() == 4:
            B, q_len, Hq, D = q.shape
            plan_opts.setdefault("q_len", q_len)
        else:
            B, Hq, D = q.shape
        num_pages, page_size, Hkv, D2 = k_pages.shape
        if D2 != D:
            raise ValueError("head dimension of q and the pools differ")
        prob = make_problem(B, Hq, Hkv, D, page_size, block_table.shape[1], num_pages, q.dtype, k_pages.dtype,
                            out_dtype)
        return cls(prob, seq_lens_host, device=q.device, **plan_opts)

    def __call__(self, q, k_pages, v_pages, block_table, seq_lens, k_scale=None, v_scale=None, out=None,
                 lse=None, want_lse=True, stream=None):
        p, plan = self.problem, self.plan
        lead = (p.B,) if plan.q_len <= 1 else (p.B, plan.q_len)  # p: the caller's problem (B sequences)
        if out is None:
            out = torch.empty(lead + (p.Hq, p.D), dtype=_lib.FD_TO_TORCH[p.out_dtype], device=q.device)
        if lse is None and want_lse:
            lse = torch.empty(lead + (p.Hq,), dtype=torch.float32, device=q.device)
        fd_decode_paged(self.plan, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, out, lse,
                        self.workspace, self.status, stream)
        return out, lse

    def host_step(self):
        """Pinned host and device blocks for step_host (see HostStep)."""
        return HostStep(self)

    def host_pipeline(self, depth=2, direct_out=True):
        """Host steps whose copies overlap other steps' decodes (see HostPipeline)."""
        return HostPipeline(self, depth, direct_out)

    def step_host(self, io, k_pages, v_pages, k_scale=None, v_scale=None, stream=None):
        """One decode step from host memory: io.q, io.block_table and
        io.seq_lens (pinned host views) are copied in with one copy, the
        decode runs, and io.out and io.lse are copied back with one copy.
        Asynchronous: synchronise the stream before reading io.out."""
        _lib.fd_decode_paged_host(self.plan, io.host_in, io.dev_in, k_pages, v_pages, k_scale, v_scale, io.dev_out,
                                  io.host_out, self.workspace, self.status, stream)

    def check(self):
        """Synchronise the decoder's device (calls may run on any stream) and
        raise FdError if the device reported an error."""
        if self.device.type == "cuda":
            torch.cuda.synchronize(self.device)
        word = int(self.status.item())
        if word:
            self.status.zero_()
            self.workspace.zero_()
            if self.device.type == "cuda":
                # the clears are queued on the current stream: finish them
                # before a call on any other stream can touch the workspace
                torch.cuda.synchronize(self.device)
            raise FdError(fd_status_from_device(word), "device status")


class HostPipeline:
    """Decode steps from and to host memory with the input copy of each step
    on a copy stream, where it overlaps the decode of the step before it:
    `depth` sets of HostStep blocks used in turn (fd_host_copy_in on the input
    copy stream, fd_decode_paged_staged on the caller's stream, ordered by
    CUDA events).  direct_out=True: the kernel stores out and lse straight
    into the mapped pinned output block; False: into the device block, and
    fd_host_copy_out on an output copy stream moves them while the next step
    decodes.  Fill io.q / io.block_table / io.seq_lens of `next_io()` before
    `submit()`; read its io.out / io.lse once the step's event `done[i]` has
    completed, and refill it no earlier than that."""

    def __init__(self, dec: PagedDecoder, depth=2, direct_out=True):
        if depth < 1:
            raise ValueError("depth must be at least 1")
        self.dec = dec
        self.direct_out = direct_out
        self.ios = [HostStep(dec) for _ in range(depth)]
        self.in_stream = torch.cuda.Stream(device=dec.device)
        self.out_stream = torch.cuda.Stream(device=dec.device)
        self.copied = [torch.cuda.Event() for _ in range(depth)]
        self.decoded = [None] * depth  # the decode that last read dev_in / wrote dev_out of set i
        self.done = [None] * depth     # set i's last step complete (results in host memory)
        self.k = 0

    def next_io(self):
        """The HostStep blocks the next submit() reads (its earlier step must be done)."""
        return self.ios[self.k % len(self.ios)]

    def submit(self, k_pages, v_pages, k_scale=None, v_scale=None, stream=None):
        """Queue one step on the blocks of next_io(); returns them."""
        i = self.k % len(self.ios)
        io = self.ios[i]
        plan = self.dec.plan
        main = stream if stream is not None else torch.cuda.current_stream(self.dec.device)
        if self.decoded[i] is not None:
            self.in_stream.wait_event(self.decoded[i])  # the decode that last read dev_in
        _lib.fd_host_copy_in(plan, io.host_in, io.dev_in, self.in_stream)
        self.copied[i].record(self.in_stream)
        main.wait_event(self.copied[i])
        if not self.direct_out and self.done[i] is not None:
            main.wait_event(self.done[i])  # the output copy that last read dev_out
        _lib.fd_decode_paged_staged(plan, io.dev_in, k_pages, v_pages, k_scale, v_scale, io.dev_out,
                                    io.host_out if self.direct_out else None, self.dec.workspace,
                                    self.dec.status, main)
        dec_ev = torch.cuda.Event()
        dec_ev.record(main)
        self.decoded[i] = dec_ev
        if self.direct_out:
            self.done[i] = dec_ev
        else:
            self.out_stream.wait_event(dec_ev)
            _lib.fd_host_copy_out(plan, io.dev_out, io.host_out, self.out_stream)
            ev = torch.cuda.Event()
            ev.record(self.out_stream)
            self.done[i] = ev
        self.k += 1
        return io


def append_kv(q_dtype, k_new, v_new, k_pages, v_pages, block_table, seq_lens, k_scale=None, v_scale=None,
              status=None, stream=None):
    """Write k_new/v_new [B, Hkv, D] at position seq_lens[b]; seq_lens is not advanced."""
    B, Hkv, D = k_new.shape
    num_pages, page_size, _, _ = k_pages.shape
    prob = make_problem(B, Hkv, Hkv, D, page_size, block_table.shape[1], num_pages, q_dtype, k_pages.dtype)
    fd_append_kv(prob, k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, status, stream)


def merge_states(o_part, m, d, out_dtype=torch.float32, want_lse=True, stream=None):
    """Merge partial states o_part [B,Hq,S,D], m/d [B,Hq,S] -> (out [B,Hq,D], lse)."""
    B, Hq, S, D = o_part.shape
    out = torch.empty((B, Hq, D), dtype=out_dtype, device=o_part.device)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=o_part.device) if want_lse else None
    fd_merge_states(o_part, m, d, out, lse, stream)
    return out, lse


class HostStep:
    """The host-side blocks of fd_decode_paged_host for one decoder: a pinned
    input block holding q, block_table and seq_lens, a pinned output block
    holding out and lse (typed views of both), and their device twins."""

    def __init__(self, dec: PagedDecoder):
        p, plan = dec.plan.problem, dec.plan  # p.B counts query rows (B * q_len)
        lay = _lib.fd_host_io_layout_for(plan)
        self.layout = lay
        self.host_in = torch.empty(lay.in_bytes, dtype=torch.uint8).pin_memory()
        self.host_out = torch.empty(lay.out_bytes, dtype=torch.uint8).pin_memory()
        self.dev_in = torch.empty(lay.in_bytes, dtype=torch.uint8, device=dec.device)
        self.dev_out = torch.empty(lay.out_bytes, dtype=torch.uint8, device=dec.device)
        qt, ot = _lib.FD_TO_TORCH[p.q_dtype], _lib.FD_TO_TORCH[p.out_dtype]
        kv_rows = plan.kv_rows if plan.kv_rows > 0 else p.B

        def view(buf, off, n, dtype, shape):
            nb = n * torch.empty((), dtype=dtype).element_size()
            return buf[off:off + nb].view(dtype).view(shape)

        lead = (p.B,) if plan.q_len <= 1 else (kv_rows, plan.q_len)
        self.q = view(self.host_in, lay.q_offset, p.B * p.Hq * p.D, qt, lead + (p.Hq, p.D))
        self.block_table = view(self.host_in, lay.block_table_offset, kv_rows * p.max_blocks_per_seq, torch.int32,
                                (kv_rows, p.max_blocks_per_seq))
        self.seq_lens = view(self.host_in, lay.seq_lens_offset, kv_rows, torch.int32, (kv_rows,))
        self.out = view(self.host_out, lay.out_offset, p.B * p.Hq * p.D, ot, lead + (p.Hq, p.D))
        self.lse = view(self.host_out, lay.lse_offset, p.B * p.Hq, torch.float32, lead + (p.Hq,))
