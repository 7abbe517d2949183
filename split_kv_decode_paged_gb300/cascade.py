"""Cascade (shared-prefix) decode: the tokens every sequence shares are
attended in one pass for all q rows, each sequence's own tokens in another,
and the two normalised states are merged (vLLM's cascade attention, "FlashAttention
與 FlashInfer": a shared prefix is computed once; the merge is the
stage-two rescale formula with d = 1).

All compute runs in libfd.  Prefix pass: fd_decode_paged with a shared_kv
plan -- the prefix is one KV row and the B*G q rows of each KV head are packed
16 to a work item, so each prefix tile read feeds 16 query rows.  Suffix pass:
fd_decode_paged.  Then fd_merge_two.  The prefix must fill whole pages.
"""
from __future__ import annotations

import torch

from . import _lib


class CascadeDecoder:
    """Plans and workspaces for the two passes of a shared-prefix decode."""

    def __init__(self, B, Hq, Hkv, D, page_size, num_pages, prefix_blocks, suffix_max_blocks, prefix_len,
                 suffix_lens_host, q_dtype, kv_dtype, device="cuda", **plan_opts):
        if prefix_len % page_size:
            raise ValueError("the shared prefix must fill whole pages")
        self.B, self.Hq, self.D = B, Hq, D
        self.q_dtype = q_dtype
        self.device = torch.device(device)
        self.prob_p = _lib.make_problem(B, Hq, Hkv, D, page_size, prefix_blocks, num_pages, q_dtype, kv_dtype,
                                        torch.float32)
        self.prob_s = _lib.make_problem(B, Hq, Hkv, D, page_size, suffix_max_blocks, num_pages, q_dtype, kv_dtype,
                                        torch.float32)
        self.plan_p = _lib.fd_plan(self.prob_p, [prefix_len], shared_kv=1, **plan_opts)
        self.plan_s = _lib.fd_plan(self.prob_s, suffix_lens_host, **plan_opts)
        mk = lambda plan: torch.zeros(max(256, plan.workspace_bytes), dtype=torch.uint8, device=self.device)
        self.ws_p, self.ws_s = mk(self.plan_p), mk(self.plan_s)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        f32 = dict(dtype=torch.float32, device=self.device)
        self.out_p, self.lse_p = torch.empty((B, Hq, D), **f32), torch.empty((B, Hq), **f32)
        self.out_s, self.lse_s = torch.empty((B, Hq, D), **f32), torch.empty((B, Hq), **f32)

    def __call__(self, q, k_pages, v_pages, prefix_table, prefix_len_dev, suffix_table, suffix_lens,
                 k_scale=None, v_scale=None, out=None, lse=None, stream=None):
        """prefix_table int32 [1, prefix_blocks]; prefix_len_dev int32 [1];
        suffix_table int32 [B, suffix_max_blocks]; suffix_lens int32 [B]."""
        if out is None:
            out = torch.empty((self.B, self.Hq, self.D), dtype=q.dtype, device=q.device)
        if lse is None:
            lse = torch.empty((self.B, self.Hq), dtype=torch.float32, device=q.device)
        _lib.fd_decode_paged(self.plan_p, q, k_pages, v_pages, k_scale, v_scale, prefix_table, prefix_len_dev,
                             self.out_p, self.lse_p, self.ws_p, self.status, stream)
        _lib.fd_decode_paged(self.plan_s, q, k_pages, v_pages, k_scale, v_scale, suffix_table, suffix_lens,
                             self.out_s, self.lse_s, self.ws_s, self.status, stream)
        _lib.fd_merge_two(self.out_p, self.lse_p, self.out_s, self.lse_s, out, lse, stream)
        return out, lse

    def check(self):
        """Synchronise the device and raise FdError if a kernel reported an error."""
        if self.device.type == "cuda":
            torch.cuda.synchronize(self.device)
        word = int(self.status.item())
        if word:
            self.status.zero_()
            self.ws_p.zero_()
            self.ws_s.zero_()
            if self.device.type == "cuda":
                # finish the clears before a call on another stream runs
                torch.cuda.synchronize(self.device)
            raise _lib.FdError(_lib.fd_status_from_device(word), "device status")
