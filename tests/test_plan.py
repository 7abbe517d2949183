"""Host tests of the split-count planner (fd_plan): the pages' worked
examples, their policy statements, and plan invariants."""
import os

import pytest
import torch

from split_kv_decode_paged_gb300 import _lib
from split_kv_decode_paged_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name, key):
    out = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].split()
        if line and line[0] == key:
            out.append([int(x) for x in line[1:]])
    return out


def _prob(B, Hq, Hkv, L, D=128, ps=16, dt=torch.bfloat16, kv=None):
    return _lib.make_problem(B, Hq, Hkv, D, ps, (L + ps - 1) // ps + 1, B * ((L + ps - 1) // ps + 1), dt,
                             kv or dt)


@pytest.mark.parametrize("row", _rows("cookbook_split_examples.txt", "example"))
def test_cookbook_split_examples(fdlib, row):
    sms, B, Hq, Hkv, L, margin, lo, hi = row
    plan = _lib.fd_plan(_prob(B, Hq, Hkv, L), [L] * B, num_sms=sms, split_margin_pct=margin)
    splits = (L + plan.chunk_tokens - 1) // plan.chunk_tokens
    assert lo <= splits <= hi, (splits, plan.as_dict())


@pytest.mark.parametrize("row", _rows("cookbook_split_examples.txt", "chunks"))
def test_cookbook_split_ranges(fdlib, row):
    L, S, chunk = row
    plan = _lib.fd_plan(_prob(1, 8, 8, L), [L], num_sms=132, num_splits=S)
    assert plan.chunk_tokens == chunk and plan.num_splits == S


def test_short_sequences_are_not_split(fdlib):
    # lpnh.cn "进阶突破": short sequences are not split, very long ones heavily.
    for L in (1, 64, 300, 512):
        plan = _lib.fd_plan(_prob(1, 32, 8, L), [L], num_sms=148)
        assert plan.num_splits == 1
    splits = []
    for L in (4096, 16384, 131072):
        plan = _lib.fd_plan(_prob(1, 32, 8, L), [L], num_sms=148)
        splits.append((L + plan.chunk_tokens - 1) // plan.chunk_tokens)
    assert splits[0] > 1 and splits[-1] >= splits[0]


def test_long_context_config_split_range(fdlib):
    # The 131072-token single request: roughly 16 to 64 splits on 148 SMs.
    for sms in (148, 152):
        plan = _lib.fd_plan(_prob(1, 32, 8, 131072, ps=64), [131072], num_sms=sms)
        assert 16 <= plan.num_splits <= 64


def test_full_batch_of_equal_lengths_is_not_split(fdlib):
    # "Inference Cookbook" §6.3: no split once batch x heads fills the SMs.
    plan = _lib.fd_plan(_prob(64, 32, 8, 4096), [4096] * 64, num_sms=148, split_margin_pct=18)
    assert plan.num_splits == 1


def test_plan_invariants(fdlib):
    for cfg in (1, 2, 3, 4, 5):
        spec = W.CONFIGS[cfg]
        lens = W.draw_lengths(spec, torch.Generator().manual_seed(W.config_seed(cfg)))
        mb = int((int(lens.max()) + spec.page_size - 1) // spec.page_size)
        prob = _lib.make_problem(spec.B, spec.Hq, spec.Hkv, spec.D, spec.page_size, mb, spec.B * mb,
                                 W._DT[spec.q], W._DT[spec.kv])
        plan = _lib.fd_plan(prob, lens, num_sms=148)
        assert plan.chunk_tokens % plan.tile_tokens == 0
        assert plan.capacity_tokens >= int(lens.max())
        assert 1 <= plan.num_splits <= 512 and plan.grid_ctas <= 148 * max(1, plan.ctas_per_sm)
        assert plan.smem_bytes <= 232448 and 2 <= plan.stages <= 8
        rows = spec.B * spec.Hq
        assert plan.workspace_bytes >= (rows * plan.num_splits * (spec.D + 2) * 4 if plan.num_splits > 1 else 0)
        # headroom for growth widens the capacity
        plan2 = _lib.fd_plan(prob, lens, num_sms=148, max_seq_len=int(lens.max()) + 1000) \
            if int(lens.max()) + 1000 <= spec.page_size * mb else plan
        assert plan2.capacity_tokens >= plan.capacity_tokens


def test_head_subgroups_and_shared_kv(fdlib):
    # groups above 16 heads are sliced into 16-row items
    prob = _lib.make_problem(2, 64, 2, 128, 16, 64, 200, torch.bfloat16, torch.bfloat16)
    plan = _lib.fd_plan(prob, [1000, 1000], num_sms=148, num_splits=1)
    assert plan.head_subgroups == 2 and plan.row_fold == 1 and plan.kv_rows == 2
    assert plan.work_items_hint == 2 * 2 * 2
    # shared KV: 64 q sequences x 4 heads per KV head -> 16 items per (chunk, kvh)
    prob = _lib.make_problem(64, 32, 8, 128, 16, 256, 300, torch.bfloat16, torch.bfloat16)
    plan = _lib.fd_plan(prob, [4096], num_sms=148, shared_kv=1, num_splits=1)
    assert plan.row_fold == 64 and plan.kv_rows == 1 and plan.head_subgroups == 16
    assert plan.work_items_hint == 8 * 16


@pytest.mark.parametrize("kv,ps,B,tile_opt,want_tile,want_stages", [
    (torch.float8_e4m3fn, 128, 256, 0, 256, 3),    # E4M3 default: 256-token stages when they fit
    (torch.float8_e4m3fn, 32, 64, 0, 256, 3),
    (torch.float8_e4m3fn, 16, 256, 0, 128, None),  # 16-token pages: 16 boxes per 256 tokens is too many
    (torch.float8_e4m3fn, 128, 4096, 0, 128, None),  # dispatch tables leave no room for 3 x 256 tokens
    (torch.float8_e4m3fn, 128, 256, 128, 128, None),  # explicit request
    (torch.bfloat16, 128, 256, 256, 128, 3),       # 256-token stages are E4M3 only
    (torch.bfloat16, 16, 1024, 0, 128, 3),
    (torch.bfloat16, 16, 1712, 0, 128, 3),         # the dispatch tables (~6 B per sequence) set
    (torch.bfloat16, 16, 1728, 0, 128, 3),         # where 3 stages stop fitting beside the epilogue
    (torch.bfloat16, 16, 4475, 0, 128, 3),         # scratch (16-bit K/V: then it moves into a
    (torch.bfloat16, 16, 4480, 0, 128, 2),         # stage) and where they stop fitting at all ...
    (torch.float8_e4m3fn, 128, 1712, 0, 256, 3),   # ... and where 256-token E4M3 stages do
    (torch.float8_e4m3fn, 128, 1728, 0, 128, None),
    (torch.bfloat16, 16, 8192, 0, 128, 2),         # the largest batch still plans
])
def test_stage_shape_selection(kv, ps, B, tile_opt, want_tile, want_stages):
    # items of 8000 tokens: long enough that the one-CTA-per-SM shape is kept
    prob = _lib.make_problem(B, 64, 8, 128, ps, 8192 // ps, B * (8192 // ps), torch.bfloat16, kv)
    plan = _lib.fd_plan(prob, [8000] * B, num_sms=152, tile_tokens=tile_opt)
    assert plan.tile_tokens == want_tile
    assert plan.chunk_tokens % plan.tile_tokens == 0
    assert plan.smem_bytes <= 232448
    if want_stages is not None:
        assert plan.stages == want_stages
    # the epilogue scratch moves into a stage only where that buys a stage:
    # 16-bit K/V (1728 <= B <= 4475 here), and E4M3 only on the two-CTA
    # shape with 2 KB boxes (16-token pages)
    if kv == torch.float8_e4m3fn:
        assert plan.scratch_in_stage == (ps == 16 and plan.ctas_per_sm == 2)
    else:
        assert plan.scratch_in_stage == (1728 <= B <= 4475)


@pytest.mark.parametrize("Hq,ps,B,want_tile,want_stages", [
    (128, 128, 64, 256, 2),    # G = 16 (two 8-head tiles): two 256-token stages
    (96, 32, 64, 256, 2),      # G = 12
    (128, 16, 64, 128, 5),     # 16-token pages: 256-token stages need too many boxes
    (64, 128, 64, 256, 3),     # G = 8: three
])
def test_fp8_two_head_tiles_take_two_256_token_stages(Hq, ps, B, want_tile, want_stages):
    prob = _lib.make_problem(B, Hq, 8, 128, ps, 4096 // ps, B * (4096 // ps), torch.bfloat16,
                             torch.float8_e4m3fn)
    plan = _lib.fd_plan(prob, [4000] * B, num_sms=152)
    assert (plan.tile_tokens, plan.stages, plan.ctas_per_sm) == (want_tile, want_stages, 1)
    # an explicit request keeps 128-token stages
    assert _lib.fd_plan(prob, [4000] * B, num_sms=152, tile_tokens=128).tile_tokens == 128


SM_SMEM, RESERVED = 233472, 1024  # GB300 shared memory per SM and reserved per CTA


@pytest.mark.parametrize("kv,ps,B,L,want_two", [
    (torch.bfloat16, 16, 512, 256, True),      # short items: two CTAs per SM, 64-token stages
    (torch.bfloat16, 16, 512, 1024, True),     # 4 KB boxes (16-token pages, D = 128): items
    (torch.bfloat16, 16, 2048, 2048, True),    # of up to 4096 tokens
    (torch.bfloat16, 16, 512, 4096, True),
    (torch.bfloat16, 64, 512, 512, True),      # 16 KB boxes: below 1024 tokens
    (torch.bfloat16, 64, 512, 768, True),
    (torch.bfloat16, 64, 512, 1024, False),    # long enough for the default shape
    (torch.bfloat16, 64, 4480, 1024, True),    # ... unless the default lost a stage to its tables
    (torch.bfloat16, 64, 4480, 2048, False),
    (torch.float8_e4m3fn, 128, 512, 512, True),
    (torch.float8_e4m3fn, 128, 512, 1536, True),
    (torch.float8_e4m3fn, 128, 512, 3072, False),  # 256-token stages win on long items
    (torch.float8_e4m3fn, 128, 2048, 2048, True),   # ... unless the tables took them away
    (torch.float8_e4m3fn, 16, 512, 3072, True),     # 16-token pages: always two CTAs
    (torch.bfloat16, 16, 16, 256, False),      # 128 items cannot fill two CTAs on every SM
])
def test_short_items_take_two_ctas_per_sm(kv, ps, B, L, want_two):
    """The planner's shape for many short work items: two persistent CTAs per
    SM (one streams while the other is between items)."""
    nb = 4096 // ps
    assert L <= nb * ps
    prob = _lib.make_problem(B, 32, 8, 128, ps, nb, B * nb, torch.bfloat16, kv)
    plan = _lib.fd_plan(prob, [L] * B, num_sms=152)
    if want_two:
        # 16-bit K/V: 64-token stages (4 warps); E4M3: 128-token stages (4 warps x 2 sub-tiles)
        want_tile = 128 if kv == torch.float8_e4m3fn else 64
        assert plan.tile_tokens == want_tile and plan.ctas_per_sm == 2 and plan.grid_ctas == 2 * 152
        assert plan.stages >= 2 and plan.smem_bytes <= (SM_SMEM - 2 * RESERVED) // 2
    else:
        assert plan.ctas_per_sm == 1 and plan.grid_ctas <= 152 and plan.tile_tokens >= 128


@pytest.mark.parametrize("B,H,D,L,kv,want_two,want_splits", [
    (1, 32, 128, 4096, torch.float16, True, 8),      # single-sequence MHA: 8 splits of 512
    (1, 32, 128, 2048, torch.float16, True, 8),      # 8 splits of 256
    (1, 32, 64, 8192, torch.float16, True, 9),       # 2 KB boxes: 9 splits of 960
    (1, 32, 128, 16384, torch.float16, False, 4),    # long items, 4 KB boxes: one CTA per SM
    (1, 4, 64, 256, torch.float16, False, 1),        # short sequence: not split
    (1, 32, 128, 1024, torch.float16, False, 4),     # at most 2 x 256 tokens would remain per item
    (1, 32, 128, 4096, torch.float8_e4m3fn, True, 8),  # E4M3: 128-token stages of 4 warps x 2
    (1, 32, 128, 8192, torch.float16, True, 9),      # 320 items on one CTA per SM cannot balance
    (1, 16, 128, 8192, torch.float16, False, 10),    # ... left alone with 431-token items, 4 KB boxes
    (1, 16, 128, 8192, torch.float8_e4m3fn, True, 16),  # ... taken with 2 KB boxes
])
def test_small_grids_take_two_ctas_per_sm(fdlib, B, H, D, L, kv, want_two, want_splits):
    """Fewer work items than SMs: two CTAs per SM with the most splits whose
    items fit the 2 x SM slots, when the items stay short or the boxes small."""
    prob = _prob(B, H, H, L, D=D, dt=torch.bfloat16 if kv == torch.float8_e4m3fn else kv, kv=kv)
    plan = _lib.fd_plan(prob, [L] * B, num_sms=152)
    assert plan.num_splits == want_splits
    if want_two:
        assert plan.ctas_per_sm == 2 and plan.tile_tokens == (128 if kv == torch.float8_e4m3fn else 64)
        assert plan.work_items_hint <= 2 * 152 and plan.chunk_tokens >= 256
    else:
        assert plan.ctas_per_sm == 1


def test_short_items_rule_respects_explicit_options_and_registers(fdlib):
    prob = _lib.make_problem(512, 32, 8, 128, 16, 64, 512 * 64, torch.bfloat16, torch.bfloat16)
    assert _lib.fd_plan(prob, [256] * 512, num_sms=152, tile_tokens=128).tile_tokens == 128
    p1 = _lib.fd_plan(prob, [256] * 512, num_sms=152, ctas_per_sm=1)
    assert p1.grid_ctas <= 152
    # 16 query heads per KV head at D = 128: two 5-warp CTAs do not fit the
    # register file, so the one-CTA shape stays
    prob16 = _lib.make_problem(512, 128, 8, 128, 16, 64, 512 * 64, torch.bfloat16, torch.bfloat16)
    p16 = _lib.fd_plan(prob16, [256] * 512, num_sms=152)
    assert p16.grid_ctas <= 152 and p16.tile_tokens == 128
    # the same at D = 64 does fit
    prob64 = _lib.make_problem(512, 128, 8, 64, 16, 64, 512 * 64, torch.bfloat16, torch.bfloat16)
    assert _lib.fd_plan(prob64, [256] * 512, num_sms=152).grid_ctas == 304
