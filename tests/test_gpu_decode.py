"""GPU parity tests: the CUDA decode path (through the C ABI) against the fp64
oracle on the same seeded inputs, plus bit-exact paging and device-error
reporting.  Bars: out max-abs <= 2e-3 and lse <= 1e-3 for f16/bf16 K/V,
out <= 3e-2 for E4M3 K/V (oracle on the dequantised stored values), plus half
an output ulp when the output is f16/bf16.  The five benchmark workloads are
checked row by row in test_gpu_configs.py."""
import numpy as np
import pytest
import torch

import split_kv_decode_paged_gb300 as fd
from split_kv_decode_paged_gb300 import _lib
from split_kv_decode_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_close, gpu_decode, oracle_full

pytestmark = pytest.mark.gpu


def _spec(name, B, Hq, Hkv, D, ps, kv, q, lens, pool=("factor", 1.5), k_mult=1.0, extra_blocks=0):
    return W.Spec(name, B=B, Hq=Hq, Hkv=Hkv, D=D, page_size=ps, kv=kv, q=q, lens=("list", list(lens)),
                  pool=pool, k_mult=k_mult, extra_blocks=extra_blocks)


def _run_and_check(spec, seed, out_dtype=None, **plan_opts):
    wl = W.make(spec, seed, "cpu")
    out, lse, dec = gpu_decode(wl.to("cuda"), out_dtype=out_dtype, **plan_opts)
    ref_o, ref_l = oracle_full(wl)
    err = assert_close(spec.kv, out, lse, ref_o, ref_l, what=f"{spec.name} {plan_opts}")
    return err, dec


@pytest.mark.parametrize("fuse", [1, 0])
@pytest.mark.parametrize("splits", [1, 2, 3, 4, 7])
def test_tiny_mha_forced_splits(fdlib, splits, fuse):
    spec = W.CONFIGS[1]
    wl = W.make_config(1, "cpu")
    out, lse, dec = gpu_decode(wl.to("cuda"), num_splits=splits, fuse_merge=fuse)
    ref_o, ref_l = oracle_full(wl)
    assert_close(spec.kv, out, lse, ref_o, ref_l, what=f"cfg1 S={splits}")


SMALL = [
    # name, B, Hq, Hkv, D, ps, kv, q, lens
    ("mha f16 d64", 2, 4, 4, 64, 16, "f16", "f16", [1, 200]),
    ("gqa bf16 g4", 3, 16, 4, 128, 16, "bf16", "bf16", [64, 65, 1000]),
    ("gqa bf16 g8 ps32", 2, 16, 2, 128, 32, "bf16", "bf16", [33, 777]),
    ("gqa f16 g2 ps48", 2, 8, 4, 128, 48, "f16", "f16", [47, 500]),
    ("gqa bf16 g16", 2, 32, 2, 128, 16, "bf16", "bf16", [100, 300]),
    ("gqa bf16 g3", 2, 6, 2, 64, 64, "bf16", "bf16", [5, 129]),
    ("fp8 bf16q g8 ps128", 3, 16, 2, 128, 128, "e4m3", "bf16", [16, 130, 1500]),
    ("fp8 f16q g4 ps16", 2, 8, 2, 128, 16, "e4m3", "f16", [31, 400]),
    ("fp8 bf16q d64 g1", 2, 2, 2, 64, 64, "e4m3", "bf16", [70, 9]),
    ("fp8 bf16q g16", 1, 32, 2, 128, 128, "e4m3", "bf16", [700]),
    ("empty and one token", 3, 8, 2, 128, 16, "bf16", "bf16", [0, 1, 17]),
    ("gqa bf16 g20 (two head sub-groups)", 2, 40, 2, 128, 16, "bf16", "bf16", [90, 700]),
    ("gqa bf16 g32", 2, 64, 2, 128, 64, "bf16", "bf16", [300, 1200]),
    ("mqa f16 g48 d64", 1, 48, 1, 64, 16, "f16", "f16", [517]),
    ("fp8 g32", 2, 64, 2, 128, 128, "e4m3", "bf16", [200, 900]),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("out32", [False, True], ids=["out-native", "out-f32"])
def test_small_shapes(fdlib, case, splits, out32):
    spec = _spec(*case)
    _run_and_check(spec, seed=7 + splits, out_dtype=torch.float32 if out32 else None, num_splits=splits)


@pytest.mark.parametrize("kv,q", [("bf16", "bf16"), ("f16", "f16"), ("e4m3", "bf16")])
def test_fp32_output(fdlib, kv, q):
    spec = _spec("f32 out", 2, 8, 2, 128, 16, kv, q, [90, 333])
    _run_and_check(spec, seed=3, out_dtype=torch.float32, num_splits=2)


def test_paged_equals_contiguous_bitexact(fdlib):
    """Same tokens laid out under a random page permutation and under an
    identity table give bit-identical GPU results for the same plan."""
    spec = _spec("perm", 3, 16, 4, 128, 16, "bf16", "bf16", [100, 1000, 2500])
    wl = W.make(spec, 11, "cpu")
    ps = spec.page_size
    lens = wl.seq_lens.tolist()
    npg = [(L + ps - 1) // ps for L in lens]
    total = sum(npg)
    kc = torch.empty((total,) + tuple(wl.k_pages.shape[1:]), dtype=wl.k_pages.dtype)
    vc = torch.empty_like(kc)
    bt2 = torch.full_like(wl.block_table, -1)
    cur = 0
    for b, n in enumerate(npg):
        for j in range(n):
            src = int(wl.block_table[b, j])
            kc[cur] = wl.k_pages[src]
            vc[cur] = wl.v_pages[src]
            bt2[b, j] = cur
            cur += 1
    wl2 = W.Workload(spec, wl.q, kc, vc, None, None, bt2, wl.seq_lens, total)
    for splits in (1, 3):
        o1, l1, _ = gpu_decode(wl.to("cuda"), num_splits=splits, num_sms=148)
        o2, l2, _ = gpu_decode(wl2.to("cuda"), num_splits=splits, num_sms=148)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_workspace_counters_return_to_zero(fdlib):
    wl = W.make_config(4, "cuda")
    dec = fd.PagedDecoder.for_pools(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens.cpu())
    for _ in range(3):
        dec(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    ctr = dec.workspace[dec.plan.ws_counters:].view(torch.int32)
    assert int(ctr.abs().sum()) == 0
    dec.check()


def test_bad_page_is_flagged_not_faulted(fdlib):
    spec = _spec("bad", 2, 8, 2, 128, 16, "bf16", "bf16", [100, 300])
    wl = W.make(spec, 5, "cuda")
    bt = wl.block_table.clone()
    bt[1, 3] = -1
    bt[0, 2] = wl.num_pages + 5
    dec = fd.PagedDecoder.for_pools(wl.q, wl.k_pages, wl.v_pages, bt, wl.seq_lens.cpu())
    dec(wl.q, wl.k_pages, wl.v_pages, bt, wl.seq_lens)
    torch.cuda.synchronize()
    word = int(dec.status.item())
    assert word & _lib.FD_DEV_BAD_PAGE
    with pytest.raises(fd.FdError) as ei:
        dec.check()
    assert ei.value.code == _lib.FD_ERR_BAD_PAGE
    # the context is still usable and a clean call still matches the oracle
    _run_and_check(spec, seed=5)


def test_length_above_capacity_is_flagged(fdlib):
    spec = _spec("cap", 1, 8, 2, 128, 16, "bf16", "bf16", [200], extra_blocks=20)
    wl = W.make(spec, 6, "cuda")
    dec = fd.PagedDecoder.for_pools(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens.cpu())
    longer = wl.seq_lens + dec.plan.capacity_tokens
    dec(wl.q, wl.k_pages, wl.v_pages, wl.block_table, longer)
    torch.cuda.synchronize()
    assert int(dec.status.item()) & _lib.FD_DEV_CAPACITY
    with pytest.raises(fd.FdError):
        dec.check()


def test_cuda_graph_replay_matches_eager(fdlib):
    wl = W.make_config(2, "cuda")
    dec = fd.PagedDecoder.for_pools(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens.cpu())
    out = torch.empty_like(wl.q)
    lse = torch.empty(wl.q.shape[:2], dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            dec(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens, out=out, lse=lse)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref_out, ref_lse = out.clone(), lse.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dec(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens, out=out, lse=lse)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    dec.check()


def test_plan_reused_while_lengths_grow(fdlib):
    """A plan made with headroom serves later steps after appends (the
    caller advances seq_lens, as the cookbook's decode loop does)."""
    spec = _spec("grow", 2, 8, 2, 128, 16, "bf16", "bf16", [300, 47], extra_blocks=2)
    wl = W.make(spec, 8, "cpu")
    g = wl.to("cuda")
    dec = fd.PagedDecoder.for_pools(g.q, g.k_pages, g.v_pages, g.block_table, wl.seq_lens,
                                    max_seq_len=int(wl.seq_lens.max()) + 20)
    lens = g.seq_lens.clone()
    gen = torch.Generator().manual_seed(3)
    for step in range(3):
        kn = torch.randn((2, 2, 128), generator=gen).to(torch.bfloat16).cuda()
        vn = torch.randn((2, 2, 128), generator=gen).to(torch.bfloat16).cuda()
        fd.append_kv(torch.bfloat16, kn, vn, g.k_pages, g.v_pages, g.block_table, lens)
        lens += 1
        out, lse = dec(g.q, g.k_pages, g.v_pages, g.block_table, lens)
        torch.cuda.synchronize()
        dec.check()
        cpu = W.Workload(spec, wl.q, g.k_pages.cpu(), g.v_pages.cpu(), None, None, wl.block_table, lens.cpu(),
                         wl.num_pages)
        ref_o, ref_l = oracle_full(cpu)
        assert_close("bf16", out, lse, ref_o, ref_l, f"grow step {step}")


@pytest.mark.parametrize("B,splits,kv", [(96, 2, "bf16"), (97, 2, "bf16"), (100, 2, "bf16"), (1000, 3, "bf16"),
                                         (8192, 2, "bf16"), (2100, 2, "e4m3")])
def test_large_batches_many_row_blocks(fdlib, B, splits, kv):
    """Batches spanning many 32-row blocks of the dispatch tables (and the
    maximum batch): ragged lengths with empty rows, rows shorter than one chunk
    and rows split in several, so full-chunk and partial-chunk items both occur;
    every (row, head) checked against the oracle.  Up to 96 rows the producer
    builds the tables alone, from 97 on every warp of the CTA does."""
    rng = np.random.default_rng(B + splits)
    lens = rng.integers(0, 400, B)
    lens[rng.choice(B, B // 10, replace=False)] = 0
    lens[rng.choice(B, B // 20, replace=False)] = 256  # exactly two full 128-token tiles
    spec = _spec(f"B={B}", B, 8, 2, 64, 16, kv, "bf16", lens.tolist())
    err, dec = _run_and_check(spec, 7 + B, num_splits=splits)
    assert dec.plan.num_splits > 1  # the requested count rounds to whole 128-token tiles


@pytest.mark.parametrize("ps,splits,Hq", [(128, 0, 16), (32, 3, 16), (64, 2, 32)])
def test_fp8_256_token_stages(fdlib, ps, splits, Hq):
    """E4M3 pools with 256-token stages (8 consumer warps x 2 sub-tiles, the
    pairwise epilogue combine): ragged lengths, empty and one-token rows, rows
    ending inside a stage, split and unsplit; G = 8 and G = 16 (two head tiles)."""
    lens = [0, 1, 255, 256, 257, 700, 3000, 130]
    spec = _spec(f"fp8 t256 ps={ps}", len(lens), Hq, 2, 128, ps, "e4m3", "bf16", lens)
    err, dec = _run_and_check(spec, 11 + ps, num_splits=splits, tile_tokens=256)
    assert dec.plan.tile_tokens == 256


@pytest.mark.parametrize("fuse", [1, 0])
@pytest.mark.parametrize("L,splits,want", [(65536, 512, 512), (40000, 300, 157)])
def test_many_splits_up_to_the_maximum(fdlib, L, splits, want, fuse):
    """The largest split count (512 chunks of one 128-token tile) and a count
    past 32 that is not a power of two: the merge's weights span several
    lanes' worth of splits, fused (last-CTA) and in the separate kernel."""
    spec = _spec(f"L={L} S={splits}", 2, 8, 2, 64, 64, "bf16", "bf16", [L, L // 3])
    err, dec = _run_and_check(spec, 5 + splits, num_splits=splits, fuse_merge=fuse)
    assert dec.plan.num_splits == want


@pytest.mark.parametrize("kv,q,ps,D,Hq,Hkv,two", [("bf16", "bf16", 16, 128, 32, 8, True),
                                                   ("e4m3", "bf16", 128, 128, 32, 8, True),
                                                   ("f16", "f16", 32, 64, 32, 8, True),
                                                   ("e4m3", "f16", 64, 128, 32, 8, True),
                                                   ("bf16", "bf16", 16, 64, 32, 2, True),
                                                   ("e4m3", "bf16", 16, 64, 32, 2, None)])
def test_short_items_two_ctas_per_sm(fdlib, kv, q, ps, D, Hq, Hkv, two):
    """Many short sequences: the planner runs two CTAs per SM with 4 consumer
    warps each (64-token stages for 16-bit K/V, 128-token stages of two
    sub-tiles per warp for E4M3); every row against the oracle, with empty,
    one-token and page-boundary lengths among them; G = 4, and G = 16 at
    D = 64 (two 8-head tiles per item).  Whether the E4M3 instance with two
    head tiles fits twice on an SM depends on its register count (two CTAs
    leave at most 168 per thread); the device's occupancy query decides, and
    either shape must match the oracle."""
    rng = np.random.default_rng(31 + ps)
    B = 700
    lens = rng.integers(1, 700, B)
    lens[::50] = 0
    lens[1::50] = 1
    lens[2::50] = ps
    spec = _spec(f"short {kv} G={Hq // Hkv}", B, Hq, Hkv, D, ps, kv, q, lens.tolist())
    err, dec = _run_and_check(spec, 17 + ps + Hkv)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if two is None and dec.plan.ctas_per_sm == 1:
        assert dec.plan.grid_ctas <= sms
        return
    assert dec.plan.ctas_per_sm == 2 and dec.plan.grid_ctas == 2 * sms
    assert dec.plan.tile_tokens == (128 if kv == "e4m3" else 64)


@pytest.mark.parametrize("Hq,D,splits,fuse", [(16, 128, 0, 1), (16, 128, 3, 1), (32, 64, 2, 0), (32, 64, 4, 1)])
def test_fp8_two_ctas_128_token_stages(fdlib, Hq, D, splits, fuse):
    """E4M3 pools with two CTAs per SM and 128-token stages of 4 warps x 2
    sub-tiles (the short-item shape), forced: G = 8 and, at D = 64, G = 16
    (two head tiles); split with the fused and the separate merge."""
    lens = [0, 1, 127, 128, 129, 700, 3000, 255, 256, 64]
    spec = _spec(f"fp8 4x2 G={Hq // 2} D={D}", len(lens), Hq, 2, D, 64, "e4m3", "bf16", lens)
    err, dec = _run_and_check(spec, 41 + D + splits, num_splits=splits, fuse_merge=fuse, tile_tokens=128, ctas_per_sm=2)
    assert dec.plan.tile_tokens == 128 and dec.plan.ctas_per_sm == 2


@pytest.mark.parametrize("kv,q,D,H,L,B", [("f16", "f16", 64, 32, 8192, 1),
                                          ("f16", "f16", 128, 32, 2048, 1),
                                          ("bf16", "bf16", 128, 16, 4096, 2),
                                          ("f16", "f16", 128, 32, 3000, 1),
                                          ("e4m3", "bf16", 128, 32, 3000, 1),
                                          ("f16", "f16", 128, 32, 8192, 1)])  # an imbalanced one-CTA plan
def test_small_grids_two_ctas_per_sm(fdlib, kv, q, D, H, L, B):
    """Fewer items than SMs: the planner's small-grid shape (two CTAs per SM,
    64-token stages, more splits, fused merge) against the oracle on every
    row; one length is not a multiple of the chunk, so the last split is
    ragged."""
    spec = _spec(f"small grid {kv} D={D} L={L}", B, H, H, D, 16, kv, q, [L] * B, pool=("factor", 2.0))
    err, dec = _run_and_check(spec, 61 + D + L)
    assert dec.plan.ctas_per_sm == 2 and dec.plan.num_splits > 4
    assert dec.plan.tile_tokens == (128 if kv == "e4m3" else 64)


@pytest.mark.parametrize("kv,G,D,ps,splits,fuse,opts", [
    ("bf16", 16, 128, 16, 0, 1, {}),         # two head tiles, D = 128: 3 stages instead of 2
    ("bf16", 16, 128, 64, 12, 1, {}),        # many splits: the merge weights in the held stage
    ("bf16", 12, 128, 32, 5, 0, {}),         # ragged head tiles, separate merge
    ("bf16", 4, 128, 16, 0, 1, {"tile_tokens": 64, "ctas_per_sm": 2}),   # two CTAs per SM: 3 stages
    ("bf16", 4, 64, 16, 20, 1, {"tile_tokens": 64, "ctas_per_sm": 2}),
    ("e4m3", 4, 128, 16, 0, 1, {"tile_tokens": 128, "ctas_per_sm": 2}),  # E4M3, 2 KB boxes
    ("e4m3", 8, 128, 16, 12, 1, {"tile_tokens": 128, "ctas_per_sm": 2}),
    ("e4m3", 8, 64, 16, 3, 0, {"tile_tokens": 128, "ctas_per_sm": 2}),
])
def test_epilogue_scratch_in_the_held_stage(fdlib, kv, G, D, ps, splits, fuse, opts):
    """Plans whose epilogue scratch lives in each item's last stage (held by
    the consumers until the epilogue and the fused merge are over, so that
    another stage fits): every row against the oracle, with empty, one-token,
    page-boundary and ragged lengths, several items per CTA so that held
    stages are refilled for the next item."""
    lens = [0, 1, 15, 16, 17, 300, 2900, 4100, 64, 999, 129, 2048]
    spec = _spec(f"held-stage scratch {kv} G={G} D={D}", len(lens), 2 * G, 2, D, ps, kv, "bf16", lens)
    err, dec = _run_and_check(spec, 73 + G + D + splits, num_splits=splits, fuse_merge=fuse, **opts)
    assert dec.plan.scratch_in_stage == 1 and dec.plan.stages >= 3
