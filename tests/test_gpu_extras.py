"""GPU parity of fd_decode_paged_ex (cache_batch_idx and cache_leftpad,
"Inference Cookbook" §5.2-5.3) against the oracle's decode_paged_ex."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from split_kv_decode_paged_gb300 import _lib
from split_kv_decode_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_close, record_errors

pytestmark = pytest.mark.gpu

_CODE = {torch.float16: orc.F16, torch.bfloat16: orc.BF16, torch.float8_e4m3fn: orc.E4M3}


def _run(kv, q, ps, cache_lens, batch_idx, leftpad, Hq=16, Hkv=2, D=128, num_splits=0, fuse=1, seed=0,
         expect_flag=0, out32=False):
    Bc = len(cache_lens)
    spec = W.Spec("ex", B=Bc, Hq=Hq, Hkv=Hkv, D=D, page_size=ps, kv=kv, q=q, lens=("list", cache_lens))
    wl = W.make(spec, 50 + seed, "cpu")
    Bq = len(batch_idx) if batch_idx is not None else Bc
    gen = torch.Generator().manual_seed(seed)
    qv = torch.randn((Bq, Hq, D), generator=gen).to(wl.q.dtype)
    rows = np.arange(Bc) if batch_idx is None else np.asarray(batch_idx)
    lp = np.zeros(Bc, np.int64) if leftpad is None else np.asarray(leftpad)
    # the left-padded tokens hold NaN: any that leaks into a result shows up
    for r in range(Bc):
        for t in range(int(lp[r])):
            page, slot = int(wl.block_table[r, t // ps]), t % ps
            if kv == "e4m3":
                wl.k_pages.view(torch.uint8)[page, slot] = 0x7F
                wl.v_pages.view(torch.uint8)[page, slot] = 0x7F
            else:
                wl.k_pages[page, slot] = float("nan")
                wl.v_pages[page, slot] = float("nan")
    attended = [int(cache_lens[r] - lp[r]) if 0 <= r < Bc else 0 for r in rows]
    out_dtype = torch.float32 if out32 else wl.q.dtype
    prob = _lib.make_problem(Bq, Hq, Hkv, D, ps, wl.max_blocks, wl.num_pages, wl.q.dtype, wl.k_pages.dtype,
                             out_dtype)
    plan = _lib.fd_plan(prob, attended, num_splits=num_splits, fuse_merge=fuse)
    g = wl.to("cuda")
    bi = None if batch_idx is None else torch.tensor(batch_idx, dtype=torch.int32, device="cuda")
    lpd = None if leftpad is None else torch.tensor(leftpad, dtype=torch.int32, device="cuda")
    out = torch.empty((Bq, Hq, D), dtype=out_dtype, device="cuda")
    lse = torch.empty((Bq, Hq), dtype=torch.float32, device="cuda")
    ws = torch.zeros(max(256, plan.workspace_bytes), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.fd_decode_paged_ex(plan, qv.cuda(), g.k_pages, g.v_pages, g.k_scale, g.v_scale, g.block_table, g.seq_lens,
                            out, lse, ws, cache_batch_idx=bi, cache_leftpad=lpd,
                            cache_rows=Bc if batch_idx is not None else 0, status=status)
    torch.cuda.synchronize()
    if expect_flag:
        assert int(status.item()) & expect_flag
        return
    assert int(status.item()) == 0
    p = orc.problem(Bq, Hq, Hkv, D, ps, wl.max_blocks, wl.num_pages, _CODE[wl.q.dtype], _CODE[wl.k_pages.dtype])
    ro, rl = orc.decode_paged_ex(p, Bc, None if batch_idx is None else np.asarray(batch_idx, np.int32),
                                 None if leftpad is None else np.asarray(leftpad, np.int32), qv, wl.k_pages,
                                 wl.v_pages, wl.k_scale, wl.v_scale, wl.block_table, wl.seq_lens)
    name = f"ex kv={kv} ps={ps} splits={num_splits} fuse={fuse}"
    err_o, err_l = assert_close(kv, out, lse, ro, rl, name)
    record_errors(name, out_dtype=str(out_dtype).replace("torch.", ""), out_max_abs_err=err_o,
                  lse_max_abs_err=err_l)


@pytest.mark.parametrize("out32", [False, True], ids=["out-native", "out-f32"])
@pytest.mark.parametrize("splits,fuse", [(0, 1), (1, 1), (3, 1), (3, 0)])
def test_leftpad_unaligned_starts(fdlib, splits, fuse, out32):
    lens = [300, 1000, 40, 513]
    _run("bf16", "bf16", 16, lens, None, [0, 37, 40, 129], num_splits=splits, fuse=fuse, out32=out32)


@pytest.mark.parametrize("ps", [16, 64, 128])
def test_batch_index_subset_with_repeats(fdlib, ps):
    lens = [100, 700, 33, 1500, 260]
    _run("bf16", "bf16", ps, lens, [3, 0, 3, 4, 1], None, num_splits=2)


@pytest.mark.parametrize("out32", [False, True], ids=["out-native", "out-f32"])
def test_fp8_batch_index_and_leftpad(fdlib, out32):
    lens = [400, 1300, 90]
    _run("e4m3", "bf16", 128, lens, [2, 1, 1, 0], [3, 200, 89], Hq=16, Hkv=2, num_splits=2, out32=out32)


def test_f16_leftpad_small_pages(fdlib):
    _run("f16", "f16", 16, [250, 64], None, [249, 1], Hq=8, Hkv=8, D=64, num_splits=4)


def _large_batch_case(seed):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 600, 200)
    bi = rng.integers(0, 200, 300)
    lp = np.array([int(rng.integers(0, n)) for n in lens])
    return lens.tolist(), bi.tolist(), lp.tolist()


@pytest.mark.parametrize("out32", [False, True], ids=["out-native", "out-f32"])
@pytest.mark.parametrize("splits", [0, 2])
def test_large_batch_index_and_leftpad(fdlib, splits, out32):
    """300 q rows over 200 cache rows (permuted, with repeats) and left
    padding: a batch of this size has its dispatch tables built by every warp
    of the CTA, so cache-row indexing and padding go through that path."""
    lens, bi, lp = _large_batch_case(11)
    _run("bf16", "bf16", 16, lens, bi, lp, num_splits=splits, out32=out32)


def test_large_batch_bad_index_is_flagged(fdlib):
    """An index outside the cache in a large batch is flagged (not faulted)."""
    lens, bi, lp = _large_batch_case(12)
    bi[150] = len(lens)
    _run("bf16", "bf16", 16, lens, bi, lp, num_splits=2, expect_flag=_lib.FD_DEV_BAD_PAGE)
