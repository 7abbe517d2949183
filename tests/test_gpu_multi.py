"""GPU parity of the multi-token (causal) decode: q_len query tokens per
sequence, token i of them attending the cached tokens [0, L - q_len + i + 1)
("Inference Cookbook" §3.2-3.3, flash_attn_with_kvcache with causal=True after
the new tokens were appended; "FlashDecoding 与 FlashInfer 深度解析" §3.1, the
append mode), against the oracle's decode_paged_multi on every row."""
import numpy as np
import pytest
import torch

import split_kv_decode_paged_gb300 as fd
from oracle import oracle as orc
from split_kv_decode_paged_gb300 import _lib
from split_kv_decode_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_close, record_errors

pytestmark = pytest.mark.gpu

_CODE = {torch.float16: orc.F16, torch.bfloat16: orc.BF16, torch.float8_e4m3fn: orc.E4M3}


def _run(kv, q, ps, D, Hq, Hkv, q_len, lens, seed, out32=False, **plan_opts):
    spec = W.Spec("multi", B=len(lens), Hq=Hq, Hkv=Hkv, D=D, page_size=ps, kv=kv, q=q, lens=("list", list(lens)))
    wl = W.make(spec, seed, "cpu")
    gen = torch.Generator().manual_seed(seed + 1)
    qm = torch.randn((len(lens), q_len, Hq, D), generator=gen).to(wl.q.dtype)
    g = wl.to("cuda")
    dec = fd.PagedDecoder.for_pools(qm.cuda(), g.k_pages, g.v_pages, g.block_table, wl.seq_lens,
                                    out_dtype=torch.float32 if out32 else None, **plan_opts)
    assert dec.plan.q_len == q_len
    out, lse = dec(qm.cuda(), g.k_pages, g.v_pages, g.block_table, g.seq_lens, g.k_scale, g.v_scale)
    torch.cuda.synchronize()
    dec.check()
    assert out.shape == (len(lens), q_len, Hq, D) and lse.shape == (len(lens), q_len, Hq)
    p = orc.problem(len(lens), Hq, Hkv, D, ps, wl.max_blocks, wl.num_pages, _CODE[wl.q.dtype], _CODE[wl.k_pages.dtype])
    ro, rl = orc.decode_paged_multi(p, q_len, qm, wl.k_pages, wl.v_pages, wl.k_scale, wl.v_scale, wl.block_table,
                                    wl.seq_lens)
    name = f"multi {kv} G={Hq // Hkv} q_len={q_len} {plan_opts}"
    err_o, err_l = assert_close(kv, out, lse, ro, rl, name)
    record_errors(name, out_dtype=str(out.dtype).replace("torch.", ""), out_max_abs_err=err_o, lse_max_abs_err=err_l)
    return out, lse, dec


CASES = [
    # kv, q, ps, D, Hq, Hkv, q_len, lens
    ("bf16", "bf16", 16, 128, 32, 8, 4, [4, 17, 300, 2000, 129]),     # G x q_len = 16 rows: two head tiles
    ("f16", "f16", 32, 64, 8, 8, 2, [2, 3, 64, 65, 1000]),            # MHA
    ("e4m3", "bf16", 128, 128, 16, 2, 2, [2, 130, 700, 3000]),        # FP8 pages, 16 rows
    ("bf16", "bf16", 64, 128, 16, 4, 8, [8, 9, 200, 1500]),           # 32 rows: two 16-row sub-groups
    ("bf16", "bf16", 16, 128, 8, 8, 3, [3, 40, 517]),                 # G = 1, q_len 3 (one head tile)
]


@pytest.mark.parametrize("out32", [False, True], ids=["out-native", "out-f32"])
@pytest.mark.parametrize("splits,fuse", [(0, 1), (3, 1), (3, 0)])
@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-G{c[4] // c[5]}-q{c[6]}" for c in CASES])
def test_multi_token_vs_oracle(fdlib, case, splits, fuse, out32):
    kv, q, ps, D, Hq, Hkv, q_len, lens = case
    _run(kv, q, ps, D, Hq, Hkv, q_len, lens, seed=13 + q_len + splits, out32=out32, num_splits=splits,
         fuse_merge=fuse)


def test_multi_token_one_equals_plain_decode(fdlib):
    """q_len = 1 through the multi-token path is the plain decode, bit for bit."""
    spec = W.Spec("m1", B=3, Hq=16, Hkv=4, D=128, page_size=16, kv="bf16", q="bf16", lens=("list", [1, 300, 2000]))
    wl = W.make(spec, 5, "cuda")
    dec = fd.PagedDecoder.for_pools(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens.cpu())
    ref_o, ref_l = dec(wl.q, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens)
    q4 = wl.q.view(3, 1, 16, 128)
    dm = fd.PagedDecoder.for_pools(q4, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens.cpu())
    out, lse = dm(q4, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert torch.equal(out.view(3, 16, 128), ref_o) and torch.equal(lse.view(3, 16), ref_l)


def test_multi_token_many_short_sequences(fdlib):
    """Many short sequences with two query tokens each (the dispatch tables of
    a large batch, built by every warp), every row against the oracle; the
    causal shape is one CTA per SM with 128-token stages."""
    rng = np.random.default_rng(3)
    lens = rng.integers(2, 500, 700)
    out, lse, dec = _run("bf16", "bf16", 16, 128, 32, 8, 2, lens.tolist(), seed=21)
    assert dec.plan.ctas_per_sm == 1 and dec.plan.tile_tokens == 128


def test_multi_token_cache_shorter_than_query_is_flagged(fdlib):
    spec = W.Spec("short", B=2, Hq=8, Hkv=2, D=128, page_size=16, kv="bf16", q="bf16", lens=("list", [10, 2]))
    wl = W.make(spec, 3, "cuda")
    qm = torch.randn((2, 4, 8, 128), device="cuda").to(torch.bfloat16)
    dec = fd.PagedDecoder.for_pools(qm, wl.k_pages, wl.v_pages, wl.block_table, [10, 4])  # plan lengths >= q_len
    dec(qm, wl.k_pages, wl.v_pages, wl.block_table, wl.seq_lens)
    torch.cuda.synchronize()
    assert int(dec.status.item()) & _lib.FD_DEV_CAPACITY
    with pytest.raises(fd.FdError):
        dec.check()


def test_multi_token_host_step_matches_device_call(fdlib):
    """fd_decode_paged_host with two query tokens per sequence: one packed
    input copy, the decode, the output block; bit-identical to the
    device-buffer call."""
    spec = W.Spec("mh", B=3, Hq=16, Hkv=4, D=128, page_size=16, kv="bf16", q="bf16", lens=("list", [2, 300, 1500]))
    wl = W.make(spec, 9, "cpu")
    g = wl.to("cuda")
    qm = torch.randn((3, 2, 16, 128), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    dec = fd.PagedDecoder.for_pools(qm.cuda(), g.k_pages, g.v_pages, g.block_table, wl.seq_lens)
    ref_out, ref_lse = dec(qm.cuda(), g.k_pages, g.v_pages, g.block_table, g.seq_lens)
    torch.cuda.synchronize()
    io = dec.host_step()
    assert io.q.shape == (3, 2, 16, 128) and io.lse.shape == (3, 2, 16)
    io.q.copy_(qm)
    io.block_table.copy_(wl.block_table)
    io.seq_lens.copy_(wl.seq_lens)
    dec.step_host(io, g.k_pages, g.v_pages)
    torch.cuda.synchronize()
    dec.check()
    assert torch.equal(io.out.view(torch.uint8), ref_out.cpu().view(torch.uint8))
    assert torch.equal(io.lse.view(torch.int32), ref_lse.cpu().view(torch.int32))
