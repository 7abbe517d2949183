"""Host I/O block layout of fd_decode_paged_host (host logic, no GPU): every
region starts on a 256-byte boundary, regions do not overlap, and each holds
its array (block table and seq_lens sized by the plan's KV rows)."""
import pytest
import torch

from split_kv_decode_paged_gb300 import _lib


def _regions(lay, prob, kv_rows):
    e = {torch.float16: 2, torch.bfloat16: 2, torch.float32: 4}
    rows = prob.B * prob.Hq
    qb = rows * prob.D * 2
    ob = rows * prob.D * (4 if prob.out_dtype == _lib.FD_F32 else 2)
    ins = [(lay.q_offset, qb), (lay.block_table_offset, kv_rows * prob.max_blocks_per_seq * 4),
           (lay.seq_lens_offset, kv_rows * 4)]
    outs = [(lay.out_offset, ob), (lay.lse_offset, rows * 4)]
    return ins, outs


def _check(regions, total):
    regions = sorted(regions)
    for (o, n) in regions:
        assert o % 256 == 0 and n > 0
    for (o1, n1), (o2, _) in zip(regions, regions[1:]):
        assert o1 + n1 <= o2
    last_o, last_n = regions[-1]
    assert last_o + last_n <= total and total % 256 == 0


@pytest.mark.parametrize("B,Hq,Hkv,D,ps,mb,out,shared", [
    (4, 8, 2, 128, 16, 10, torch.bfloat16, 0),
    (64, 32, 8, 128, 16, 512, torch.bfloat16, 0),
    (3, 5, 5, 64, 64, 3, torch.float32, 0),
    (16, 32, 8, 128, 16, 300, torch.bfloat16, 1),
])
def test_layout_regions(B, Hq, Hkv, D, ps, mb, out, shared):
    prob = _lib.make_problem(B, Hq, Hkv, D, ps, mb, 4096, torch.bfloat16, torch.bfloat16, out)
    lens = [min(mb * ps, 100 + 37 * i) for i in range(B)]
    plan = _lib.fd_plan(prob, lens[:1] if shared else lens, num_sms=152, shared_kv=shared)
    kv_rows = plan.kv_rows
    assert kv_rows == (1 if shared else B)
    lay = _lib.fd_host_io_layout_for(plan)
    ins, outs = _regions(lay, prob, kv_rows)
    _check(ins, lay.in_bytes)
    _check(outs, lay.out_bytes)
