"""GPU fd_append_kv_rotary against the oracle's rotary append, bit for bit
(keys and queries rotated at position seq_lens[b], values copied), then a
decode over the rotated cache against the oracle."""
import numpy as np
import pytest
import torch

import split_kv_decode_paged_gb300 as fd
from oracle import oracle as orc
from split_kv_decode_paged_gb300 import _lib
from tests.gpu_helpers import assert_close

pytestmark = pytest.mark.gpu


def _tables(max_pos, half, base=10000.0):
    inv = 1.0 / base ** (np.arange(half) / half)
    ang = np.arange(max_pos)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


@pytest.mark.parametrize("kv", ["bf16", "f16", "e4m3"])
@pytest.mark.parametrize("interleaved,rd", [(0, 128), (1, 128), (0, 64)])
def test_rotary_append_bitexact(fdlib, kv, interleaved, rd):
    rng = np.random.default_rng(7)
    B, Hq, Hkv, D, ps = 3, 16, 4, 128, 16
    num_pages, maxb = 40, 4
    dt = {"bf16": torch.bfloat16, "f16": torch.float16, "e4m3": torch.float8_e4m3fn}[kv]
    qdt = torch.float16 if kv == "f16" else torch.bfloat16
    bt = torch.from_numpy(rng.permutation(num_pages)[: B * maxb].reshape(B, maxb).astype(np.int32))
    lens = torch.tensor([0, 17, 63], dtype=torch.int32)
    g = torch.Generator().manual_seed(1)
    if kv == "e4m3":
        kp = torch.randint(0, 0x7F, (num_pages, ps, Hkv, D), generator=g, dtype=torch.uint8).view(dt)
        vp = torch.randint(0, 0x7F, (num_pages, ps, Hkv, D), generator=g, dtype=torch.uint8).view(dt)
        ks = (torch.rand((num_pages, Hkv), generator=g) * 0.02 + 0.005).float()
        vs = (torch.rand((num_pages, Hkv), generator=g) * 0.02 + 0.005).float()
    else:
        kp = torch.randn((num_pages, ps, Hkv, D), generator=g).to(dt)
        vp = torch.randn((num_pages, ps, Hkv, D), generator=g).to(dt)
        ks = vs = None
    kn = torch.randn((B, Hkv, D), generator=g).to(qdt)
    vn = torch.randn((B, Hkv, D), generator=g).to(qdt)
    q = torch.randn((B, Hq, D), generator=g).to(qdt)
    c, s = _tables(128, rd // 2)
    code = {"bf16": orc.BF16, "f16": orc.F16, "e4m3": orc.E4M3}[kv]
    qcode = orc.F16 if qdt == torch.float16 else orc.BF16
    p = orc.problem(B, Hq, Hkv, D, ps, maxb, num_pages, qcode, code)
    rk, rv, rq = orc.append_kv_rotary(p, qcode, kn, vn, kp, vp, ks, vs, bt, lens, c, s, rd, interleaved, q)

    gk, gv, gq = kp.cuda(), vp.cuda(), q.cuda()
    prob = _lib.make_problem(B, Hq, Hkv, D, ps, maxb, num_pages, qdt, dt)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.fd_append_kv_rotary(prob, kn.cuda(), vn.cuda(), gk, gv, None if ks is None else ks.cuda(),
                             None if vs is None else vs.cuda(), bt.cuda(), lens.cuda(), torch.from_numpy(c).cuda(),
                             torch.from_numpy(s).cuda(), interleaved=interleaved, q_inout=gq, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(orc.raw(gk.cpu()), rk)
    assert np.array_equal(orc.raw(gv.cpu()), rv)
    assert np.array_equal(orc.raw(gq.cpu()), rq)


def test_rotary_append_then_decode(fdlib):
    rng = np.random.default_rng(8)
    B, Hq, Hkv, D, ps = 2, 8, 2, 128, 16
    num_pages, maxb = 30, 10
    bt = torch.from_numpy(rng.permutation(num_pages)[: B * maxb].reshape(B, maxb).astype(np.int32))
    lens = torch.tensor([100, 37], dtype=torch.int32)
    g = torch.Generator().manual_seed(2)
    kp = torch.randn((num_pages, ps, Hkv, D), generator=g).to(torch.bfloat16)
    vp = torch.randn((num_pages, ps, Hkv, D), generator=g).to(torch.bfloat16)
    kn = torch.randn((B, Hkv, D), generator=g).to(torch.bfloat16)
    vn = torch.randn((B, Hkv, D), generator=g).to(torch.bfloat16)
    q = torch.randn((B, Hq, D), generator=g).to(torch.bfloat16)
    c, s = _tables(512, 64)
    gk, gv, gq = kp.cuda(), vp.cuda(), q.cuda()
    prob = _lib.make_problem(B, Hq, Hkv, D, ps, maxb, num_pages, torch.bfloat16, torch.bfloat16)
    _lib.fd_append_kv_rotary(prob, kn.cuda(), vn.cuda(), gk, gv, None, None, bt.cuda(), lens.cuda(),
                             torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(), q_inout=gq)
    new_lens = (lens + 1).cuda()
    dec = fd.PagedDecoder(prob, (lens + 1).tolist())
    out, lse = dec(gq, gk, gv, bt.cuda(), new_lens)
    torch.cuda.synchronize()
    dec.check()
    p = orc.problem(B, Hq, Hkv, D, ps, maxb, num_pages, orc.BF16, orc.BF16)
    rk, rv, rq = orc.append_kv_rotary(p, orc.BF16, kn, vn, kp, vp, None, None, bt, lens, c, s, 128, 0, q)
    ro, rl = orc.decode_paged(p, rq, rk, rv, None, None, bt, lens + 1)
    assert_close("bf16", out, lse, ro, rl, "rotary append then decode")


def test_rotary_position_beyond_table_is_flagged(fdlib):
    B, Hkv, D, ps = 1, 2, 64, 16
    kp = torch.zeros((4, ps, Hkv, D), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    bt = torch.tensor([[0, 1, 2, 3]], dtype=torch.int32, device="cuda")
    lens = torch.tensor([40], dtype=torch.int32, device="cuda")
    c = torch.ones((32, 16), dtype=torch.float32, device="cuda")
    s = torch.zeros((32, 16), dtype=torch.float32, device="cuda")
    kn = torch.ones((B, Hkv, D), dtype=torch.bfloat16, device="cuda")
    prob = _lib.make_problem(B, Hkv, Hkv, D, ps, 4, 4, torch.bfloat16, torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _lib.fd_append_kv_rotary(prob, kn, kn, kp, vp, None, None, bt, lens, c, s, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & _lib.FD_DEV_CAPACITY
    assert not kp.float().abs().sum().item()  # nothing written
