"""GPU tests of fd_append_kv (bit-exact against the oracle's append, the rest
of each pool unchanged) and fd_merge_states (against the oracle's merge)."""
import numpy as np
import pytest
import torch

import split_kv_decode_paged_gb300 as fd
from split_kv_decode_paged_gb300 import _lib
from oracle import oracle as orc
from tests.gpu_helpers import merge_bar

pytestmark = pytest.mark.gpu

_CODE = {torch.float16: orc.F16, torch.bfloat16: orc.BF16, torch.float8_e4m3fn: orc.E4M3}


def _pool_case(kv_dtype, q_dtype, B=5, Hkv=4, D=128, ps=16, seed=0):
    g = torch.Generator().manual_seed(seed)
    num_pages = 40
    lens = torch.tensor([0, 15, 16, 33, 47][:B], dtype=torch.int32)
    maxb = 4
    perm = torch.randperm(num_pages, generator=g)[: B * maxb].to(torch.int32)
    bt = perm.view(B, maxb).clone()
    shape = (num_pages, ps, Hkv, D)
    if kv_dtype == torch.float8_e4m3fn:
        kp = torch.randint(0, 0x7F, shape, generator=g, dtype=torch.uint8).view(torch.float8_e4m3fn)
        vp = torch.randint(0, 0x7F, shape, generator=g, dtype=torch.uint8).view(torch.float8_e4m3fn)
        ks = (torch.rand((num_pages, Hkv), generator=g) * 0.05 + 0.001).float()
        vs = (torch.rand((num_pages, Hkv), generator=g) * 0.05 + 0.001).float()
    else:
        kp = torch.randn(shape, generator=g).to(kv_dtype)
        vp = torch.randn(shape, generator=g).to(kv_dtype)
        ks = vs = None
    new_dtype = q_dtype if kv_dtype == torch.float8_e4m3fn else kv_dtype
    kn = (torch.randn((B, Hkv, D), generator=g) * 3).to(new_dtype)
    vn = (torch.randn((B, Hkv, D), generator=g) * 3).to(new_dtype)
    kn[0, 0, :4] = torch.tensor([1e4, -1e4, 0.0, -0.0])  # saturation and signed zero
    return kp, vp, ks, vs, bt, lens, kn, vn, new_dtype


@pytest.mark.parametrize("kv,q", [(torch.bfloat16, torch.bfloat16), (torch.float16, torch.float16),
                                  (torch.float8_e4m3fn, torch.bfloat16), (torch.float8_e4m3fn, torch.float16)])
def test_append_bitexact_vs_oracle(fdlib, kv, q):
    kp, vp, ks, vs, bt, lens, kn, vn, new_dtype = _pool_case(kv, q)
    B, Hkv, D = kn.shape
    num_pages, ps = kp.shape[0], kp.shape[1]
    p = orc.problem(B, Hkv, Hkv, D, ps, bt.shape[1], num_pages, _CODE[q], _CODE[kv])
    ref_k, ref_v = orc.append_kv(p, _CODE[new_dtype], kn, vn, kp, vp, ks, vs, bt, lens)
    gk, gv = kp.cuda(), vp.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fd.append_kv(q, kn.cuda(), vn.cuda(), gk, gv, bt.cuda(), lens.cuda(),
                 None if ks is None else ks.cuda(), None if vs is None else vs.cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(orc.raw(gk.cpu()), ref_k)
    assert np.array_equal(orc.raw(gv.cpu()), ref_v)


def test_append_bad_page_flagged(fdlib):
    kp, vp, ks, vs, bt, lens, kn, vn, _ = _pool_case(torch.bfloat16, torch.bfloat16)
    bt[2, 1] = -1           # seq 2 has L = 16 -> column 1
    lens[4] = 4 * 16 + 3    # beyond the table's columns
    gk, gv = kp.cuda(), vp.cuda()
    before_k = gk.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    fd.append_kv(torch.bfloat16, kn.cuda(), vn.cuda(), gk, gv, bt.cuda(), lens.cuda(), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & _lib.FD_DEV_BAD_PAGE
    # the skipped sequences wrote nothing; the others did
    changed = (gk.view(torch.int16) != before_k.view(torch.int16)).any(dim=(2, 3)).nonzero().tolist()
    assert {(int(bt[0, 0]), 0), (int(bt[1, 0]), 15), (int(bt[3, 2]), 1)} == {tuple(x) for x in changed}


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_merge_states_vs_oracle(fdlib, out_dtype):
    g = torch.Generator().manual_seed(1)
    B, Hq, S, D = 3, 5, 7, 128
    o = torch.randn((B, Hq, S, D), generator=g, dtype=torch.float64)
    m = torch.randn((B, Hq, S), generator=g, dtype=torch.float64) * 4
    d = torch.rand((B, Hq, S), generator=g, dtype=torch.float64) * 10 + 0.5
    m[0, 0, 2] = -float("inf"); d[0, 0, 2] = 0; o[0, 0, 2] = 0     # an empty chunk
    m[1, 2, :] = -float("inf"); d[1, 2, :] = 0; o[1, 2, :] = 0     # an all-empty row
    o32, m32, d32 = o.float(), m.float(), d.float()
    out, lse = fd.merge_states(o32.cuda(), m32.cuda(), d32.cuda(), out_dtype=out_dtype)
    torch.cuda.synchronize()
    for b in range(B):
        for h in range(Hq):
            ro, rl = orc.merge_states(o32[b, h].double().numpy(), m32[b, h].double().numpy(),
                                      d32[b, h].double().numpy())
            got = out[b, h].double().cpu().numpy()
            assert (np.abs(got - ro) <= merge_bar(ro, out_dtype)).all(), (b, h)
            gl = float(lse[b, h])
            if rl == -np.inf:
                assert gl == -np.inf and not got.any()
            else:
                assert abs(gl - rl) < 1e-5


def _merge_case(B, Hq, S, D, seed, offset=0):
    g = torch.Generator().manual_seed(seed)
    n = B * Hq * S * D
    buf = torch.empty(n + offset, dtype=torch.float32)
    o = buf[offset:].view(B, Hq, S, D)
    o.copy_(torch.randn((B, Hq, S, D), generator=g))
    m = torch.randn((B, Hq, S), generator=g) * 4
    d = torch.rand((B, Hq, S), generator=g) * 10 + 0.5
    m[0, 0, S // 2] = -float("inf"); d[0, 0, S // 2] = 0; o[0, 0, S // 2] = 0   # an empty chunk
    m[B - 1, Hq - 1, :] = -float("inf"); d[B - 1, Hq - 1, :] = 0; o[B - 1, Hq - 1] = 0  # an all-empty row
    return buf, o, m, d


@pytest.mark.parametrize("S,D,offset", [(1, 128, 0), (9, 96, 0), (40, 64, 0), (33, 50, 0), (70, 33, 0),
                                        (8, 256, 0), (12, 128, 1)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_merge_states_shapes_vs_oracle(fdlib, S, D, offset, out_dtype):
    """Odd head sizes, more than 32 splits and a partial-state base that is only
    4-byte aligned (scalar loads) against the oracle's merge."""
    B, Hq = 2, 3
    buf, o, m, d = _merge_case(B, Hq, S, D, 100 + S + D, offset)
    gbuf = buf.cuda()
    go = gbuf[offset:].view(B, Hq, S, D)
    out, lse = fd.merge_states(go, m.cuda(), d.cuda(), out_dtype=out_dtype)
    torch.cuda.synchronize()
    for b in range(B):
        for h in range(Hq):
            ro, rl = orc.merge_states(o[b, h].double().numpy(), m[b, h].double().numpy(), d[b, h].double().numpy())
            got = out[b, h].double().cpu().numpy()
            assert (np.abs(got - ro) <= merge_bar(ro, out_dtype)).all(), (b, h)
            gl = float(lse[b, h])
            if rl == -np.inf:
                assert gl == -np.inf and not got.any()
            else:
                assert abs(gl - rl) < 1e-5
