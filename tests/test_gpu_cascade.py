"""Cascade (shared-prefix) decode: prefix pass + suffix pass + fd_merge_two
must equal the plain attention over the concatenated tokens (the oracle's
decode over per-sequence tables listing the prefix pages then the own pages)."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from split_kv_decode_paged_gb300 import _lib
from split_kv_decode_paged_gb300 import workloads as W
from split_kv_decode_paged_gb300.cascade import CascadeDecoder
from tests.gpu_helpers import assert_close, merge_bar, oracle_full, record_errors

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("out32", [False, True], ids=["out-native", "out-f32"])
@pytest.mark.parametrize("kv,q,ps,prefix,suffix", [
    ("bf16", "bf16", 16, 1024, [0, 1, 37, 300, 1000]),
    ("f16", "f16", 64, 256, [5, 64, 129]),
    ("e4m3", "bf16", 128, 512, [200, 0, 700]),
])
def test_cascade_equals_flat_attention(fdlib, kv, q, ps, prefix, suffix, out32):
    spec = W.Spec("cascade", B=len(suffix), Hq=16, Hkv=4, D=128, page_size=ps, kv=kv, q=q, lens=("const", 1))
    sp = W.make_shared_prefix(spec, 31, prefix, suffix, "cpu")
    g = sp.flat.to("cuda")
    cas = CascadeDecoder(spec.B, spec.Hq, spec.Hkv, spec.D, ps, sp.flat.num_pages, sp.prefix_table.shape[1],
                         sp.suffix_table.shape[1], prefix, sp.suffix_lens, g.q.dtype, g.k_pages.dtype)
    out = torch.empty(g.q.shape, dtype=torch.float32 if out32 else g.q.dtype, device="cuda")
    out, lse = cas(g.q, g.k_pages, g.v_pages, sp.prefix_table.cuda(),
                   torch.tensor([prefix], dtype=torch.int32, device="cuda"), sp.suffix_table.cuda(),
                   sp.suffix_lens.cuda(), g.k_scale, g.v_scale, out=out)
    torch.cuda.synchronize()
    cas.check()
    ref_o, ref_l = oracle_full(sp.flat)
    err_o, err_l = assert_close(kv, out, lse, ref_o, ref_l, f"cascade {kv}")
    record_errors(f"cascade {kv} ps={ps} prefix={prefix}", out_dtype=str(out.dtype).replace("torch.", ""),
                  out_max_abs_err=err_o, lse_max_abs_err=err_l)


def test_merge_two_vs_oracle(fdlib):
    g = torch.Generator().manual_seed(4)
    rows, D = 37, 128
    oa, ob = torch.randn((rows, D), generator=g), torch.randn((rows, D), generator=g)
    la, lb = torch.randn(rows, generator=g) * 3, torch.randn(rows, generator=g) * 3
    la[0] = -float("inf"); lb[1] = -float("inf"); la[2] = lb[2] = -float("inf")
    out = torch.empty((rows, D), device="cuda")
    lse = torch.empty(rows, device="cuda")
    _lib.fd_merge_two(oa.cuda(), la.cuda(), ob.cuda(), lb.cuda(), out, lse)
    torch.cuda.synchronize()
    for r in range(rows):
        ro, rl = orc.merge_states(np.stack([oa[r].double().numpy(), ob[r].double().numpy()]),
                                  np.array([la[r].item(), lb[r].item()]), np.ones(2))
        assert (np.abs(out[r].double().cpu().numpy() - ro) <= merge_bar(ro, torch.float32)).all(), r
        if rl == -np.inf:
            assert lse[r].item() == -np.inf and not out[r].any()
        else:
            assert abs(lse[r].item() - rl) < 1e-5
