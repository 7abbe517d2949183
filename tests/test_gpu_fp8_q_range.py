"""E4M3 K/V with a bf16 query over bf16's whole exponent range.

The E4M3 path multiplies q by K on the f16 tensor-core product; q enters it
scaled per head by a power of two, so bf16 values above f16's range
(65504) or below its normal range (6.1e-5) keep every bit.  The query is
scaled by 2^e and the page scales of K by 2^-e (both exact), so the scores
keep their size while q alone leaves f16's range; the oracle sees the same
stored values ("Inference Cookbook" §7: FP8 KV with descale factors, the
query in its own dtype)."""
import pytest
import torch

from split_kv_decode_paged_gb300 import workloads as W
from tests.gpu_helpers import assert_close, gpu_decode, oracle_full, record_errors

pytestmark = pytest.mark.gpu


def _case(q_exp_per_head, k_exp, seed, ps=128, lens=(130, 900, 2000), Hq=16):
    spec = W.Spec("fp8 q range", B=len(lens), Hq=Hq, Hkv=2, D=128, page_size=ps, kv="e4m3", q="bf16",
                  lens=("list", list(lens)))
    wl = W.make(spec, seed, "cpu")
    e = torch.tensor(q_exp_per_head, dtype=torch.float64)[None, :, None]
    q = (wl.q.double() * torch.exp2(e)).to(torch.bfloat16)
    assert torch.equal(q.double(), wl.q.double() * torch.exp2(e))  # exact power-of-two scaling
    ks = (wl.k_scale.double() * 2.0 ** k_exp).float()
    return W.Workload(spec, q, wl.k_pages, wl.v_pages, ks, wl.v_scale, wl.block_table, wl.seq_lens, wl.num_pages)


@pytest.mark.parametrize("out32", [False, True], ids=["out-native", "out-f32"])
@pytest.mark.parametrize("q_exp", [-22, -16, 17, 20])
def test_fp8_q_outside_f16_range(fdlib, q_exp, out32):
    """Every head's q scaled by 2^q_exp (|q| up to ~1e6, or down to ~1e-7),
    K's scales by 2^-q_exp."""
    wl = _case([q_exp] * 16, -q_exp, seed=71 + q_exp)
    out, lse, dec = gpu_decode(wl.to("cuda"), out_dtype=torch.float32 if out32 else None, num_splits=2)
    ref_o, ref_l = oracle_full(wl)
    err_o, err_l = assert_close("e4m3", out, lse, ref_o, ref_l, f"q x 2^{q_exp}")
    record_errors(f"e4m3 q x 2^{q_exp}", out_dtype=str(out.dtype).replace("torch.", ""), out_max_abs_err=err_o,
                  lse_max_abs_err=err_l)


@pytest.mark.parametrize("Hq", [16, 8])
def test_fp8_q_heads_of_different_magnitudes(fdlib, Hq):
    """Heads of one work item at magnitudes 2^-12 .. 2^4 (each head is scaled
    on its own; two 8-head tiles with Hq=16, one with Hq=8)."""
    exps = [-12, -6, 0, 4, -3, 2, -9, 1, 3, -1, 0, -12, 4, -5, 2, 0][:Hq]
    wl = _case(exps, 0, seed=80 + Hq, ps=64, lens=(64, 700, 3001), Hq=Hq)
    out, lse, dec = gpu_decode(wl.to("cuda"), out_dtype=torch.float32, num_splits=0)
    ref_o, ref_l = oracle_full(wl)
    assert_close("e4m3", out, lse, ref_o, ref_l, "per-head magnitudes")
