"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs."""
import numpy as np
import torch

from oracle import oracle as orc
import split_kv_decode_paged_gb300 as fd
from split_kv_decode_paged_gb300 import _lib
from split_kv_decode_paged_gb300 import workloads as W

# Tolerances on |out - oracle| and |lse - oracle| (decode-attention parity bar).
TOL_OUT = {"f16": 2e-3, "bf16": 2e-3, "e4m3": 3e-2}
TOL_LSE = {"f16": 1e-3, "bf16": 1e-3, "e4m3": 3e-2}

_ORC_CODE = {torch.float16: orc.F16, torch.bfloat16: orc.BF16, torch.float8_e4m3fn: orc.E4M3,
             torch.float32: orc.F32}


def oracle_problem(wl: W.Workload):
    s = wl.spec
    return orc.problem(s.B, s.Hq, s.Hkv, s.D, s.page_size, wl.max_blocks, wl.num_pages,
                       _ORC_CODE[wl.q.dtype], _ORC_CODE[wl.k_pages.dtype])


def oracle_full(wl_cpu: W.Workload):
    p = oracle_problem(wl_cpu)
    return orc.decode_paged(p, wl_cpu.q, wl_cpu.k_pages, wl_cpu.v_pages, wl_cpu.k_scale, wl_cpu.v_scale,
                            wl_cpu.block_table, wl_cpu.seq_lens)


def oracle_pairs(wl_cpu: W.Workload, pairs):
    p = oracle_problem(wl_cpu)
    return orc.decode_paged_pairs(p, wl_cpu.q, wl_cpu.k_pages, wl_cpu.v_pages, wl_cpu.k_scale,
                                  wl_cpu.v_scale, wl_cpu.block_table, wl_cpu.seq_lens, pairs)


def gpu_decode(wl_gpu: W.Workload, out_dtype=None, **plan_opts):
    dec = fd.PagedDecoder.for_pools(wl_gpu.q, wl_gpu.k_pages, wl_gpu.v_pages, wl_gpu.block_table,
                                    wl_gpu.seq_lens.cpu(), out_dtype=out_dtype, **plan_opts)
    out, lse = dec(wl_gpu.q, wl_gpu.k_pages, wl_gpu.v_pages, wl_gpu.block_table, wl_gpu.seq_lens,
                   wl_gpu.k_scale, wl_gpu.v_scale)
    torch.cuda.synchronize()
    dec.check()
    return out, lse, dec


_MANT = {torch.bfloat16: 7, torch.float16: 10, torch.float32: 23}


def half_ulp(ref, dtype):
    """Half a unit in the last place of `dtype` at |ref| (normal range): the
    rounding error the output format itself adds to an exact result."""
    a = np.maximum(np.abs(ref), 2.0 ** -14)
    return np.exp2(np.floor(np.log2(a)) - _MANT[dtype] - 1)


def assert_close(kv, out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    """out: |gpu - oracle| <= TOL_OUT + half an ulp of the output dtype at the
    oracle value (the computation's bar plus the output format's own
    rounding); lse (fp32): |gpu - oracle| <= TOL_LSE."""
    o = out_gpu.detach().to(torch.float64).cpu().numpy()
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - out_ref)
    bound = TOL_OUT[kv] + half_ulp(out_ref, out_gpu.dtype)
    worst = np.unravel_index(np.argmax(err - bound), err.shape) if err.size else None
    err_o = float(err.max()) if err.size else 0.0
    assert (err <= bound).all(), (f"{what}: out error {err[worst]:.3e} at {worst} (ref {out_ref[worst]:.4f}) "
                                  f"> bound {bound[worst]:.3e}; max error {err_o:.3e}")
    if lse_gpu is not None:
        l = lse_gpu.detach().to(torch.float64).cpu().numpy()
        both_inf = np.isneginf(l) & np.isneginf(lse_ref)
        diff = np.where(both_inf, 0.0, l - np.where(both_inf, 0.0, lse_ref))
        err_l = np.abs(np.where(both_inf, 0.0, diff)).max() if l.size else 0.0
        assert err_l <= TOL_LSE[kv], f"{what}: lse max-abs error {err_l:.3e} > {TOL_LSE[kv]}"
    return err_o
