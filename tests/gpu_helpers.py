"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and the fp64 oracle on the same seeded inputs."""
import json
import os

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


def merge_bar(ref, out_dtype):
    """Bar for the merge kernels: one unit in the last place of the output
    format at the oracle value, plus 1e-6 (a merge is a handful of fp32
    operations on exact inputs followed by one rounding to the output)."""
    return 2.0 * half_ulp(ref, out_dtype) + 1e-6


def assert_close(kv, out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    """Parity bar against the fp64 oracle.

    out, fp32 output: |gpu - oracle| <= TOL_OUT[kv] (the flat bar: 2e-3 for
    16-bit K/V, 3e-2 for E4M3).  out, f16/bf16 output: TOL_OUT[kv] plus half
    an ulp of the output dtype at the oracle value -- rounding an exact result
    to bf16 alone moves it by up to 1.95e-3 for |out| in [0.5, 1), so the flat
    bar plus the format's own rounding is the bar for a rounded output.
    lse (always fp32): |gpu - oracle| <= TOL_LSE[kv], -inf matching -inf.
    Returns (max out error, max lse error)."""
    o = out_gpu.detach().to(torch.float64).cpu().numpy()
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    err = np.abs(o - out_ref)
    bound = TOL_OUT[kv] + (0.0 if out_gpu.dtype == torch.float32 else half_ulp(out_ref, out_gpu.dtype))
    bound = np.broadcast_to(bound, err.shape)
    worst = np.unravel_index(np.argmax(err - bound), err.shape) if err.size else None
    err_o = float(err.max()) if err.size else 0.0
    assert (err <= bound).all(), (f"{what}: out error {err[worst]:.3e} at {worst} (ref {out_ref[worst]:.4f}) "
                                  f"> bound {bound[worst]:.3e}; max error {err_o:.3e}")
    err_l = 0.0
    if lse_gpu is not None:
        l = lse_gpu.detach().to(torch.float64).cpu().numpy()
        both_inf = np.isneginf(l) & np.isneginf(lse_ref)
        assert (np.isneginf(l) == np.isneginf(lse_ref)).all(), f"{what}: -inf lse mismatch"
        diff = np.where(both_inf, 0.0, l - np.where(both_inf, 0.0, lse_ref))
        err_l = float(np.abs(diff).max()) if l.size else 0.0
        assert err_l <= TOL_LSE[kv], f"{what}: lse max-abs error {err_l:.3e} > {TOL_LSE[kv]}"
    return err_o, err_l


def record_errors(name, **fields):
    """Append one JSON line of measured parity errors to the file named by
    FD_PARITY_REPORT (nothing happens when it is unset)."""
    path = os.environ.get("FD_PARITY_REPORT")
    if not path:
        return
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "a") as f:
        f.write(json.dumps({"case": name, **fields}) + "\n")
