"""ctypes wrapper around liboracle.so, the fp64 CPU oracle.

TEST INFRASTRUCTURE ONLY.  Imported by tests/, by the package smoke check and
by bench.py's CPU-baseline leg; never by the CUDA product path.  It does not
import the CUDA package, and the CUDA package does not import it.

Arrays are passed as raw storage: 16-bit formats as uint16 bit patterns,
E4M3 as uint8 codes, fp32 as float32.  torch CPU tensors are accepted and
reinterpreted (no value conversion happens here).
"""
import ctypes
import os

import numpy as np

from . import build as _build

F16, BF16, E4M3, F32 = 0, 1, 2, 3
OK, ERR_ARG, ERR_BAD_PAGE, ERR_NOMEM = 0, 1, 2, 3

_lib = None


class Problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "B", "Hq", "Hkv", "D", "page_size", "max_blocks_per_seq", "num_pages",
        "q_dtype", "kv_dtype")]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        L.orc_f16_to_double.restype = ctypes.c_double
        L.orc_f16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_double.restype = ctypes.c_double
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_e4m3_to_double.restype = ctypes.c_double
        L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_from_float.restype = ctypes.c_uint8
        L.orc_e4m3_from_float.argtypes = [ctypes.c_float]
        L.orc_decode_paged.restype = I
        L.orc_decode_paged.argtypes = [ctypes.POINTER(Problem), P, P, P, P, P, P, P, P, P, I]
        L.orc_decode_paged_pairs.restype = I
        L.orc_decode_paged_pairs.argtypes = [ctypes.POINTER(Problem), P, P, P, P, P, P, P,
                                             P, I, P, P, I]
        L.orc_decode_paged_ex.restype = I
        L.orc_decode_paged_ex.argtypes = [ctypes.POINTER(Problem), I, P, P, P, P, P, P, P, P, P, P, P]
        L.orc_rotary_f32.restype = None
        L.orc_rotary_f32.argtypes = [P, I, I, I, P, P, I, P]
        L.orc_append_kv_rotary.restype = I
        L.orc_append_kv_rotary.argtypes = [ctypes.POINTER(Problem), I, P, P, P, P, P, P, P, P, P, P, I, I, I, P]
        L.orc_decode_paged_multi.restype = I
        L.orc_decode_paged_multi.argtypes = [ctypes.POINTER(Problem), I, P, P, P, P, P, P, P, P, P]
        L.orc_decode_contiguous.restype = I
        L.orc_decode_contiguous.argtypes = [ctypes.POINTER(Problem), I, P, P, P, P, P, P]
        L.orc_partial_state.restype = I
        L.orc_partial_state.argtypes = [ctypes.POINTER(Problem), P, P, P, P, P, P, I, I, I, I,
                                        P, P, P]
        L.orc_merge_states.restype = None
        L.orc_merge_states.argtypes = [I, I, P, P, P, P, P]
        L.orc_append_kv.restype = I
        L.orc_append_kv.argtypes = [ctypes.POINTER(Problem), I, P, P, P, P, P, P, P, P]
        _lib = L
    return _lib


_TORCH_RAW = {"torch.float16": np.uint16, "torch.bfloat16": np.uint16,
              "torch.float8_e4m3fn": np.uint8, "torch.float32": np.float32,
              "torch.int32": np.int32, "torch.uint8": np.uint8, "torch.int16": np.uint16,
              "torch.float64": np.float64}


def raw(a):
    """Contiguous numpy view of the storage of `a` (numpy array or CPU tensor)."""
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        return np.ascontiguousarray(a)
    import torch
    t = a.detach()
    if t.device.type != "cpu":
        raise ValueError("oracle inputs must be host tensors")
    t = t.contiguous()
    key = str(t.dtype)
    if key not in _TORCH_RAW:
        raise TypeError(f"unsupported dtype {t.dtype}")
    width = {np.uint16: torch.int16, np.uint8: torch.uint8}.get(_TORCH_RAW[key])
    if width is not None and t.dtype not in (torch.uint8,):
        t = t.view(width)
    return t.numpy().view(_TORCH_RAW[key])


def dtype_code(a):
    """Oracle dtype code of a torch tensor (by its dtype)."""
    key = str(a.dtype)
    return {"torch.float16": F16, "torch.bfloat16": BF16, "torch.float8_e4m3fn": E4M3,
            "torch.float32": F32}[key]


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def problem(B, Hq, Hkv, D, page_size, max_blocks_per_seq, num_pages, q_dtype, kv_dtype):
    return Problem(B, Hq, Hkv, D, page_size, max_blocks_per_seq, num_pages, q_dtype, kv_dtype)


def _check(rc, what):
    if rc == ERR_BAD_PAGE:
        raise IndexError(f"{what}: page index out of range")
    if rc != OK:
        raise ValueError(f"{what}: oracle error {rc}")


def decode_paged(p, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, nthreads=0):
    """Full-softmax decode; returns (out [B,Hq,D] f64, lse [B,Hq] f64)."""
    q, k, v = raw(q), raw(k_pages), raw(v_pages)
    ks, vs = raw(k_scale), raw(v_scale)
    bt, sl = raw(block_table).astype(np.int32), raw(seq_lens).astype(np.int32)
    out = np.zeros((p.B, p.Hq, p.D), np.float64)
    lse = np.zeros((p.B, p.Hq), np.float64)
    rc = lib().orc_decode_paged(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(ks), _ptr(vs),
                                _ptr(bt), _ptr(sl), _ptr(out), _ptr(lse), int(nthreads))
    _check(rc, "decode_paged")
    return out, lse


def decode_paged_pairs(p, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, pairs,
                       nthreads=0):
    """Decode only the listed (b, hq) pairs; returns (out [n,D], lse [n])."""
    q, k, v = raw(q), raw(k_pages), raw(v_pages)
    ks, vs = raw(k_scale), raw(v_scale)
    bt, sl = raw(block_table).astype(np.int32), raw(seq_lens).astype(np.int32)
    pr = np.ascontiguousarray(np.asarray(pairs, np.int32).reshape(-1, 2))
    n = pr.shape[0]
    out = np.zeros((n, p.D), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = lib().orc_decode_paged_pairs(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(ks),
                                      _ptr(vs), _ptr(bt), _ptr(sl), _ptr(pr), n, _ptr(out),
                                      _ptr(lse), int(nthreads))
    _check(rc, "decode_paged_pairs")
    return out, lse


def decode_paged_ex(p, cache_rows, cache_batch_idx, cache_leftpad, q, k_pages, v_pages, k_scale, v_scale,
                    block_table, seq_lens):
    """Decode with cache-row indirection and left padding; p.B = q rows."""
    q, k, v = raw(q), raw(k_pages), raw(v_pages)
    ks, vs = raw(k_scale), raw(v_scale)
    bt, sl = raw(block_table).astype(np.int32), raw(seq_lens).astype(np.int32)
    bi = None if cache_batch_idx is None else raw(cache_batch_idx).astype(np.int32)
    lp = None if cache_leftpad is None else raw(cache_leftpad).astype(np.int32)
    out = np.zeros((p.B, p.Hq, p.D), np.float64)
    lse = np.zeros((p.B, p.Hq), np.float64)
    rc = lib().orc_decode_paged_ex(ctypes.byref(p), int(cache_rows), _ptr(bi), _ptr(lp), _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl), _ptr(out), _ptr(lse))
    _check(rc, "decode_paged_ex")
    return out, lse


def decode_paged_multi(p, q_len, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens):
    """q_len causal query tokens per sequence: q [B, q_len, Hq, D] ->
    (out [B, q_len, Hq, D] f64, lse [B, q_len, Hq] f64)."""
    q, k, v = raw(q), raw(k_pages), raw(v_pages)
    ks, vs = raw(k_scale), raw(v_scale)
    bt, sl = raw(block_table).astype(np.int32), raw(seq_lens).astype(np.int32)
    out = np.zeros((p.B, q_len, p.Hq, p.D), np.float64)
    lse = np.zeros((p.B, q_len, p.Hq), np.float64)
    rc = lib().orc_decode_paged_multi(ctypes.byref(p), int(q_len), _ptr(q), _ptr(k), _ptr(v), _ptr(ks), _ptr(vs),
                                      _ptr(bt), _ptr(sl), _ptr(out), _ptr(lse))
    _check(rc, "decode_paged_multi")
    return out, lse


def decode_contiguous(p, max_seqlen, q, k_cache, v_cache, seq_lens):
    q, k, v, sl = raw(q), raw(k_cache), raw(v_cache), raw(seq_lens).astype(np.int32)
    out = np.zeros((p.B, p.Hq, p.D), np.float64)
    lse = np.zeros((p.B, p.Hq), np.float64)
    rc = lib().orc_decode_contiguous(ctypes.byref(p), int(max_seqlen), _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(sl), _ptr(out), _ptr(lse))
    _check(rc, "decode_contiguous")
    return out, lse


def partial_state(p, q, k_pages, v_pages, k_scale, v_scale, block_table, b, hq, t_begin, t_end):
    """Unnormalised partial state (o [D], m, d) over tokens [t_begin, t_end)."""
    q, k, v = raw(q), raw(k_pages), raw(v_pages)
    ks, vs, bt = raw(k_scale), raw(v_scale), raw(block_table).astype(np.int32)
    o = np.zeros((p.D,), np.float64)
    m = np.zeros((1,), np.float64)
    d = np.zeros((1,), np.float64)
    rc = lib().orc_partial_state(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(ks), _ptr(vs),
                                 _ptr(bt), int(b), int(hq), int(t_begin), int(t_end), _ptr(o),
                                 _ptr(m), _ptr(d))
    _check(rc, "partial_state")
    return o, float(m[0]), float(d[0])


def merge_states(o, m, d):
    """Merge n partial states: o [n, D], m [n], d [n] -> (out [D], lse)."""
    o = np.ascontiguousarray(o, np.float64)
    m = np.ascontiguousarray(m, np.float64)
    d = np.ascontiguousarray(d, np.float64)
    n, D = o.shape
    out = np.zeros((D,), np.float64)
    lse = np.zeros((1,), np.float64)
    lib().orc_merge_states(n, D, _ptr(o), _ptr(m), _ptr(d), _ptr(out), _ptr(lse))
    return out, float(lse[0])


def append_kv(p, new_dtype, k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table,
              seq_lens):
    """Returns new copies of (k_pages, v_pages) with the tokens appended."""
    kn, vn = raw(k_new), raw(v_new)
    k, v = raw(k_pages).copy(), raw(v_pages).copy()
    ks, vs = raw(k_scale), raw(v_scale)
    bt, sl = raw(block_table).astype(np.int32), raw(seq_lens).astype(np.int32)
    rc = lib().orc_append_kv(ctypes.byref(p), int(new_dtype), _ptr(kn), _ptr(vn), _ptr(k), _ptr(v),
                             _ptr(ks), _ptr(vs), _ptr(bt), _ptr(sl))
    _check(rc, "append_kv")
    return k, v


def f16_to_double(bits):
    return lib().orc_f16_to_double(int(bits))


def bf16_to_double(bits):
    return lib().orc_bf16_to_double(int(bits))


def e4m3_to_double(bits):
    return lib().orc_e4m3_to_double(int(bits))


def e4m3_from_float(x):
    return int(lib().orc_e4m3_from_float(float(x)))


def rotary_f32(x, rotary_dim, interleaved, cos_tab, sin_tab, pos):
    """Rotate one fp32 vector x at position pos; returns a new fp32 array."""
    x = np.ascontiguousarray(x, np.float32)
    c = np.ascontiguousarray(cos_tab, np.float32)
    s_ = np.ascontiguousarray(sin_tab, np.float32)
    y = np.zeros_like(x)
    lib().orc_rotary_f32(_ptr(x), x.size, int(rotary_dim), int(interleaved), _ptr(c), _ptr(s_), int(pos), _ptr(y))
    return y


def append_kv_rotary(p, new_dtype, k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens,
                     cos_tab, sin_tab, rotary_dim, interleaved, q=None):
    """Returns (k_pages, v_pages, q) copies after the rotary append."""
    kn, vn = raw(k_new), raw(v_new)
    k, v = raw(k_pages).copy(), raw(v_pages).copy()
    ks, vs = raw(k_scale), raw(v_scale)
    bt, sl = raw(block_table).astype(np.int32), raw(seq_lens).astype(np.int32)
    c = np.ascontiguousarray(raw(cos_tab), np.float32)
    s_ = np.ascontiguousarray(raw(sin_tab), np.float32)
    qq = None if q is None else raw(q).copy()
    rc = lib().orc_append_kv_rotary(ctypes.byref(p), int(new_dtype), _ptr(kn), _ptr(vn), _ptr(k), _ptr(v), _ptr(ks),
                                    _ptr(vs), _ptr(bt), _ptr(sl), _ptr(c), _ptr(s_), int(rotary_dim), c.shape[0],
                                    int(interleaved), _ptr(qq))
    _check(rc, "append_kv_rotary")
    return k, v, qq
