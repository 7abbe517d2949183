"""ctypes binding of libfd.so (include/fd_api.h).  Argument marshalling only.

Each function keeps the name of the C entry point it calls (fd_plan,
fd_decode_paged, fd_decode_paged_ex, fd_decode_paged_host, fd_merge_states,
fd_merge_two, fd_append_kv, fd_append_kv_rotary, ...).  Tensors are passed by
data_ptr(); the stream is torch's current CUDA stream unless given.  No
computation happens here and there is no fallback: if libfd.so is missing or
fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfd.so")

FD_OK, FD_ERR_INVALID_ARG, FD_ERR_UNSUPPORTED, FD_ERR_WORKSPACE_TOO_SMALL = 0, 1, 2, 3
FD_ERR_BAD_PAGE, FD_ERR_CUDA, FD_ERR_CAPACITY, FD_ERR_TIMEOUT = 4, 5, 6, 7
FD_DEV_BAD_PAGE, FD_DEV_CAPACITY, FD_DEV_TIMEOUT = 0x1, 0x2, 0x4
FD_F16, FD_BF16, FD_E4M3, FD_F32 = 0, 1, 2, 3

_TORCH_TO_FD = {torch.float16: FD_F16, torch.bfloat16: FD_BF16, torch.float8_e4m3fn: FD_E4M3,
                torch.float32: FD_F32}
FD_TO_TORCH = {v: k for k, v in _TORCH_TO_FD.items()}


def fd_dtype(t) -> int:
    if isinstance(t, int):
        return t
    return _TORCH_TO_FD[t]


class FdError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {fd_status_string(code)} (status {code})")


class FdProblem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int), ("D", ctypes.c_int),
                ("page_size", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int), ("num_pages", ctypes.c_int),
                ("q_dtype", ctypes.c_int), ("kv_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int)]


class FdPlanOptions(ctypes.Structure):
    _fields_ = [("num_splits", ctypes.c_int), ("num_sms", ctypes.c_int), ("fuse_merge", ctypes.c_int),
                ("max_seq_len", ctypes.c_int), ("ctas_per_sm", ctypes.c_int), ("split_margin_pct", ctypes.c_int),
                ("tile_tokens", ctypes.c_int), ("shared_kv", ctypes.c_int)]


class FdDecodeExtras(ctypes.Structure):
    _fields_ = [("cache_batch_idx", ctypes.c_void_p), ("cache_leftpad", ctypes.c_void_p),
                ("cache_rows", ctypes.c_int)]


class FdPlan(ctypes.Structure):
    _fields_ = [("problem", FdProblem), ("num_splits", ctypes.c_int), ("chunk_tokens", ctypes.c_int),
                ("tile_tokens", ctypes.c_int), ("capacity_tokens", ctypes.c_int), ("grid_ctas", ctypes.c_int),
                ("num_sms", ctypes.c_int), ("fuse_merge", ctypes.c_int), ("stages", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t),
                ("ws_partial_o", ctypes.c_size_t), ("ws_partial_md", ctypes.c_size_t),
                ("ws_counters", ctypes.c_size_t), ("work_items_hint", ctypes.c_longlong),
                ("kv_rows", ctypes.c_int), ("row_fold", ctypes.c_int), ("head_subgroups", ctypes.c_int),
                ("reserved", ctypes.c_int * 5)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_ if n not in ("problem", "reserved")}


class FdHostIoLayout(ctypes.Structure):
    _fields_ = [("q_offset", ctypes.c_size_t), ("block_table_offset", ctypes.c_size_t),
                ("seq_lens_offset", ctypes.c_size_t), ("in_bytes", ctypes.c_size_t),
                ("out_offset", ctypes.c_size_t), ("lse_offset", ctypes.c_size_t), ("out_bytes", ctypes.c_size_t)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libfd.so (built by split_kv_decode_paged_gb300.build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libfd.so not found at {path}; build it with split_kv_decode_paged_gb300.build.build()")
    L = ctypes.CDLL(path)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.fd_plan.restype = I
    L.fd_plan.argtypes = [ctypes.POINTER(FdProblem), P, ctypes.POINTER(FdPlanOptions), ctypes.POINTER(FdPlan)]
    L.fd_decode_paged.restype = I
    L.fd_decode_paged.argtypes = [ctypes.POINTER(FdPlan), P, P, P, P, P, P, P, P, P, P, S, P, P]
    L.fd_decode_paged_ex.restype = I
    L.fd_decode_paged_ex.argtypes = [ctypes.POINTER(FdPlan), P, P, P, P, P, P, P, ctypes.POINTER(FdDecodeExtras),
                                     P, P, P, S, P, P]
    L.fd_merge_states.restype = I
    L.fd_merge_states.argtypes = [P, P, P, I, I, I, I, I, P, P, P]
    L.fd_append_kv.restype = I
    L.fd_append_kv.argtypes = [ctypes.POINTER(FdProblem), P, P, P, P, P, P, P, P, P, P]
    L.fd_append_kv_rotary.restype = I
    L.fd_append_kv_rotary.argtypes = [ctypes.POINTER(FdProblem), P, P, P, P, P, P, P, P, P, P, I, I, I, P, P, P]
    L.fd_merge_two.restype = I
    L.fd_merge_two.argtypes = [P, P, P, P, I, I, I, P, P, P]
    L.fd_host_io_layout_for.restype = I
    L.fd_host_io_layout_for.argtypes = [ctypes.POINTER(FdPlan), ctypes.POINTER(FdHostIoLayout)]
    L.fd_decode_paged_host.restype = I
    L.fd_decode_paged_host.argtypes = [ctypes.POINTER(FdPlan), P, P, P, P, P, P, P, P, P, S, P, P]
    L.fd_status_string.restype = ctypes.c_char_p
    L.fd_status_string.argtypes = [I]
    L.fd_status_from_device.restype = I
    L.fd_status_from_device.argtypes = [ctypes.c_int32]
    L.fd_api_version.restype = I
    L.fd_api_version.argtypes = []
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def fd_status_string(code: int) -> str:
    return load().fd_status_string(int(code)).decode()


def fd_status_from_device(word: int) -> int:
    return load().fd_status_from_device(int(word))


def fd_api_version() -> int:
    return load().fd_api_version()


def make_problem(B, Hq, Hkv, D, page_size, max_blocks_per_seq, num_pages, q_dtype, kv_dtype, out_dtype=None):
    q = fd_dtype(q_dtype)
    return FdProblem(B, Hq, Hkv, D, page_size, max_blocks_per_seq, num_pages, q, fd_dtype(kv_dtype),
                     q if out_dtype is None else fd_dtype(out_dtype))


def fd_plan(problem: FdProblem, seq_lens_host, num_splits=0, num_sms=0, fuse_merge=1, max_seq_len=0,
            ctas_per_sm=0, split_margin_pct=0, tile_tokens=0, shared_kv=0) -> FdPlan:
    """Plan a decode call; seq_lens_host is a host int32 tensor/sequence."""
    lens = torch.as_tensor(seq_lens_host, dtype=torch.int32).cpu().contiguous()
    if lens.numel() != problem.B and not (shared_kv and lens.numel() >= 1):
        raise ValueError("seq_lens_host must have B entries")
    opts = FdPlanOptions(int(num_splits), int(num_sms), int(fuse_merge), int(max_seq_len), int(ctas_per_sm),
                         int(split_margin_pct), int(tile_tokens), int(shared_kv))
    plan = FdPlan()
    rc = load().fd_plan(ctypes.byref(problem), ctypes.c_void_p(lens.data_ptr()), ctypes.byref(opts),
                        ctypes.byref(plan))
    if rc != FD_OK:
        raise FdError(rc, "fd_plan")
    return plan


def fd_decode_paged(plan: FdPlan, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, out, lse,
                    workspace, status=None, stream=None):
    rc = load().fd_decode_paged(ctypes.byref(plan), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(k_scale),
                                _ptr(v_scale), _ptr(block_table), _ptr(seq_lens), _ptr(out), _ptr(lse),
                                _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                _ptr(status), _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_decode_paged")


def fd_decode_paged_ex(plan: FdPlan, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, out, lse,
                       workspace, cache_batch_idx=None, cache_leftpad=None, cache_rows=0, status=None, stream=None):
    ex = FdDecodeExtras(None if cache_batch_idx is None else cache_batch_idx.data_ptr(),
                        None if cache_leftpad is None else cache_leftpad.data_ptr(), int(cache_rows))
    rc = load().fd_decode_paged_ex(ctypes.byref(plan), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(k_scale),
                                   _ptr(v_scale), _ptr(block_table), _ptr(seq_lens), ctypes.byref(ex), _ptr(out),
                                   _ptr(lse), _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                   _ptr(status), _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_decode_paged_ex")


def fd_merge_states(o_part, m, d, out, lse=None, stream=None):
    """o_part [B,Hq,S,D] fp32, m/d [B,Hq,S] fp32 -> out [B,Hq,D], lse [B,Hq]."""
    B, Hq, S, D = o_part.shape
    rc = load().fd_merge_states(_ptr(o_part), _ptr(m), _ptr(d), B, Hq, S, D, fd_dtype(out.dtype), _ptr(out),
                                _ptr(lse), _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_merge_states")


def fd_append_kv(problem: FdProblem, k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens,
                 status=None, stream=None):
    rc = load().fd_append_kv(ctypes.byref(problem), _ptr(k_new), _ptr(v_new), _ptr(k_pages), _ptr(v_pages),
                             _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(seq_lens), _ptr(status),
                             _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_append_kv")


def fd_append_kv_rotary(problem: FdProblem, k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table,
                        seq_lens, rotary_cos, rotary_sin, interleaved=False, q_inout=None, status=None,
                        stream=None):
    """rotary_cos/sin: fp32 [max_pos, rotary_dim/2] on the device."""
    max_pos, half = rotary_cos.shape
    rc = load().fd_append_kv_rotary(ctypes.byref(problem), _ptr(k_new), _ptr(v_new), _ptr(k_pages), _ptr(v_pages),
                                    _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(seq_lens),
                                    _ptr(rotary_cos), _ptr(rotary_sin), 2 * half, max_pos, int(bool(interleaved)),
                                    _ptr(q_inout), _ptr(status), _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_append_kv_rotary")


def fd_merge_two(out_a, lse_a, out_b, lse_b, out, lse=None, stream=None):
    """out_a/out_b fp32 [..., D], lse_a/lse_b fp32 [...] -> out [..., D], lse."""
    D = out_a.shape[-1]
    rows = out_a.numel() // D
    rc = load().fd_merge_two(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b), rows, D, fd_dtype(out.dtype),
                             _ptr(out), _ptr(lse), _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_merge_two")


def fd_host_io_layout_for(plan: FdPlan) -> FdHostIoLayout:
    lay = FdHostIoLayout()
    rc = load().fd_host_io_layout_for(ctypes.byref(plan), ctypes.byref(lay))
    if rc != FD_OK:
        raise FdError(rc, "fd_host_io_layout_for")
    return lay


def fd_decode_paged_host(plan: FdPlan, host_in, dev_in, k_pages, v_pages, k_scale, v_scale, dev_out, host_out,
                         workspace, status=None, stream=None):
    rc = load().fd_decode_paged_host(ctypes.byref(plan), _ptr(host_in), _ptr(dev_in), _ptr(k_pages), _ptr(v_pages),
                                     _ptr(k_scale), _ptr(v_scale), _ptr(dev_out), _ptr(host_out), _ptr(workspace),
                                     int(workspace.numel() * workspace.element_size()), _ptr(status),
                                     _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_decode_paged_host")
