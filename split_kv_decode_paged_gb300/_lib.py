"""ctypes binding of libfd.so (include/fd_api.h).  Argument marshalling only.

Each function keeps the name of the C entry point it calls (fd_plan,
fd_decode_paged, fd_decode_paged_ex, fd_decode_paged_host, fd_host_copy_in,
fd_decode_paged_staged, fd_host_copy_out, fd_merge_states,
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
                ("tile_tokens", ctypes.c_int), ("shared_kv", ctypes.c_int), ("timeout_us", ctypes.c_int),
                ("debug_stall_us", ctypes.c_int), ("debug_stall_role", ctypes.c_int), ("q_len", ctypes.c_int)]


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
                ("ctas_per_sm", ctypes.c_int), ("timeout_us", ctypes.c_int), ("debug_stall_us", ctypes.c_int),
                ("debug_stall_role", ctypes.c_int), ("q_len", ctypes.c_int), ("scratch_in_stage", ctypes.c_int),
                ("reserved", ctypes.c_int * 2)]

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
    L.fd_host_copy_in.restype = I
    L.fd_host_copy_in.argtypes = [ctypes.POINTER(FdPlan), P, P, P]
    L.fd_decode_paged_staged.restype = I
    L.fd_decode_paged_staged.argtypes = [ctypes.POINTER(FdPlan), P, P, P, P, P, P, P, P, S, P, P]
    L.fd_host_copy_out.restype = I
    L.fd_host_copy_out.argtypes = [ctypes.POINTER(FdPlan), P, P, P]
    L.fd_status_string.restype = ctypes.c_char_p
    L.fd_status_string.argtypes = [I]
    L.fd_status_from_device.restype = I
    L.fd_status_from_device.argtypes = [ctypes.c_int32]
    L.fd_api_version.restype = I
    L.fd_api_version.argtypes = []
    _lib = L
    return L


def _ptr(t):
    # a plain int (or None): ctypes converts it for the c_void_p argument
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class _Args:
    """Checks of the tensors handed to one entry point against the shapes and
    dtypes the C ABI expects (the ABI sees only pointers).  Every failure
    raises ValueError before anything is launched.  Shapes, dtypes and
    layout are checked as each tensor is named; placement last (done()):
    device tensors must all sit on one CUDA device, host blocks on the CPU."""

    def __init__(self, entry):
        self.entry = entry
        self.placed = []

    def _fail(self, name, what):
        raise ValueError(f"{self.entry}: {name} {what}")

    def tensor(self, name, t, dtype=None, shape=None, min_bytes=None, host=False, optional=False):
        if t is None:
            if optional:
                return
            self._fail(name, "is required")
        if not isinstance(t, torch.Tensor):
            self._fail(name, f"must be a torch.Tensor, got {type(t).__name__}")
        if dtype is not None and t.dtype != dtype:
            self._fail(name, f"must have dtype {dtype}, got {t.dtype}")
        if shape is not None and t.shape != shape:  # torch.Size compares equal to a tuple
            self._fail(name, f"must have shape {tuple(shape)}, got {tuple(t.shape)}")
        if not t.is_contiguous():
            self._fail(name, "must be contiguous")
        if min_bytes is not None and t.nbytes < min_bytes:
            self._fail(name, f"must hold at least {min_bytes} bytes, got {t.nbytes}")
        self.placed.append((name, t, host))

    def absent(self, name, t, why):
        if t is not None:
            self._fail(name, f"must be None ({why})")

    def done(self):
        index = None
        for name, t, host in self.placed:
            if host:
                if not t.is_cpu:
                    self._fail(name, f"must be a host (CPU) tensor, got {t.device}")
                continue
            if not t.is_cuda:
                self._fail(name, f"must be a CUDA tensor, got {t.device}")
            if index is None:
                index, first = t.get_device(), t
            elif t.get_device() != index:
                self._fail(name, f"is on {t.device}, other arguments on {first.device}")


def _rows_shape(plan, t, tail):
    """Query-row tensors are [rows, *tail]; with several query tokens per
    sequence also [B, q_len, *tail] (the same memory)."""
    p = plan.problem
    flat = (p.B,) + tail
    if t is not None and t.dim() == len(tail) + 2 and plan.row_fold == max(1, plan.q_len):
        return (plan.kv_rows, max(1, plan.q_len)) + tail
    return flat


def _check_decode(entry, plan, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, out, lse, workspace,
                  status, table_rows=None, host_io=False):
    p = plan.problem
    a = _Args(entry)
    kv = FD_TO_TORCH[p.kv_dtype]
    pool = (p.num_pages, p.page_size, p.Hkv, p.D)
    rows = table_rows if table_rows is not None else (plan.kv_rows if plan.kv_rows > 0 else p.B)
    if not host_io:
        a.tensor("q", q, FD_TO_TORCH[p.q_dtype], _rows_shape(plan, q, (p.Hq, p.D)))
        a.tensor("block_table", block_table, torch.int32, (rows, p.max_blocks_per_seq))
        a.tensor("seq_lens", seq_lens, torch.int32, (rows,))
        a.tensor("out", out, FD_TO_TORCH[p.out_dtype], _rows_shape(plan, out, (p.Hq, p.D)))
        a.tensor("lse", lse, torch.float32, _rows_shape(plan, lse, (p.Hq,)), optional=True)
    a.tensor("k_pages", k_pages, kv, pool)
    a.tensor("v_pages", v_pages, kv, pool)
    if p.kv_dtype == FD_E4M3:
        a.tensor("k_scale", k_scale, torch.float32, (p.num_pages, p.Hkv))
        a.tensor("v_scale", v_scale, torch.float32, (p.num_pages, p.Hkv))
    else:
        a.absent("k_scale", k_scale, "the cache is not E4M3")
        a.absent("v_scale", v_scale, "the cache is not E4M3")
    a.tensor("workspace", workspace, None, None, min_bytes=int(plan.workspace_bytes))
    a.tensor("status", status, torch.int32, None, min_bytes=4, optional=True)
    return a


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
            ctas_per_sm=0, split_margin_pct=0, tile_tokens=0, shared_kv=0, timeout_us=0, debug_stall_us=0,
            debug_stall_role=0, q_len=0) -> FdPlan:
    """Plan a decode call; seq_lens_host is a host int32 tensor/sequence.
    timeout_us bounds every device-side wait (0 = 2 s); debug_stall_us and
    debug_stall_role are the test hook of the timeout path (0 = off); q_len
    > 1 plans q_len causal query tokens per sequence (q [B, q_len, Hq, D])."""
    lens = torch.as_tensor(seq_lens_host, dtype=torch.int32).cpu().contiguous()
    if lens.numel() != problem.B and not (shared_kv and lens.numel() >= 1):
        raise ValueError("seq_lens_host must have B entries")
    opts = FdPlanOptions(int(num_splits), int(num_sms), int(fuse_merge), int(max_seq_len), int(ctas_per_sm),
                         int(split_margin_pct), int(tile_tokens), int(shared_kv), int(timeout_us),
                         int(debug_stall_us), int(debug_stall_role), int(q_len))
    plan = FdPlan()
    rc = load().fd_plan(ctypes.byref(problem), ctypes.c_void_p(lens.data_ptr()), ctypes.byref(opts),
                        ctypes.byref(plan))
    if rc != FD_OK:
        raise FdError(rc, "fd_plan")
    return plan


def fd_decode_paged(plan: FdPlan, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, out, lse,
                    workspace, status=None, stream=None):
    _check_decode("fd_decode_paged", plan, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, out, lse,
                  workspace, status).done()
    rc = load().fd_decode_paged(ctypes.byref(plan), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(k_scale),
                                _ptr(v_scale), _ptr(block_table), _ptr(seq_lens), _ptr(out), _ptr(lse),
                                _ptr(workspace), workspace.nbytes,
                                _ptr(status), _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_decode_paged")


def fd_decode_paged_ex(plan: FdPlan, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, out, lse,
                       workspace, cache_batch_idx=None, cache_leftpad=None, cache_rows=0, status=None, stream=None):
    p = plan.problem
    rows = int(cache_rows) if cache_batch_idx is not None else (plan.kv_rows if plan.kv_rows > 0 else p.B)
    a = _check_decode("fd_decode_paged_ex", plan, q, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, out,
                      lse, workspace, status, table_rows=rows)
    a.tensor("cache_batch_idx", cache_batch_idx, torch.int32, (p.B,), optional=True)
    a.tensor("cache_leftpad", cache_leftpad, torch.int32, (rows,), optional=True)
    a.done()
    ex = FdDecodeExtras(None if cache_batch_idx is None else cache_batch_idx.data_ptr(),
                        None if cache_leftpad is None else cache_leftpad.data_ptr(), int(cache_rows))
    rc = load().fd_decode_paged_ex(ctypes.byref(plan), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(k_scale),
                                   _ptr(v_scale), _ptr(block_table), _ptr(seq_lens), ctypes.byref(ex), _ptr(out),
                                   _ptr(lse), _ptr(workspace), workspace.nbytes,
                                   _ptr(status), _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_decode_paged_ex")


def fd_merge_states(o_part, m, d, out, lse=None, stream=None):
    """o_part [B,Hq,S,D] fp32, m/d [B,Hq,S] fp32 -> out [B,Hq,D], lse [B,Hq]."""
    a = _Args("fd_merge_states")
    a.tensor("o_part", o_part, torch.float32)
    if o_part.dim() != 4:
        a._fail("o_part", f"must be 4-D [B, Hq, S, D], got shape {tuple(o_part.shape)}")
    B, Hq, S, D = o_part.shape
    a.tensor("m", m, torch.float32, (B, Hq, S))
    a.tensor("d", d, torch.float32, (B, Hq, S))
    if out is None or out.dtype not in (torch.float16, torch.bfloat16, torch.float32):
        a._fail("out", "must be a float16, bfloat16 or float32 tensor")
    a.tensor("out", out, None, (B, Hq, D))
    a.tensor("lse", lse, torch.float32, (B, Hq), optional=True)
    a.done()
    rc = load().fd_merge_states(_ptr(o_part), _ptr(m), _ptr(d), B, Hq, S, D, fd_dtype(out.dtype), _ptr(out),
                                _ptr(lse), _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_merge_states")


def _check_append(entry, p, k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens, status):
    a = _Args(entry)
    kv = FD_TO_TORCH[p.kv_dtype]
    new = FD_TO_TORCH[p.q_dtype] if p.kv_dtype == FD_E4M3 else kv
    a.tensor("k_new", k_new, new, (p.B, p.Hkv, p.D))
    a.tensor("v_new", v_new, new, (p.B, p.Hkv, p.D))
    pool = (p.num_pages, p.page_size, p.Hkv, p.D)
    a.tensor("k_pages", k_pages, kv, pool)
    a.tensor("v_pages", v_pages, kv, pool)
    if p.kv_dtype == FD_E4M3:
        a.tensor("k_scale", k_scale, torch.float32, (p.num_pages, p.Hkv))
        a.tensor("v_scale", v_scale, torch.float32, (p.num_pages, p.Hkv))
    else:
        a.absent("k_scale", k_scale, "the cache is not E4M3")
        a.absent("v_scale", v_scale, "the cache is not E4M3")
    a.tensor("block_table", block_table, torch.int32, (p.B, p.max_blocks_per_seq))
    a.tensor("seq_lens", seq_lens, torch.int32, (p.B,))
    a.tensor("status", status, torch.int32, None, min_bytes=4, optional=True)
    return a


def fd_append_kv(problem: FdProblem, k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens,
                 status=None, stream=None):
    _check_append("fd_append_kv", problem, k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table, seq_lens,
                  status).done()
    rc = load().fd_append_kv(ctypes.byref(problem), _ptr(k_new), _ptr(v_new), _ptr(k_pages), _ptr(v_pages),
                             _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(seq_lens), _ptr(status),
                             _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_append_kv")


def fd_append_kv_rotary(problem: FdProblem, k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table,
                        seq_lens, rotary_cos, rotary_sin, interleaved=False, q_inout=None, status=None,
                        stream=None):
    """rotary_cos/sin: fp32 [max_pos, rotary_dim/2] on the device."""
    a = _check_append("fd_append_kv_rotary", problem, k_new, v_new, k_pages, v_pages, k_scale, v_scale, block_table,
                      seq_lens, status)
    a.tensor("rotary_cos", rotary_cos, torch.float32)
    if rotary_cos.dim() != 2:
        a._fail("rotary_cos", f"must be 2-D [max_pos, rotary_dim / 2], got shape {tuple(rotary_cos.shape)}")
    a.tensor("rotary_sin", rotary_sin, torch.float32, tuple(rotary_cos.shape))
    a.tensor("q_inout", q_inout, FD_TO_TORCH[problem.q_dtype], (problem.B, problem.Hq, problem.D), optional=True)
    a.done()
    max_pos, half = rotary_cos.shape
    rc = load().fd_append_kv_rotary(ctypes.byref(problem), _ptr(k_new), _ptr(v_new), _ptr(k_pages), _ptr(v_pages),
                                    _ptr(k_scale), _ptr(v_scale), _ptr(block_table), _ptr(seq_lens),
                                    _ptr(rotary_cos), _ptr(rotary_sin), 2 * half, max_pos, int(bool(interleaved)),
                                    _ptr(q_inout), _ptr(status), _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_append_kv_rotary")


def fd_merge_two(out_a, lse_a, out_b, lse_b, out, lse=None, stream=None):
    """out_a/out_b fp32 [..., D], lse_a/lse_b fp32 [...] -> out [..., D], lse."""
    a = _Args("fd_merge_two")
    a.tensor("out_a", out_a, torch.float32)
    if out_a.dim() < 1:
        a._fail("out_a", "must have a last dimension D")
    a.tensor("out_b", out_b, torch.float32, tuple(out_a.shape))
    a.tensor("lse_a", lse_a, torch.float32, tuple(out_a.shape[:-1]))
    a.tensor("lse_b", lse_b, torch.float32, tuple(out_a.shape[:-1]))
    if out is None or out.dtype not in (torch.float16, torch.bfloat16, torch.float32):
        a._fail("out", "must be a float16, bfloat16 or float32 tensor")
    a.tensor("out", out, None, tuple(out_a.shape))
    a.tensor("lse", lse, torch.float32, tuple(out_a.shape[:-1]), optional=True)
    a.done()
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
    lay = fd_host_io_layout_for(plan)
    a = _check_decode("fd_decode_paged_host", plan, None, k_pages, v_pages, k_scale, v_scale, None, None, None,
                      None, workspace, status, host_io=True)
    a.tensor("host_in", host_in, None, None, min_bytes=int(lay.in_bytes), host=True)
    a.tensor("host_out", host_out, None, None, min_bytes=int(lay.out_bytes), host=True)
    a.tensor("dev_in", dev_in, None, None, min_bytes=int(lay.in_bytes))
    a.tensor("dev_out", dev_out, None, None, min_bytes=int(lay.out_bytes))
    a.done()
    rc = load().fd_decode_paged_host(ctypes.byref(plan), _ptr(host_in), _ptr(dev_in), _ptr(k_pages), _ptr(v_pages),
                                     _ptr(k_scale), _ptr(v_scale), _ptr(dev_out), _ptr(host_out), _ptr(workspace),
                                     workspace.nbytes, _ptr(status),
                                     _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_decode_paged_host")


def fd_host_copy_in(plan: FdPlan, host_in, dev_in, stream=None):
    lay = fd_host_io_layout_for(plan)
    a = _Args("fd_host_copy_in")
    a.tensor("host_in", host_in, None, None, min_bytes=int(lay.in_bytes), host=True)
    a.tensor("dev_in", dev_in, None, None, min_bytes=int(lay.in_bytes))
    a.done()
    rc = load().fd_host_copy_in(ctypes.byref(plan), _ptr(host_in), _ptr(dev_in), _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_host_copy_in")


def fd_decode_paged_staged(plan: FdPlan, dev_in, k_pages, v_pages, k_scale, v_scale, dev_out, host_out, workspace,
                           status=None, stream=None):
    lay = fd_host_io_layout_for(plan)
    a = _check_decode("fd_decode_paged_staged", plan, None, k_pages, v_pages, k_scale, v_scale, None, None, None,
                      None, workspace, status, host_io=True)
    a.tensor("dev_in", dev_in, None, None, min_bytes=int(lay.in_bytes))
    a.tensor("host_out", host_out, None, None, min_bytes=int(lay.out_bytes), host=True, optional=True)
    a.tensor("dev_out", dev_out, None, None, min_bytes=int(lay.out_bytes))
    a.done()
    rc = load().fd_decode_paged_staged(ctypes.byref(plan), _ptr(dev_in), _ptr(k_pages), _ptr(v_pages), _ptr(k_scale),
                                       _ptr(v_scale), _ptr(dev_out), _ptr(host_out), _ptr(workspace),
                                       workspace.nbytes, _ptr(status),
                                       _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_decode_paged_staged")


def fd_host_copy_out(plan: FdPlan, dev_out, host_out, stream=None):
    lay = fd_host_io_layout_for(plan)
    a = _Args("fd_host_copy_out")
    a.tensor("dev_out", dev_out, None, None, min_bytes=int(lay.out_bytes))
    a.tensor("host_out", host_out, None, None, min_bytes=int(lay.out_bytes), host=True)
    a.done()
    rc = load().fd_host_copy_out(ctypes.byref(plan), _ptr(dev_out), _ptr(host_out), _stream(stream))
    if rc != FD_OK:
        raise FdError(rc, "fd_host_copy_out")
