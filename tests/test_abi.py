"""Host-side checks of libfd.so: it builds for sm_103a, loads, exports every
entry point declared in include/fd_api.h, and rejects bad arguments before
any launch (no GPU is needed for any of this)."""
import ctypes
import os
import re

import pytest
import torch

from split_kv_decode_paged_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(fd_\w+)\s*\(", src, flags=re.M))
    return names


def test_library_exports_every_declared_symbol(fdlib):
    declared = _declared()
    assert {"fd_plan", "fd_decode_paged", "fd_merge_states", "fd_append_kv", "fd_status_string"} <= declared
    for name in declared:
        assert hasattr(fdlib, name), name
    assert _lib.fd_api_version() == 1


def test_status_strings(fdlib):
    for code in range(8):
        assert _lib.fd_status_string(code) not in ("", "unknown status")
    assert _lib.fd_status_from_device(0) == _lib.FD_OK
    assert _lib.fd_status_from_device(_lib.FD_DEV_BAD_PAGE) == _lib.FD_ERR_BAD_PAGE
    assert _lib.fd_status_from_device(_lib.FD_DEV_CAPACITY) == _lib.FD_ERR_CAPACITY
    assert _lib.fd_status_from_device(_lib.FD_DEV_TIMEOUT | 1) == _lib.FD_ERR_TIMEOUT


def _prob(**kw):
    base = dict(B=2, Hq=8, Hkv=2, D=128, page_size=16, max_blocks_per_seq=8, num_pages=64,
                q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16)
    base.update(kw)
    return _lib.make_problem(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(page_size=24), _lib.FD_ERR_INVALID_ARG),          # not a multiple of 16
    (dict(Hq=6, Hkv=4), _lib.FD_ERR_INVALID_ARG),           # Hq % Hkv != 0
    (dict(D=96), _lib.FD_ERR_UNSUPPORTED),
    (dict(q_dtype=torch.float16), _lib.FD_ERR_UNSUPPORTED),  # q/kv mismatch without fp8
    (dict(B=0), _lib.FD_ERR_INVALID_ARG),
    (dict(B=9000), _lib.FD_ERR_UNSUPPORTED),
])
def test_plan_rejects_bad_problems(fdlib, kw, code):
    p = _prob(**kw)
    with pytest.raises(_lib.FdError) as ei:
        _lib.fd_plan(p, [10] * p.B, num_sms=148)
    assert ei.value.code == code


def test_plan_rejects_lengths_beyond_table(fdlib):
    with pytest.raises(_lib.FdError) as ei:
        _lib.fd_plan(_prob(), [10, 16 * 8 + 1], num_sms=148)
    assert ei.value.code == _lib.FD_ERR_INVALID_ARG
    with pytest.raises(_lib.FdError):
        _lib.fd_plan(_prob(), [10, -1], num_sms=148)


def test_decode_rejects_before_launch(fdlib):
    """Argument errors come back as status codes; nothing reaches a GPU."""
    p = _prob()
    plan = _lib.fd_plan(p, [100, 50], num_sms=148)
    L = fdlib
    P = ctypes.c_void_p
    fake = P(1 << 20)  # never dereferenced: validation fails first
    # null q
    assert L.fd_decode_paged(ctypes.byref(plan), None, fake, fake, None, None, fake, fake, fake, None, fake,
                             plan.workspace_bytes, None, None) == _lib.FD_ERR_INVALID_ARG
    # misaligned k
    assert L.fd_decode_paged(ctypes.byref(plan), fake, P((1 << 20) + 8), fake, None, None, fake, fake, fake,
                             None, fake, plan.workspace_bytes, None, None) == _lib.FD_ERR_INVALID_ARG
    # workspace too small
    assert L.fd_decode_paged(ctypes.byref(plan), fake, fake, fake, None, None, fake, fake, fake, None, fake,
                             plan.workspace_bytes - 1, None, None) == _lib.FD_ERR_WORKSPACE_TOO_SMALL
    # scales given for a bf16 cache
    assert L.fd_decode_paged(ctypes.byref(plan), fake, fake, fake, fake, fake, fake, fake, fake, None, fake,
                             plan.workspace_bytes, None, None) == _lib.FD_ERR_INVALID_ARG
    # merge: S beyond the maximum
    assert L.fd_merge_states(fake, fake, fake, 1, 1, 5000, 128, _lib.FD_F32, fake, None,
                             None) == _lib.FD_ERR_UNSUPPORTED
    # append: fp8 cache without scales
    p8 = _prob(kv_dtype=torch.float8_e4m3fn)
    assert L.fd_append_kv(ctypes.byref(p8), fake, fake, fake, fake, None, None, fake, fake, None,
                          None) == _lib.FD_ERR_INVALID_ARG
