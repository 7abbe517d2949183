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
    assert _lib.fd_api_version() == 5


def _declared_arg_counts():
    counts = {}
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            for name, args in re.findall(r"^[A-Za-z_][\w\s\*]*?\b(fd_\w+)\s*\(([^)]*)\)\s*;", src, flags=re.M | re.S):
                args = args.strip()
                counts[name] = 0 if args in ("", "void") else args.count(",") + 1
    return counts


def test_binding_argument_counts_match_the_header(fdlib):
    """Every entry point the binding declares argtypes for takes as many
    arguments as its declaration in include/fd_api.h (a missing or extra
    argument would shift every pointer after it)."""
    counts = _declared_arg_counts()
    lib = _lib.load()
    checked = 0
    for name, n in counts.items():
        fn = getattr(lib, name)
        if fn.argtypes is None:
            continue
        assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)
        checked += 1
    assert checked >= 12


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
    # a plan whose shared memory does not hold its layout, or whose scratch
    # placement the shape cannot take
    for field, value in (("smem_bytes", plan.smem_bytes // 2), ("scratch_in_stage", 2)):
        bad = _lib.FdPlan.from_buffer_copy(plan)
        setattr(bad, field, value)
        assert L.fd_decode_paged(ctypes.byref(bad), fake, fake, fake, None, None, fake, fake, fake, None, fake,
                                 plan.workspace_bytes, None, None) == _lib.FD_ERR_INVALID_ARG, field
    p8 = _prob(kv_dtype=torch.float8_e4m3fn)
    plan8 = _lib.fd_plan(p8, [100, 50], num_sms=148, ctas_per_sm=1)  # one CTA per SM, 8 consumer warps
    assert plan8.scratch_in_stage == 0
    plan8.scratch_in_stage = 1  # only the two-CTA E4M3 shape keeps its scratch in a stage
    assert L.fd_decode_paged(ctypes.byref(plan8), fake, fake, fake, fake, fake, fake, fake, fake, None, fake,
                             plan8.workspace_bytes, None, None) == _lib.FD_ERR_INVALID_ARG
    # merge: S beyond the maximum
    assert L.fd_merge_states(fake, fake, fake, 1, 1, 5000, 128, _lib.FD_F32, fake, None,
                             None) == _lib.FD_ERR_UNSUPPORTED
    # append: fp8 cache without scales
    assert L.fd_append_kv(ctypes.byref(p8), fake, fake, fake, fake, None, None, fake, fake, None,
                          None) == _lib.FD_ERR_INVALID_ARG


def test_struct_layouts_match_the_header(tmp_path):
    """The ctypes mirrors of fd_problem, fd_plan_options, fd_plan_t and
    fd_host_io_layout have the C structs' sizes and field offsets (checked
    against the header compiled by the host C compiler)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    structs = {"fd_problem": _lib.FdProblem, "fd_plan_options": _lib.FdPlanOptions, "fd_plan_t": _lib.FdPlan,
               "fd_host_io_layout": _lib.FdHostIoLayout}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "fd_api.h"', 'int main(void) {']
    for cname, py in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    for line in filter(None, got):
        cname, fname, val = line.split()
        py = structs[cname]
        want = ctypes.sizeof(py) if fname == "size" else getattr(py, fname).offset
        assert int(val) == want, (cname, fname, int(val), want)


@pytest.mark.parametrize("kw", [dict(timeout_us=-1), dict(debug_stall_us=10), dict(debug_stall_role=1),
                                dict(debug_stall_role=3, debug_stall_us=10),
                                dict(debug_stall_role=1, debug_stall_us=2000000)])
def test_plan_rejects_bad_timeout_options(fdlib, kw):
    with pytest.raises(_lib.FdError) as ei:
        _lib.fd_plan(_prob(), [10, 20], num_sms=148, **kw)
    assert ei.value.code == _lib.FD_ERR_INVALID_ARG


def test_plan_carries_timeout_options(fdlib):
    plan = _lib.fd_plan(_prob(), [10, 20], num_sms=148, timeout_us=300, debug_stall_us=5000, debug_stall_role=2)
    assert (plan.timeout_us, plan.debug_stall_us, plan.debug_stall_role) == (300, 5000, 2)
    plan = _lib.fd_plan(_prob(), [10, 20], num_sms=148)
    assert (plan.timeout_us, plan.debug_stall_us, plan.debug_stall_role) == (0, 0, 0)
