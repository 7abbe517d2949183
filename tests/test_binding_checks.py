"""The Python binding checks every tensor against the plan or problem before
it calls into libfd (the C ABI sees only pointers, so a wrong shape, dtype,
layout or device would otherwise reach a kernel).  Each mismatch raises
ValueError naming the argument; nothing is launched, so these run on CPU."""
import pytest
import torch

from split_kv_decode_paged_gb300 import _lib

B, HQ, HKV, D, PS, MB, NP = 2, 8, 2, 128, 16, 4, 12


def _plan(kv=torch.bfloat16, q=torch.bfloat16, out=None):
    prob = _lib.make_problem(B, HQ, HKV, D, PS, MB, NP, q, kv, out)
    return _lib.fd_plan(prob, [40, 50], num_sms=152)


def _args(plan, kv=torch.bfloat16, q=torch.bfloat16, out=torch.bfloat16):
    """Correctly shaped host tensors (on the host the device check fails last)."""
    fp8 = kv == torch.float8_e4m3fn
    return dict(
        q=torch.zeros((B, HQ, D), dtype=q),
        k_pages=torch.zeros((NP, PS, HKV, D), dtype=kv), v_pages=torch.zeros((NP, PS, HKV, D), dtype=kv),
        k_scale=torch.ones((NP, HKV)) if fp8 else None, v_scale=torch.ones((NP, HKV)) if fp8 else None,
        block_table=torch.zeros((B, MB), dtype=torch.int32), seq_lens=torch.zeros((B,), dtype=torch.int32),
        out=torch.zeros((B, HQ, D), dtype=out), lse=torch.zeros((B, HQ)),
        workspace=torch.zeros(max(256, plan.workspace_bytes), dtype=torch.uint8),
        status=torch.zeros(1, dtype=torch.int32))


def _decode(plan, a):
    _lib.fd_decode_paged(plan, a["q"], a["k_pages"], a["v_pages"], a["k_scale"], a["v_scale"], a["block_table"],
                         a["seq_lens"], a["out"], a["lse"], a["workspace"], a["status"])


@pytest.mark.parametrize("name,bad,msg", [
    ("q", torch.zeros((B, HQ, 64), dtype=torch.bfloat16), "shape"),
    ("q", torch.zeros((B, HQ, D), dtype=torch.float16), "dtype"),
    ("q", torch.zeros((B, D, HQ), dtype=torch.bfloat16).transpose(1, 2), "contiguous"),
    ("k_pages", torch.zeros((NP, PS, HKV * 2, D), dtype=torch.bfloat16), "shape"),
    ("v_pages", torch.zeros((NP, PS, HKV, D), dtype=torch.float16), "dtype"),
    ("k_scale", torch.ones((NP, HKV)), "must be None"),
    ("block_table", torch.zeros((B, MB), dtype=torch.int64), "dtype"),
    ("block_table", torch.zeros((B, MB + 1), dtype=torch.int32), "shape"),
    ("seq_lens", torch.zeros((B + 1,), dtype=torch.int32), "shape"),
    ("out", torch.zeros((B, HQ, D), dtype=torch.float32), "dtype"),
    ("lse", torch.zeros((B, HQ + 1)), "shape"),
    ("workspace", torch.zeros(8, dtype=torch.uint8), "at least"),
    ("status", torch.zeros(1, dtype=torch.int64), "dtype"),
    ("q", None, "required"),
])
def test_decode_rejects_mismatched_tensors(fdlib, name, bad, msg):
    plan = _plan()
    a = _args(plan)
    a[name] = bad
    with pytest.raises(ValueError, match=f"fd_decode_paged: {name} .*{msg}"):
        _decode(plan, a)


def test_decode_requires_cuda_tensors(fdlib):
    plan = _plan()
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        _decode(plan, _args(plan))


def test_decode_fp8_needs_scales_of_the_pool_shape(fdlib):
    kv = torch.float8_e4m3fn
    plan = _plan(kv=kv)
    a = _args(plan, kv=kv)
    a["v_scale"] = None
    with pytest.raises(ValueError, match="v_scale is required"):
        _decode(plan, a)
    a = _args(plan, kv=kv)
    a["k_scale"] = torch.ones((NP, HKV + 1))
    with pytest.raises(ValueError, match="k_scale must have shape"):
        _decode(plan, a)


def test_decode_fp32_output_plan(fdlib):
    plan = _plan(out=torch.float32)
    a = _args(plan)  # bf16 out, but the plan wants fp32
    with pytest.raises(ValueError, match="out must have dtype torch.float32"):
        _decode(plan, a)


def test_decode_ex_index_shapes(fdlib):
    plan = _plan()
    a = _args(plan)
    with pytest.raises(ValueError, match="cache_batch_idx must have shape"):
        _lib.fd_decode_paged_ex(plan, a["q"], a["k_pages"], a["v_pages"], None, None, a["block_table"],
                                a["seq_lens"], a["out"], a["lse"], a["workspace"],
                                cache_batch_idx=torch.zeros(B + 1, dtype=torch.int32), cache_rows=B)
    with pytest.raises(ValueError, match="block_table must have shape"):
        # three cache rows, but a table of two
        _lib.fd_decode_paged_ex(plan, a["q"], a["k_pages"], a["v_pages"], None, None, a["block_table"],
                                a["seq_lens"], a["out"], a["lse"], a["workspace"],
                                cache_batch_idx=torch.zeros(B, dtype=torch.int32), cache_rows=3)


def test_merge_states_shapes(fdlib):
    o = torch.zeros((2, 3, 4, 64))
    m = torch.zeros((2, 3, 4))
    with pytest.raises(ValueError, match="d must have shape"):
        _lib.fd_merge_states(o, m, torch.zeros((2, 3, 5)), torch.zeros((2, 3, 64)))
    with pytest.raises(ValueError, match="o_part must have dtype"):
        _lib.fd_merge_states(o.double(), m, m, torch.zeros((2, 3, 64)))
    with pytest.raises(ValueError, match="out must have shape"):
        _lib.fd_merge_states(o, m, m, torch.zeros((2, 3, 32)))
    with pytest.raises(ValueError, match="out must be a float16, bfloat16 or float32"):
        _lib.fd_merge_states(o, m, m, torch.zeros((2, 3, 64), dtype=torch.int32))
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        _lib.fd_merge_states(o, m, m, torch.zeros((2, 3, 64)))


def test_merge_two_shapes(fdlib):
    oa, la = torch.zeros((5, 64)), torch.zeros(5)
    with pytest.raises(ValueError, match="lse_b must have shape"):
        _lib.fd_merge_two(oa, la, oa.clone(), torch.zeros(4), torch.zeros((5, 64)))
    with pytest.raises(ValueError, match="out_b must have shape"):
        _lib.fd_merge_two(oa, la, torch.zeros((5, 32)), la, torch.zeros((5, 64)))


def test_append_shapes(fdlib):
    prob = _lib.make_problem(B, HKV, HKV, D, PS, MB, NP, torch.bfloat16, torch.bfloat16)
    kp = torch.zeros((NP, PS, HKV, D), dtype=torch.bfloat16)
    bt = torch.zeros((B, MB), dtype=torch.int32)
    sl = torch.zeros((B,), dtype=torch.int32)
    new = torch.zeros((B, HKV, D), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="k_new must have shape"):
        _lib.fd_append_kv(prob, torch.zeros((B, HKV + 1, D), dtype=torch.bfloat16), new, kp, kp.clone(), None, None,
                          bt, sl)
    with pytest.raises(ValueError, match="v_new must have dtype"):
        _lib.fd_append_kv(prob, new, new.half(), kp, kp.clone(), None, None, bt, sl)
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        _lib.fd_append_kv(prob, new, new.clone(), kp, kp.clone(), None, None, bt, sl)
    # E4M3 cache: new rows come in q's dtype and the scales are required
    prob8 = _lib.make_problem(B, HKV, HKV, D, PS, MB, NP, torch.bfloat16, torch.float8_e4m3fn)
    kp8 = torch.zeros((NP, PS, HKV, D), dtype=torch.float8_e4m3fn)
    with pytest.raises(ValueError, match="k_scale is required"):
        _lib.fd_append_kv(prob8, new, new.clone(), kp8, kp8.clone(), None, None, bt, sl)
    with pytest.raises(ValueError, match="rotary_sin must have shape"):
        _lib.fd_append_kv_rotary(prob, new, new.clone(), kp, kp.clone(), None, None, bt, sl, torch.zeros((10, 32)),
                                 torch.zeros((10, 16)))


def test_staged_host_step_blocks(fdlib):
    plan = _plan()
    a = _args(plan)
    lay = _lib.fd_host_io_layout_for(plan)
    with pytest.raises(ValueError, match="host_in must hold at least"):
        _lib.fd_host_copy_in(plan, torch.zeros(8, dtype=torch.uint8), torch.zeros(lay.in_bytes, dtype=torch.uint8))
    with pytest.raises(ValueError, match="dev_in must hold at least"):
        _lib.fd_decode_paged_staged(plan, torch.zeros(8, dtype=torch.uint8), a["k_pages"], a["v_pages"], None, None,
                                    torch.zeros(lay.out_bytes, dtype=torch.uint8),
                                    torch.zeros(lay.out_bytes, dtype=torch.uint8), a["workspace"])


def test_host_copy_out_blocks(fdlib):
    plan = _plan()
    lay = _lib.fd_host_io_layout_for(plan)
    with pytest.raises(ValueError, match="dev_out must hold at least"):
        _lib.fd_host_copy_out(plan, torch.zeros(8, dtype=torch.uint8), torch.zeros(lay.out_bytes, dtype=torch.uint8))
    with pytest.raises(ValueError, match="host_out must hold at least"):
        _lib.fd_host_copy_out(plan, torch.zeros(lay.out_bytes, dtype=torch.uint8), torch.zeros(8, dtype=torch.uint8))


def test_host_step_blocks(fdlib):
    plan = _plan()
    a = _args(plan)
    lay = _lib.fd_host_io_layout_for(plan)
    with pytest.raises(ValueError, match="host_in must hold at least"):
        _lib.fd_decode_paged_host(plan, torch.zeros(8, dtype=torch.uint8), torch.zeros(lay.in_bytes,
                                  dtype=torch.uint8), a["k_pages"], a["v_pages"], None, None,
                                  torch.zeros(lay.out_bytes, dtype=torch.uint8), torch.zeros(lay.out_bytes,
                                  dtype=torch.uint8), a["workspace"])
