"""Pins for the oracle's rotary embedding ("Inference Cookbook" §3.4):
identity and quarter-turn angles, the complex-multiplication form in fp64,
the interleaved/half-split permutation identity, pass-through of elements
past rotary_dim, and the rotary append against torch's roundings."""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc


def _tables(max_pos, half, base=10000.0):
    inv = 1.0 / base ** (np.arange(half) / half)
    ang = np.arange(max_pos)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def test_zero_angle_is_identity_and_quarter_turn_swaps():
    x = np.random.default_rng(0).standard_normal(64).astype(np.float32)
    c = np.ones((1, 32), np.float32); s = np.zeros((1, 32), np.float32)
    assert np.array_equal(orc.rotary_f32(x, 64, 0, c, s, 0), x)
    y = orc.rotary_f32(x, 64, 0, np.zeros((1, 32), np.float32), np.ones((1, 32), np.float32), 0)
    assert np.array_equal(y[:32], -x[32:]) and np.array_equal(y[32:], x[:32])


@pytest.mark.parametrize("interleaved", [0, 1])
def test_matches_complex_rotation(interleaved):
    rng = np.random.default_rng(1)
    c, s = _tables(50, 16)
    for pos in (0, 7, 49):
        x = rng.standard_normal(48).astype(np.float32)
        y = orc.rotary_f32(x, 32, interleaved, c, s, pos)
        i1 = np.arange(0, 32, 2) if interleaved else np.arange(16)
        i2 = i1 + 1 if interleaved else i1 + 16
        z = (x[i1].astype(np.float64) + 1j * x[i2]) * (c[pos].astype(np.float64) + 1j * s[pos])
        bound = 4 * 2.0 ** -24 * (np.abs(x[i1]) + np.abs(x[i2]))
        assert np.all(np.abs(y[i1] - z.real) <= bound) and np.all(np.abs(y[i2] - z.imag) <= bound)
        assert np.array_equal(y[32:], x[32:])  # past rotary_dim: unchanged


def test_interleaved_is_half_split_under_permutation():
    rng = np.random.default_rng(2)
    c, s = _tables(10, 32)
    x = rng.standard_normal(64).astype(np.float32)
    perm = np.concatenate([np.arange(0, 64, 2), np.arange(1, 64, 2)])  # pairs (2i,2i+1) -> (i, i+32)
    y_int = orc.rotary_f32(x, 64, 1, c, s, 5)
    y_half = orc.rotary_f32(x[perm], 64, 0, c, s, 5)
    assert np.array_equal(y_int[perm], y_half)


@pytest.mark.parametrize("kv", ["bf16", "f16", "e4m3"])
def test_rotary_append_vs_torch_rounding(kv):
    rng = np.random.default_rng(3)
    B, Hq, Hkv, D, ps, rd = 2, 4, 2, 64, 16, 48
    num_pages = 6
    bt = np.array([[0, 1], [2, 3]], np.int32)
    lens = np.array([5, 20], np.int32)
    dt = {"bf16": torch.bfloat16, "f16": torch.float16, "e4m3": torch.float8_e4m3fn}[kv]
    qdt = torch.bfloat16 if kv != "f16" else torch.float16
    kp = torch.zeros((num_pages, ps, Hkv, D), dtype=torch.uint8 if kv == "e4m3" else dt)
    vp = torch.zeros_like(kp)
    if kv == "e4m3":
        kp = kp.view(torch.float8_e4m3fn); vp = vp.view(torch.float8_e4m3fn)
    ks = np.full((num_pages, Hkv), 0.02, np.float32) if kv == "e4m3" else None
    vs = ks
    kn = torch.from_numpy(rng.standard_normal((B, Hkv, D)).astype(np.float32)).to(qdt)
    vn = torch.from_numpy(rng.standard_normal((B, Hkv, D)).astype(np.float32)).to(qdt)
    q = torch.from_numpy(rng.standard_normal((B, Hq, D)).astype(np.float32)).to(qdt)
    c, s = _tables(64, rd // 2)
    code = {"bf16": orc.BF16, "f16": orc.F16, "e4m3": orc.E4M3}[kv]
    qcode = orc.BF16 if qdt == torch.bfloat16 else orc.F16
    p = orc.problem(B, Hq, Hkv, D, ps, 2, num_pages, qcode, code)
    k2, v2, q2 = orc.append_kv_rotary(p, qcode, kn, vn, kp, vp, ks, vs, bt, lens, c, s, rd, 0, q)
    for b in range(B):
        page, slot = bt[b, lens[b] // ps], lens[b] % ps
        for h in range(Hkv):
            yk = orc.rotary_f32(kn[b, h].float().numpy(), rd, 0, c, s, int(lens[b]))
            yv = vn[b, h].float().numpy()
            if kv == "e4m3":
                ref_k = (torch.from_numpy(yk) / 0.02).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                ref_v = (torch.from_numpy(yv) / 0.02).float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            else:
                ref_k = orc.raw(torch.from_numpy(yk).to(dt)); ref_v = orc.raw(torch.from_numpy(yv).to(dt))
            assert np.array_equal(k2[page, slot, h], ref_k)
            assert np.array_equal(v2[page, slot, h], ref_v)
        for h in range(Hq):
            yq = orc.rotary_f32(q[b, h].float().numpy(), rd, 0, c, s, int(lens[b]))
            assert np.array_equal(q2[b, h], orc.raw(torch.from_numpy(yq).to(qdt)))
