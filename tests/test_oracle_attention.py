"""Pins for the oracle's attention, partial-state, merge and append functions.

Each check compares the oracle with something other than itself: closed
forms (single token, identical keys, zero query, two-key logistic), brute
force in 50-digit arithmetic, the pages' merge-equals-unsplit property over
arbitrary partitions, the paged-vs-contiguous identity, the GQA head map and
the page's worked block-table example.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from tests.paged_cases import build_paged, round_to, to_storage

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _problem(B, Hq, Hkv, D, ps, max_blocks, num_pages, q_code=orc.F32, kv_code=orc.F32):
    return orc.problem(B, Hq, Hkv, D, ps, max_blocks, num_pages, q_code, kv_code)


def _case(B, Hq, Hkv, D, lens, ps, seed, kv_code=orc.F32, kscale=1.0):
    rng = np.random.default_rng(seed)
    Lmax = max(lens)
    K = round_to(rng.standard_normal((B, Lmax, Hkv, D)) * kscale, kv_code)
    V = round_to(rng.standard_normal((B, Lmax, Hkv, D)), kv_code)
    Q = round_to(rng.standard_normal((B, Hq, D)), orc.F32)
    kp, vp, bt, npages = build_paged(K, V, lens, ps, rng, kv_code=kv_code)
    p = _problem(B, Hq, Hkv, D, ps, bt.shape[1], npages, orc.F32, kv_code)
    q = to_storage(Q, orc.F32)
    return p, Q, K, V, q, kp, vp, bt, np.asarray(lens, np.int32)


def test_single_token_returns_v():
    p, Q, K, V, q, kp, vp, bt, lens = _case(2, 4, 2, 8, [1, 1], 4, seed=1)
    out, lse = orc.decode_paged(p, q, kp, vp, None, None, bt, lens)
    G = p.Hq // p.Hkv
    for b in range(2):
        for h in range(4):
            assert np.array_equal(out[b, h], V[b, 0, h // G])
            s0 = float(np.dot(Q[b, h], K[b, 0, h // G])) / math.sqrt(8)
            assert abs(lse[b, h] - s0) <= 1e-14 * max(1.0, abs(s0))


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(2)
    B, Hq, Hkv, D, L, ps = 1, 2, 1, 16, 37, 8
    k0 = round_to(rng.standard_normal(D), orc.F32)
    K = np.broadcast_to(k0, (B, L, Hkv, D)).copy()
    V = round_to(rng.standard_normal((B, L, Hkv, D)), orc.F32)
    Q = round_to(rng.standard_normal((B, Hq, D)), orc.F32)
    kp, vp, bt, n = build_paged(K, V, [L], ps, rng)
    p = _problem(B, Hq, Hkv, D, ps, bt.shape[1], n)
    out, lse = orc.decode_paged(p, to_storage(Q, orc.F32), kp, vp, None, None, bt, np.array([L], np.int32))
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], V[0, :, 0].mean(axis=0), rtol=0, atol=1e-14)
        s = float(np.dot(Q[0, h], k0)) / math.sqrt(D)
        assert abs(lse[0, h] - (s + math.log(L))) < 1e-13


def test_zero_query_gives_mean_and_log_length():
    p, Q, K, V, q, kp, vp, bt, lens = _case(3, 2, 1, 8, [5, 19, 64], 16, seed=3)
    q0 = to_storage(np.zeros((3, 2, 8)), orc.F32)
    out, lse = orc.decode_paged(p, q0, kp, vp, None, None, bt, lens)
    for b, L in enumerate(lens):
        for h in range(2):
            np.testing.assert_allclose(out[b, h], V[b, :L, 0].mean(axis=0), rtol=0, atol=1e-14)
            assert abs(lse[b, h] - math.log(L)) < 1e-14


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(4)
    B, Hq, Hkv, D, L, ps = 1, 1, 1, 4, 50, 16
    K = np.zeros((B, L, Hkv, D))
    V = round_to(rng.standard_normal((B, L, Hkv, D)), orc.F32)
    Q = np.zeros((B, Hq, D))
    Q[0, 0, 0] = 1.0
    star = 23
    K[0, star, 0, 0] = 80.0  # score 80 / sqrt(4) = 40 above every other key
    kp, vp, bt, n = build_paged(K, V, [L], ps, rng)
    p = _problem(B, Hq, Hkv, D, ps, bt.shape[1], n)
    out, lse = orc.decode_paged(p, to_storage(Q, orc.F32), kp, vp, None, None, bt, np.array([L], np.int32))
    bound = (L - 1) * math.exp(-40.0) * 2 * np.abs(V).max()
    assert np.abs(out[0, 0] - V[0, star, 0]).max() <= bound
    assert abs(lse[0, 0] - 40.0) <= L * math.exp(-40.0)


def test_two_keys_logistic_closed_form():
    # q = e0, k0 = a e0, k1 = 0, D = 4: s0 = a/2, s1 = 0, so the weight of
    # key 0 is the logistic function 1 / (1 + exp(-a/2)).
    D = 4
    for a in (-6.0, -1.0, 0.0, 0.5, 3.0, 10.0):
        K = np.zeros((1, 2, 1, D))
        K[0, 0, 0, 0] = a
        V = np.array([[[[1.0, -2.0, 0.5, 4.0]], [[-3.0, 0.25, 2.0, -1.0]]]])
        Q = np.zeros((1, 1, D))
        Q[0, 0, 0] = 1.0
        rng = np.random.default_rng(5)
        kp, vp, bt, n = build_paged(K, V, [2], 16, rng)
        p = _problem(1, 1, 1, D, 16, bt.shape[1], n)
        out, lse = orc.decode_paged(p, to_storage(Q, orc.F32), kp, vp, None, None, bt, np.array([2], np.int32))
        w0 = 1.0 / (1.0 + math.exp(-a / 2))
        np.testing.assert_allclose(out[0, 0], w0 * V[0, 0, 0] + (1 - w0) * V[0, 1, 0], rtol=0, atol=1e-15)
        assert abs(lse[0, 0] - math.log1p(math.exp(a / 2))) < 1e-15


def test_bruteforce_50_digits():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    for seed in range(6):
        rng = np.random.default_rng(100 + seed)
        B, Hkv, G, D, ps = 2, 2, 2, 4, 2
        Hq = Hkv * G
        lens = [int(rng.integers(1, 9)), int(rng.integers(1, 9))]
        p, Q, K, V, q, kp, vp, bt, ln = _case(B, Hq, Hkv, D, lens, ps, seed=200 + seed)
        out, lse = orc.decode_paged(p, q, kp, vp, None, None, bt, ln)
        for b in range(B):
            for h in range(Hq):
                kvh = h // G
                s = [mp.fsum(mp.mpf(float(Q[b, h, d])) * mp.mpf(float(K[b, t, kvh, d])) for d in range(D))
                     / mp.sqrt(D) for t in range(lens[b])]
                e = [mp.exp(x) for x in s]
                Z = mp.fsum(e)
                for d in range(D):
                    ref = mp.fsum(e[t] * mp.mpf(float(V[b, t, kvh, d])) for t in range(lens[b])) / Z
                    assert abs(float(ref) - out[b, h, d]) < 1e-14
                assert abs(float(mp.log(Z)) - lse[b, h]) < 1e-14


@pytest.mark.parametrize("L", [1, 2, 16, 37, 100])
def test_merge_of_any_partition_equals_unsplit(L):
    p, Q, K, V, q, kp, vp, bt, lens = _case(1, 2, 1, 8, [L], 4, seed=L)
    out, lse = orc.decode_paged(p, q, kp, vp, None, None, bt, lens)
    rng = np.random.default_rng(L)
    partitions = [[0, L]]
    for S in range(1, L + 1):  # contiguous uniform splits, like the pages' chunks
        c = -(-L // S)
        partitions.append(sorted(set([min(L, i * c) for i in range(S + 1)] + [L])))
    for _ in range(10):  # random uneven splits with empty pieces
        cuts = sorted(rng.integers(0, L + 1, size=int(rng.integers(1, 6))).tolist())
        partitions.append([0] + cuts + [L])
    for h in range(2):
        for edges in partitions:
            parts = [orc.partial_state(p, q, kp, vp, None, None, bt, 0, h, a, b)
                     for a, b in zip(edges[:-1], edges[1:])]
            o = np.stack([x[0] for x in parts])
            m = np.array([x[1] for x in parts])
            d = np.array([x[2] for x in parts])
            mo, ml = orc.merge_states(o, m, d)
            np.testing.assert_allclose(mo, out[0, h], rtol=0, atol=1e-12)
            assert abs(ml - lse[0, h]) < 1e-12


def test_merge_rescale_closed_form():
    # Two partial states with m = (0, ln 3), d = (1, 1): alpha = (1/3, 1).
    o = np.array([[3.0, 0.0], [0.0, 6.0]])
    out, lse = orc.merge_states(o, np.array([0.0, math.log(3.0)]), np.array([1.0, 1.0]))
    # sum alpha_i o_i = (1, 6); d_global = 4/3 -> out = (0.75, 4.5); lse = ln 3 + ln(4/3) = ln 4
    np.testing.assert_allclose(out, [0.75, 4.5], rtol=0, atol=1e-15)
    assert abs(lse - math.log(4.0)) < 1e-15
    # empty states are ignored; all-empty gives zeros and -inf
    out2, lse2 = orc.merge_states(np.zeros((2, 2)), np.array([-np.inf, -np.inf]), np.zeros(2))
    assert np.all(out2 == 0) and lse2 == -np.inf


def test_paged_gather_equals_contiguous_bitexact():
    rng = np.random.default_rng(9)
    B, Hq, Hkv, D, ps = 3, 8, 2, 32, 16
    lens = [1, 45, 130]
    Lmax = max(lens)
    for code in (orc.F16, orc.BF16):
        K = round_to(rng.standard_normal((B, Lmax, Hkv, D)), code)
        V = round_to(rng.standard_normal((B, Lmax, Hkv, D)), code)
        Q = round_to(rng.standard_normal((B, Hq, D)), code)
        kp, vp, bt, n = build_paged(K, V, lens, ps, rng, kv_code=code)
        p = _problem(B, Hq, Hkv, D, ps, bt.shape[1], n, code, code)
        q = to_storage(Q, code)
        ln = np.asarray(lens, np.int32)
        o1, l1 = orc.decode_paged(p, q, kp, vp, None, None, bt, ln)
        o2, l2 = orc.decode_contiguous(p, Lmax, q, to_storage(K, code), to_storage(V, code), ln)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_gqa_maps_query_head_to_kv_head_group():
    rng = np.random.default_rng(10)
    B, Hkv, G, D, L = 1, 4, 3, 8, 20
    Hq = Hkv * G
    K = round_to(rng.standard_normal((B, L, Hkv, D)), orc.F32)
    V = np.zeros((B, L, Hkv, D))
    for kvh in range(Hkv):
        V[:, :, kvh, :] = kvh + 1.0
    kp, vp, bt, n = build_paged(K, V, [L], 16, rng)
    p = _problem(B, Hq, Hkv, D, 16, bt.shape[1], n)
    q = to_storage(round_to(rng.standard_normal((B, Hq, D)), orc.F32), orc.F32)
    out, _ = orc.decode_paged(p, q, kp, vp, None, None, bt, np.array([L], np.int32))
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], (h // G) + 1.0, rtol=0, atol=1e-14)


def test_fp8_pages_are_decoded_and_scaled():
    # One token per sequence: out = decode(v_code) * v_scale exactly;
    # lse = (q . decode(k_code) * k_scale) / sqrt(D).
    D, ps = 4, 16
    kcodes = np.array([0x38, 0xB8, 0x01, 0x7E], np.uint8)   # 1, -1, 2^-9, 448
    vcodes = np.array([0x40, 0x08, 0xC4, 0x3C], np.uint8)   # 2, 2^-6, -3, 1.5
    kp = np.full((2, ps, 1, D), 0x7F, np.uint8)
    vp = np.full((2, ps, 1, D), 0x7F, np.uint8)
    kp[1, 0, 0] = kcodes
    vp[1, 0, 0] = vcodes
    ks = np.array([[np.nan], [0.5]], np.float32)
    vs = np.array([[np.nan], [0.25]], np.float32)
    q = np.array([[[1.0, 2.0, 4.0, 0.125]]], np.float32)
    bt = np.array([[1]], np.int32)
    p = orc.problem(1, 1, 1, D, ps, 1, 2, orc.F32, orc.E4M3)
    out, lse = orc.decode_paged(p, q, kp, vp, ks, vs, bt, np.array([1], np.int32))
    np.testing.assert_array_equal(out[0, 0], np.array([2.0, 2.0 ** -6, -3.0, 1.5]) * 0.25)
    kval = np.array([1.0, -1.0, 2.0 ** -9, 448.0]) * 0.5
    assert abs(lse[0, 0] - float(np.dot(q[0, 0], kval)) / 2.0) < 1e-14


def test_empty_sequence_and_bad_page():
    p, Q, K, V, q, kp, vp, bt, lens = _case(2, 2, 1, 8, [0, 3], 16, seed=11)
    out, lse = orc.decode_paged(p, q, kp, vp, None, None, bt, np.array([0, 3], np.int32))
    assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf)
    assert np.all(np.isfinite(out[1]))
    bad = bt.copy()
    bad[1, 0] = -1
    with pytest.raises(IndexError):
        orc.decode_paged(p, q, kp, vp, None, None, bad, np.array([0, 3], np.int32))
    bad[1, 0] = p.num_pages
    with pytest.raises(IndexError):
        orc.decode_paged(p, q, kp, vp, None, None, bad, np.array([0, 3], np.int32))


def _read_golden(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *vals = line.split()
                rows.setdefault(key, []).append(vals)
    return rows


def test_cookbook_block_table_worked_example():
    g = _read_golden("cookbook_paged_example.txt")
    ps = int(g["page_size"][0][0])
    npages = int(g["num_pages"][0][0])
    bt = np.array([[int(x) for x in r[1:]] for r in sorted(g["block_table"], key=lambda r: int(r[0]))], np.int32)
    lens = np.array([int(r[1]) for r in sorted(g["seq_len"], key=lambda r: int(r[0]))], np.int32)
    pool = np.zeros((npages, ps, 1, 1))
    for page in range(npages):
        pool[page, :, 0, 0] = 1000.0 * page + np.arange(ps)
    kp = to_storage(np.zeros_like(pool), orc.F32)
    vp = to_storage(pool, orc.F32)
    p = orc.problem(2, 1, 1, 1, ps, bt.shape[1], npages, orc.F32, orc.F32)
    out, lse = orc.decode_paged(p, np.zeros((2, 1, 1), np.float32), kp, vp, None, None, bt, lens)
    for b, frac in sorted(g["expected"], key=lambda r: int(r[0])):
        b = int(b)
        assert abs(out[b, 0, 0] - float(Fraction(frac))) < 1e-9
        assert abs(lse[b, 0] - math.log(lens[b])) < 1e-14


def test_append_writes_only_the_new_slot():
    rng = np.random.default_rng(12)
    B, Hkv, D, ps = 3, 2, 8, 16
    lens = np.array([0, 15, 33], np.int32)
    num_pages = 10
    bt = np.array([[4, -1, -1], [7, 2, -1], [1, 3, 9]], np.int32)
    kp = torch.randn(num_pages, ps, Hkv, D, dtype=torch.float32).to(torch.bfloat16)
    vp = torch.randn(num_pages, ps, Hkv, D, dtype=torch.float32).to(torch.bfloat16)
    kn = torch.randn(B, Hkv, D).to(torch.bfloat16)
    vn = torch.randn(B, Hkv, D).to(torch.bfloat16)
    p = orc.problem(B, Hkv, Hkv, D, ps, 3, num_pages, orc.BF16, orc.BF16)
    k2, v2 = orc.append_kv(p, orc.BF16, kn, vn, kp, vp, None, None, bt, lens)
    kr, vr = orc.raw(kp), orc.raw(vp)
    expect_k, expect_v = kr.copy(), vr.copy()
    for b, L in enumerate(lens):
        page, slot = bt[b, L // ps], L % ps
        expect_k[page, slot] = orc.raw(kn)[b]
        expect_v[page, slot] = orc.raw(vn)[b]
    assert np.array_equal(k2, expect_k) and np.array_equal(v2, expect_v)


def test_append_fp8_quantises_with_page_scale():
    B, Hkv, D, ps = 2, 1, 16, 16
    lens = np.array([3, 16], np.int32)
    bt = np.array([[0, -1], [1, 2]], np.int32)
    kp = np.zeros((3, ps, Hkv, D), np.uint8)
    vp = np.zeros((3, ps, Hkv, D), np.uint8)
    ks = np.array([[0.5], [2.0], [0.01]], np.float32)
    vs = np.array([[0.25], [4.0], [1.0]], np.float32)
    x = torch.linspace(-6, 6, B * Hkv * D).reshape(B, Hkv, D).to(torch.bfloat16)
    p = orc.problem(B, 1, 1, D, ps, 2, 3, orc.BF16, orc.E4M3)
    k2, v2 = orc.append_kv(p, orc.BF16, x, x, kp, vp, ks, vs, bt, lens)
    xf = x.to(torch.float32)
    for b, L in enumerate(lens):
        page, slot = bt[b, L // ps], L % ps
        for which, pool, sc in ((0, k2, ks), (1, v2, vs)):
            y = (xf[b, 0] / float(sc[page, 0])).clamp(-448, 448)
            ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            assert np.array_equal(pool[page, slot, 0], ref)
    # untouched pages/slots stay zero
    touched = {(0, 3), (2, 0)}
    for page in range(3):
        for slot in range(ps):
            if (page, slot) not in touched:
                assert not k2[page, slot].any() and not v2[page, slot].any()
