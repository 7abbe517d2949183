"""Pins for the oracle's pair-list entry (decode of chosen (b, hq) pairs).

The pair-list decode is what the large-batch parity checks and the bench's
CPU baseline call.  It must give, for every listed pair, exactly the row the
full decode gives for that (sequence, query head): same gather, same token
order, same fp64 arithmetic.  These tests pin it to the full decode (itself
pinned by closed forms and brute force) bit for bit, with the pairs shuffled,
repeated and spread over several thread counts, plus a closed form on the
pair path itself (one-token sequences return their V row), so a swapped or
mis-strided (b, hq) decode fails here rather than as a GPU mismatch.
"""
import math

import numpy as np
import pytest

from oracle import oracle as orc
from tests.paged_cases import build_paged, round_to, to_storage


def _case(B, Hq, Hkv, D, lens, ps, seed):
    rng = np.random.default_rng(seed)
    Lmax = max(max(lens), 1)
    K = round_to(rng.standard_normal((B, Lmax, Hkv, D)), orc.F32)
    V = round_to(rng.standard_normal((B, Lmax, Hkv, D)), orc.F32)
    Q = round_to(rng.standard_normal((B, Hq, D)), orc.F32)
    kp, vp, bt, npages = build_paged(K, V, lens, ps, rng)
    p = orc.problem(B, Hq, Hkv, D, ps, bt.shape[1], npages, orc.F32, orc.F32)
    return p, Q, K, V, to_storage(Q, orc.F32), kp, vp, bt, np.asarray(lens, np.int32)


@pytest.mark.parametrize("nthreads", [1, 3, 16])
def test_pairs_equal_full_decode_rows_bitexact(nthreads):
    # B != Hq and Hq != Hkv, so a swapped (b, hq) or a wrong stride reads a
    # different row (or fails the range check)
    B, Hq, Hkv, D = 5, 6, 2, 16
    p, Q, K, V, q, kp, vp, bt, lens = _case(B, Hq, Hkv, D, [0, 1, 17, 64, 40], 16, seed=21)
    full_o, full_l = orc.decode_paged(p, q, kp, vp, None, None, bt, lens)
    rng = np.random.default_rng(nthreads)
    pairs = [(b, h) for b in range(B) for h in range(Hq)]
    rng.shuffle(pairs)
    pairs = pairs + pairs[:7] + [(B - 1, Hq - 1), (0, 0)]  # repeats
    out, lse = orc.decode_paged_pairs(p, q, kp, vp, None, None, bt, lens, pairs, nthreads=nthreads)
    assert out.shape == (len(pairs), D) and lse.shape == (len(pairs),)
    for i, (b, h) in enumerate(pairs):
        assert np.array_equal(out[i], full_o[b, h]), (b, h)
        assert (lse[i] == full_l[b, h]) or (np.isneginf(lse[i]) and np.isneginf(full_l[b, h])), (b, h)


def test_pairs_fp8_pool_bitexact():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, D, ps = 3, 8, 2, 32, 16
    lens = [5, 33, 70]
    Lmax = max(lens)
    K = round_to(rng.standard_normal((B, Lmax, Hkv, D)), orc.F32)
    V = round_to(rng.standard_normal((B, Lmax, Hkv, D)), orc.F32)
    kp, vp, bt, npages = build_paged(K, V, lens, ps, rng)
    # quantise the pools to E4M3 codes with a per-(page, kvh) scale
    import torch
    kf = kp.to(torch.float32).nan_to_num(0.0)
    vf = vp.to(torch.float32).nan_to_num(0.0)
    ks = (kf.abs().amax(dim=(1, 3)) / 448).clamp_min(1e-12)
    vs = (vf.abs().amax(dim=(1, 3)) / 448).clamp_min(1e-12)
    kc = (kf / ks[:, None, :, None]).to(torch.float8_e4m3fn)
    vc = (vf / vs[:, None, :, None]).to(torch.float8_e4m3fn)
    Q = round_to(rng.standard_normal((B, Hq, D)), orc.BF16)
    p = orc.problem(B, Hq, Hkv, D, ps, bt.shape[1], npages, orc.BF16, orc.E4M3)
    q = to_storage(Q, orc.BF16)
    sl = np.asarray(lens, np.int32)
    full_o, full_l = orc.decode_paged(p, q, kc, vc, ks, vs, bt, sl)
    pairs = [(2, 7), (0, 0), (1, 3), (2, 7), (1, 4)]
    out, lse = orc.decode_paged_pairs(p, q, kc, vc, ks, vs, bt, sl, pairs, nthreads=2)
    for i, (b, h) in enumerate(pairs):
        assert np.array_equal(out[i], full_o[b, h]) and lse[i] == full_l[b, h]


def test_pairs_one_token_closed_form():
    """One-token sequences: the listed pair's output is its KV head's V row
    and its lse is the scaled score, whatever order the pairs come in."""
    B, Hq, Hkv, D = 4, 4, 2, 8
    p, Q, K, V, q, kp, vp, bt, lens = _case(B, Hq, Hkv, D, [1, 1, 1, 1], 16, seed=9)
    G = Hq // Hkv
    pairs = [(3, 0), (0, 3), (2, 1), (1, 2)]
    out, lse = orc.decode_paged_pairs(p, q, kp, vp, None, None, bt, lens, pairs, nthreads=4)
    for i, (b, h) in enumerate(pairs):
        assert np.array_equal(out[i], V[b, 0, h // G])
        s0 = float(np.dot(Q[b, h], K[b, 0, h // G])) / math.sqrt(D)
        assert abs(lse[i] - s0) <= 1e-14 * max(1.0, abs(s0))


def test_pairs_out_of_range_rejected():
    p, Q, K, V, q, kp, vp, bt, lens = _case(2, 4, 2, 8, [3, 4], 16, seed=2)
    for bad in ([(2, 0)], [(0, 4)], [(-1, 0)], [(0, -1)]):
        with pytest.raises(ValueError):
            orc.decode_paged_pairs(p, q, kp, vp, None, None, bt, lens, bad)
