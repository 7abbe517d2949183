"""Pins for the oracle's cache-row indirection and left padding ("Inference
Cookbook" §5.2 cache_batch_idx, §5.3 cache_leftpad), against independent
rebuilds of the cache: a re-gathered sub-batch and a cache without the
padded tokens."""
import numpy as np
import pytest

from oracle import oracle as orc
from tests.paged_cases import build_paged, round_to, to_storage


def _cache(Bc, Hq, Hkv, D, lens, ps, seed):
    rng = np.random.default_rng(seed)
    Lmax = max(lens)
    K = round_to(rng.standard_normal((Bc, Lmax, Hkv, D)), orc.BF16)
    V = round_to(rng.standard_normal((Bc, Lmax, Hkv, D)), orc.BF16)
    kp, vp, bt, n = build_paged(K, V, lens, ps, rng, kv_code=orc.BF16)
    return rng, K, V, kp, vp, bt, n


def test_no_indirection_equals_plain_decode():
    lens = [5, 40, 77]
    rng, K, V, kp, vp, bt, n = _cache(3, 8, 2, 32, lens, 16, 1)
    q = to_storage(round_to(rng.standard_normal((3, 8, 32)), orc.BF16), orc.BF16)
    p = orc.problem(3, 8, 2, 32, 16, bt.shape[1], n, orc.BF16, orc.BF16)
    o1, l1 = orc.decode_paged(p, q, kp, vp, None, None, bt, np.array(lens, np.int32))
    o2, l2 = orc.decode_paged_ex(p, 3, None, None, q, kp, vp, None, None, bt, np.array(lens, np.int32))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_batch_index_equals_regathered_sub_batch():
    lens = [12, 50, 3, 90, 33]
    rng, K, V, kp, vp, bt, n = _cache(5, 4, 2, 32, lens, 16, 2)
    idx = np.array([3, 0, 3, 4], np.int32)          # subset with a repeat
    q = to_storage(round_to(rng.standard_normal((4, 4, 32)), orc.BF16), orc.BF16)
    p = orc.problem(4, 4, 2, 32, 16, bt.shape[1], n, orc.BF16, orc.BF16)
    o1, l1 = orc.decode_paged_ex(p, 5, idx, None, q, kp, vp, None, None, bt, np.array(lens, np.int32))
    o2, l2 = orc.decode_paged(p, q, kp, vp, None, None, bt[idx], np.array(lens, np.int32)[idx])
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("lp", [[0, 0], [1, 17], [16, 33], [40, 100]])
def test_leftpad_equals_cache_without_padded_tokens(lp):
    lens = [40, 100]
    rng, K, V, kp, vp, bt, n = _cache(2, 4, 1, 16, lens, 16, 3)
    q = to_storage(round_to(rng.standard_normal((2, 4, 16)), orc.BF16), orc.BF16)
    p = orc.problem(2, 4, 1, 16, 16, bt.shape[1], n, orc.BF16, orc.BF16)
    o1, l1 = orc.decode_paged_ex(p, 2, None, np.array(lp, np.int32), q, kp, vp, None, None, bt,
                                 np.array(lens, np.int32))
    # rebuild a cache that holds only tokens [lp, L) of each row
    lens2 = [L - a for L, a in zip(lens, lp)]
    Lm = max(max(lens2), 1)
    K2 = np.zeros((2, Lm, 1, 16)); V2 = np.zeros((2, Lm, 1, 16))
    for b in range(2):
        K2[b, :lens2[b]] = K[b, lp[b]:lens[b]]
        V2[b, :lens2[b]] = V[b, lp[b]:lens[b]]
    kp2, vp2, bt2, n2 = build_paged(K2, V2, [max(x, 0) for x in lens2], 16, np.random.default_rng(9),
                                    kv_code=orc.BF16)
    p2 = orc.problem(2, 4, 1, 16, 16, bt2.shape[1], n2, orc.BF16, orc.BF16)
    o2, l2 = orc.decode_paged(p2, q, kp2, vp2, None, None, bt2, np.array(lens2, np.int32))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_bad_index_and_leftpad_rejected():
    lens = [10, 20]
    rng, K, V, kp, vp, bt, n = _cache(2, 2, 1, 16, lens, 16, 4)
    q = to_storage(np.zeros((2, 2, 16)), orc.BF16)
    p = orc.problem(2, 2, 1, 16, 16, bt.shape[1], n, orc.BF16, orc.BF16)
    with pytest.raises(ValueError):
        orc.decode_paged_ex(p, 2, np.array([0, 2], np.int32), None, q, kp, vp, None, None, bt,
                            np.array(lens, np.int32))
    with pytest.raises(ValueError):
        orc.decode_paged_ex(p, 2, None, np.array([0, 21], np.int32), q, kp, vp, None, None, bt,
                            np.array(lens, np.int32))
