"""Pins for the oracle's multi-token (causal) decode: q_len query tokens per
sequence, token i of q_len attending the cached tokens [0, L - q_len + i + 1)
("Inference Cookbook" §3.2-3.3, causal attention after the new tokens were
appended; "FlashDecoding 与 FlashInfer 深度解析" §3.1, the append mode).

Checked against: a dense causal attention written with numpy matrices and an
explicit mask (a different formulation of the same definition), a 50-digit
brute force, the plain decode (q_len = 1, and the last query token, which
sees every cached token), and NaN poisoning of the tokens a query must not
see."""
import math

import numpy as np
import pytest

from oracle import oracle as orc
from tests.paged_cases import build_paged, round_to, to_storage


def _case(B, q_len, Hq, Hkv, D, lens, ps, seed):
    rng = np.random.default_rng(seed)
    Lmax = max(lens)
    K = round_to(rng.standard_normal((B, Lmax, Hkv, D)), orc.F32)
    V = round_to(rng.standard_normal((B, Lmax, Hkv, D)), orc.F32)
    Q = round_to(rng.standard_normal((B, q_len, Hq, D)), orc.F32)
    kp, vp, bt, npages = build_paged(K, V, lens, ps, rng)
    p = orc.problem(B, Hq, Hkv, D, ps, bt.shape[1], npages, orc.F32, orc.F32)
    return p, Q, K, V, to_storage(Q, orc.F32), kp, vp, bt, np.asarray(lens, np.int32)


def _dense_causal(Q, K, V, lens, Hq, Hkv):
    """Causal attention as matrices: S = Q K^T / sqrt(D) over all cached
    tokens of the KV head, mask[i, t] = t <= L - q_len + i, softmax, times V."""
    B, q_len, _, D = Q.shape
    G = Hq // Hkv
    out = np.zeros(Q.shape)
    lse = np.zeros((B, q_len, Hq))
    for b in range(B):
        L = int(lens[b])
        for h in range(Hq):
            k = K[b, :L, h // G]              # [L, D]
            v = V[b, :L, h // G]
            S = Q[b, :, h] @ k.T / math.sqrt(D)   # [q_len, L]
            mask = np.arange(L)[None, :] <= (L - q_len + np.arange(q_len))[:, None]
            S = np.where(mask, S, -np.inf)
            m = S.max(axis=1, keepdims=True)
            W = np.exp(S - m)
            Z = W.sum(axis=1, keepdims=True)
            out[b, :, h] = (W @ v) / Z
            lse[b, :, h] = (m + np.log(Z))[:, 0]
    return out, lse


@pytest.mark.parametrize("q_len,lens", [(1, [5, 40]), (2, [2, 33]), (4, [4, 17]), (7, [9, 64])])
def test_multi_matches_dense_causal_attention(q_len, lens):
    B, Hq, Hkv, D = 2, 6, 2, 16
    p, Q, K, V, q, kp, vp, bt, sl = _case(B, q_len, Hq, Hkv, D, lens, 16, seed=q_len)
    out, lse = orc.decode_paged_multi(p, q_len, q, kp, vp, None, None, bt, sl)
    ro, rl = _dense_causal(Q, K, V, sl, Hq, Hkv)
    np.testing.assert_allclose(out, ro, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, rl, rtol=0, atol=1e-13)


def test_multi_q_len_one_is_the_plain_decode():
    B, Hq, Hkv, D = 3, 8, 2, 16
    p, Q, K, V, q, kp, vp, bt, sl = _case(B, 1, Hq, Hkv, D, [1, 20, 77], 16, seed=5)
    out, lse = orc.decode_paged_multi(p, 1, q, kp, vp, None, None, bt, sl)
    q1 = to_storage(Q[:, 0], orc.F32)
    ro, rl = orc.decode_paged(p, q1, kp, vp, None, None, bt, sl)
    assert np.array_equal(out[:, 0], ro) and np.array_equal(lse[:, 0], rl)


def test_multi_last_token_sees_the_whole_cache():
    """The last query token's row equals the plain decode over all L tokens;
    token i equals the plain decode over the first L - q_len + i + 1."""
    B, q_len, Hq, Hkv, D = 2, 5, 4, 2, 8
    p, Q, K, V, q, kp, vp, bt, sl = _case(B, q_len, Hq, Hkv, D, [5, 30], 16, seed=6)
    out, lse = orc.decode_paged_multi(p, q_len, q, kp, vp, None, None, bt, sl)
    for i in range(q_len):
        qi = to_storage(Q[:, i], orc.F32)
        sli = (sl - q_len + i + 1).astype(np.int32)
        ro, rl = orc.decode_paged(p, qi, kp, vp, None, None, bt, sli)
        assert np.array_equal(out[:, i], ro) and np.array_equal(lse[:, i], rl)


def test_multi_bruteforce_50_digits():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    B, q_len, Hq, Hkv, D = 1, 3, 2, 1, 4
    p, Q, K, V, q, kp, vp, bt, sl = _case(B, q_len, Hq, Hkv, D, [6], 4, seed=7)
    out, lse = orc.decode_paged_multi(p, q_len, q, kp, vp, None, None, bt, sl)
    L = 6
    for i in range(q_len):
        for h in range(Hq):
            n = L - q_len + i + 1
            s = [mp.fsum(mp.mpf(float(Q[0, i, h, d])) * mp.mpf(float(K[0, t, 0, d])) for d in range(D)) / mp.sqrt(D)
                 for t in range(n)]
            e = [mp.e ** x for x in s]
            Z = mp.fsum(e)
            for d in range(D):
                ref = mp.fsum(e[t] * mp.mpf(float(V[0, t, 0, d])) for t in range(n)) / Z
                assert abs(out[0, i, h, d] - float(ref)) < 1e-14
            assert abs(lse[0, i, h] - float(mp.log(Z))) < 1e-14


def test_multi_hides_future_tokens():
    """NaN in the last cached token reaches only the last query token; NaN in
    token L - q_len + 1 reaches every token from the second on."""
    B, q_len, Hq, Hkv, D, L, ps = 1, 4, 2, 1, 8, 12, 4
    p, Q, K, V, q, kp, vp, bt, sl = _case(B, q_len, Hq, Hkv, D, [L], ps, seed=8)
    base, _ = orc.decode_paged_multi(p, q_len, q, kp, vp, None, None, bt, sl)
    for t_bad, first_hit in ((L - 1, q_len - 1), (L - q_len + 1, 1)):
        k2 = kp.clone()
        page, slot = int(bt[0, t_bad // ps]), t_bad % ps
        k2[page, slot] = float("nan")
        out, _ = orc.decode_paged_multi(p, q_len, q, k2, vp, None, None, bt, sl)
        for i in range(q_len):
            if i < first_hit:
                assert np.array_equal(out[0, i], base[0, i])
            else:
                assert np.isnan(out[0, i]).all()


def test_multi_rejects_caches_shorter_than_the_query():
    p, Q, K, V, q, kp, vp, bt, sl = _case(1, 3, 2, 1, 8, [2], 4, seed=9)
    with pytest.raises(ValueError):
        orc.decode_paged_multi(p, 3, q, kp, vp, None, None, bt, sl)
