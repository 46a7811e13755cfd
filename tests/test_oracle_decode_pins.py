"""Pins for decoding against a key/value cache in the CPU oracle ("causal_cache": the Nq
newest of L cached positions attend every position up to their own; [JY] Transformer 翻译样例
> Decoder and Transformer 训练样例).

Each ``check_*`` raises AssertionError when the oracle breaks the fact it pins; the planted
mistake at the end aligns the mask top-left and must be caught.
"""
import math

import numpy as np
import pytest

from oracle import mha_ref


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def check_full_cache_is_training_causal_mask():
    # all L positions are new queries: the training-time causal mask
    g = _rng(1)
    B, H, N, d = 2, 2, 7, 4
    Q, K, V = (g.standard_normal((B, H, N, d)) for _ in range(3))
    kl = np.full(B, N, np.int32)
    assert np.array_equal(mha_ref.sdpa_ref(Q, K, V, "causal_cache", kl),
                          mha_ref.sdpa_ref(Q, K, V, "causal"))


def test_full_cache_is_training_causal_mask():
    check_full_cache_is_training_causal_mask()


def check_single_new_token_sees_whole_prefix():
    # one new query: it is the last cached position and attends all L of them
    g = _rng(2)
    B, H, Nk, d = 3, 2, 11, 4
    Q = g.standard_normal((B, H, 1, d))
    K, V = g.standard_normal((B, H, Nk, d)), g.standard_normal((B, H, Nk, d))
    kl = np.array([1, 6, 11], np.int32)
    assert np.array_equal(mha_ref.sdpa_ref(Q, K, V, "causal_cache", kl),
                          mha_ref.sdpa_ref(Q, K, V, "key_padding", kl))


def test_single_new_token_sees_whole_prefix():
    check_single_new_token_sees_whole_prefix()


def check_step_by_step_equals_parallel_causal():
    # generating position t with the cache of positions 0..t gives row t of the causal
    # attention over the whole sequence ([JY] Transformer 训练样例: training computes all
    # positions at once under the causal mask; generation computes them one at a time)
    g = _rng(3)
    H, T, d = 2, 9, 4
    Q, K, V = (g.standard_normal((1, H, T, d)) for _ in range(3))
    full = mha_ref.sdpa_ref(Q, K, V, "causal")
    cap = 16
    Kc, Vc = np.zeros((1, H, cap, d)), np.zeros((1, H, cap, d))
    for t in range(T):
        Kc[:, :, t], Vc[:, :, t] = K[:, :, t], V[:, :, t]
        o = mha_ref.sdpa_ref(Q[:, :, t:t + 1], Kc, Vc, "causal_cache",
                             np.array([t + 1], np.int32))
        assert np.allclose(o[:, :, 0], full[:, :, t], rtol=1e-13, atol=1e-13)
    # several new queries at once: the last 3 rows
    o3 = mha_ref.sdpa_ref(Q[:, :, T - 3:], Kc, Vc, "causal_cache", np.array([T], np.int32))
    assert np.allclose(o3, full[:, :, T - 3:], rtol=1e-13, atol=1e-13)


def test_step_by_step_equals_parallel_causal():
    check_step_by_step_equals_parallel_causal()


def check_entries_past_the_cache_length_never_matter():
    g = _rng(4)
    B, H, Nq, Nk, d = 2, 1, 3, 12, 4
    Q = g.standard_normal((B, H, Nq, d))
    K, V = g.standard_normal((B, H, Nk, d)), g.standard_normal((B, H, Nk, d))
    kl = np.array([5, 9], np.int32)
    O = mha_ref.sdpa_ref(Q, K, V, "causal_cache", kl)
    K2, V2 = K.copy(), V.copy()
    for b in range(B):
        K2[b, :, kl[b]:] = 30.0
        V2[b, :, kl[b]:] = -4.0
    assert np.array_equal(mha_ref.sdpa_ref(Q, K2, V2, "causal_cache", kl), O)


def test_entries_past_the_cache_length_never_matter():
    check_entries_past_the_cache_length_never_matter()


def check_bruteforce_tiny():
    g = _rng(5)
    for Nq, L, Nk in [(1, 1, 1), (2, 5, 6), (3, 3, 4), (4, 7, 9)]:
        Q = g.standard_normal((1, 1, Nq, 3))
        K, V = g.standard_normal((1, 1, Nk, 3)), g.standard_normal((1, 1, Nk, 3))
        O = mha_ref.sdpa_ref(Q, K, V, "causal_cache", np.array([L], np.int32))[0, 0]
        for i in range(Nq):
            pos = L - Nq + i
            s = {j: float(np.dot(Q[0, 0, i], K[0, 0, j])) / math.sqrt(3) for j in range(pos + 1)}
            mx = max(s.values())
            e = {j: math.exp(x - mx) for j, x in s.items()}
            tot = sum(e.values())
            expect = sum(e[j] / tot * V[0, 0, j] for j in e)
            assert np.allclose(O[i], expect, rtol=1e-12, atol=1e-12)


def test_bruteforce_tiny():
    check_bruteforce_tiny()


def test_more_queries_than_cached_positions_is_rejected():
    with pytest.raises(ValueError):
        mha_ref.allowed_keys("causal_cache", 4, 8, key_len=3)
    with pytest.raises(ValueError):
        mha_ref.allowed_keys("causal_cache", 2, 8)


def test_plant_top_left_alignment_is_caught(monkeypatch):
    orig = mha_ref.allowed_keys

    def wrong(mask, Nq, Nk, key_len=None, rows=None, window=None):
        if mask != "causal_cache":
            return orig(mask, Nq, Nk, key_len, rows, window)
        i = (np.arange(Nq) if rows is None else np.asarray(rows))[:, None]
        return np.arange(Nk)[None, :] <= i   # forgets that the queries are the newest rows

    monkeypatch.setattr(mha_ref, "allowed_keys", wrong)
    with pytest.raises(AssertionError):
        check_single_new_token_sees_whole_prefix()
    with pytest.raises(AssertionError):
        check_step_by_step_equals_parallel_causal()
