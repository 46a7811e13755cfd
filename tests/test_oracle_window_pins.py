"""Pins for restricted self-attention in the CPU oracle ([JY] Self-Attention的优势: each
position attends a neighbourhood of size r; read as the keys j with |i - j| <= w, r = 2w+1).

Each ``check_*`` raises AssertionError when the oracle breaks the fact it pins; the planted
mistakes at the end swap a wrong window into the oracle and show that a pin catches it.
"""
import math

import numpy as np
import pytest

from oracle import mha_ref


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _qkv(seed, B=1, H=2, N=9, d=4):
    g = _rng(seed)
    return (g.standard_normal((B, H, N, d)), g.standard_normal((B, H, N, d)),
            g.standard_normal((B, H, N, d)))


def check_wide_window_is_full_attention():
    Q, K, V = _qkv(1)
    N = Q.shape[2]
    full = mha_ref.sdpa_ref(Q, K, V, "none")
    for w in (N - 1, N, 5 * N):
        assert np.array_equal(mha_ref.sdpa_ref(Q, K, V, "window", window=w), full)


def test_wide_window_is_full_attention():
    check_wide_window_is_full_attention()


def check_zero_window_returns_values():
    # only the key at the query's own position: weight exactly 1
    Q, K, V = _qkv(2)
    assert np.array_equal(mha_ref.sdpa_ref(Q, K, V, "window", window=0), V)


def test_zero_window_returns_values():
    check_zero_window_returns_values()


def check_radius_one_closed_form():
    # w = 1: row i averages v_{i-1}, v_i, v_{i+1} with weights exp(s_ij) / sum (edges: two keys)
    Q, K, V = _qkv(3, B=1, H=1, N=6, d=3)
    q, k, v = Q[0, 0], K[0, 0], V[0, 0]
    O = mha_ref.sdpa_ref(Q, K, V, "window", window=1)[0, 0]
    for i in range(6):
        js = [j for j in (i - 1, i, i + 1) if 0 <= j < 6]
        e = [math.exp(sum(q[i, t] * k[j, t] for t in range(3)) / math.sqrt(3)) for j in js]
        tot = sum(e)
        expect = [sum(e[a] / tot * v[j, t] for a, j in enumerate(js)) for t in range(3)]
        assert np.allclose(O[i], expect, rtol=1e-13, atol=1e-13)


def test_radius_one_closed_form():
    check_radius_one_closed_form()


def check_keys_outside_band_never_matter():
    Q, K, V = _qkv(4, N=12)
    w = 2
    O = mha_ref.sdpa_ref(Q, K, V, "window", window=w)
    i = 6
    K2, V2 = K.copy(), V.copy()
    far = [j for j in range(12) if abs(j - i) > w]
    K2[:, :, far] = 50.0
    V2[:, :, far] = -9.0
    O2 = mha_ref.sdpa_ref(Q, K2, V2, "window", window=w)
    assert np.array_equal(O2[:, :, i], O[:, :, i])
    near = [j for j in range(12) if abs(j - i) <= w]
    V3 = V.copy()
    V3[:, :, near[0]] += 1.0
    assert not np.array_equal(mha_ref.sdpa_ref(Q, K, V3, "window", window=w)[:, :, i],
                              O[:, :, i])


def test_keys_outside_band_never_matter():
    check_keys_outside_band_never_matter()


def check_bruteforce_tiny():
    for seed, (N, w) in enumerate([(1, 0), (5, 1), (7, 2), (8, 3)]):
        Q, K, V = _qkv(10 + seed, B=1, H=1, N=N, d=3)
        O = mha_ref.sdpa_ref(Q, K, V, "window", window=w)[0, 0]
        for i in range(N):
            s = {j: float(np.dot(Q[0, 0, i], K[0, 0, j])) / math.sqrt(3)
                 for j in range(N) if abs(i - j) <= w}
            mx = max(s.values())
            e = {j: math.exp(x - mx) for j, x in s.items()}
            tot = sum(e.values())
            expect = sum(e[j] / tot * V[0, 0, j] for j in e)
            assert np.allclose(O[i], expect, rtol=1e-12, atol=1e-12)


def test_bruteforce_tiny():
    check_bruteforce_tiny()


def test_window_needs_self_attention_and_a_radius():
    with pytest.raises(ValueError):
        mha_ref.allowed_keys("window", 4, 5, window=1)
    with pytest.raises(ValueError):
        mha_ref.allowed_keys("window", 4, 4)
    with pytest.raises(ValueError):
        mha_ref.allowed_keys("window", 4, 4, window=-1)


# ----------------------------------------------- planted mistakes: each must trip some pin

def _plant(monkeypatch, band):
    orig = mha_ref.allowed_keys

    def wrong(mask, Nq, Nk, key_len=None, rows=None, window=None):
        if mask != "window":
            return orig(mask, Nq, Nk, key_len, rows, window)
        i = (np.arange(Nq) if rows is None else np.asarray(rows))[:, None]
        j = np.arange(Nk)[None, :]
        return band(i, j, window)

    monkeypatch.setattr(mha_ref, "allowed_keys", wrong)


def test_plant_strict_band_is_caught(monkeypatch):
    _plant(monkeypatch, lambda i, j, w: np.abs(j - i) < w)  # drops the band's edges
    with pytest.raises(AssertionError):
        check_radius_one_closed_form()
    with pytest.raises(AssertionError):
        check_bruteforce_tiny()


def test_plant_one_sided_band_is_caught(monkeypatch):
    _plant(monkeypatch, lambda i, j, w: (j <= i) & (i - j <= w))  # looks back only
    with pytest.raises(AssertionError):
        check_radius_one_closed_form()
    with pytest.raises(AssertionError):
        check_wide_window_is_full_attention()
