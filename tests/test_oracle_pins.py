"""Pins for the CPU oracle: facts the pages and the mathematics fix, independent of the oracle.

Each ``check_*`` function raises AssertionError when the oracle breaks the fact it pins.
The planted-mistake tests at the end swap a deliberately wrong step into the oracle (on the
CPU) and show that at least one pin catches it.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle  # noqa: F401  (package import must work on its own)
from oracle import mha_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------- softmax rows sum to one

def check_rows_sum_to_one():
    g = _rng(1)
    q, k = g.standard_normal((7, 16)), g.standard_normal((9, 16))
    for mask, L in [("none", None), ("key_padding", 4)]:
        allowed = mha_ref.allowed_keys(mask, 7, 9, L)
        w = mha_ref.attention_weights_ref(q, k, allowed)
        assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12, rtol=0)
        assert np.all(w[~allowed] == 0.0)
        assert np.all(w[allowed] > 0.0)
    k2 = g.standard_normal((7, 16))
    allowed = mha_ref.allowed_keys("causal", 7, 7)
    w = mha_ref.attention_weights_ref(q, k2, allowed)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12, rtol=0)
    assert np.all(w[~allowed] == 0.0)


def test_rows_sum_to_one():
    check_rows_sum_to_one()


# ------------------------------------------------------ identical keys -> mean of values

@pytest.mark.parametrize("mask", ["none", "causal", "key_padding"])
def test_identical_keys_give_mean_of_values(mask):
    g = _rng(2)
    B, H, N, d = 2, 2, 6, 8
    Q = g.standard_normal((B, H, N, d))
    K = np.broadcast_to(g.standard_normal((B, H, 1, d)), (B, H, N, d)).copy()
    V = g.standard_normal((B, H, N, d))
    key_len = np.array([3, 6], np.int32) if mask == "key_padding" else None
    O = mha_ref.sdpa_ref(Q, K, V, mask, key_len)
    for b in range(B):
        for i in range(N):
            if mask == "none":
                sel = slice(0, N)
            elif mask == "causal":
                sel = slice(0, i + 1)
            else:
                sel = slice(0, int(key_len[b]))
            np.testing.assert_allclose(O[b, :, i], V[b, :, sel].mean(axis=1), atol=1e-12, rtol=0)


# ---------------------------------------- orthogonal key + large matching query selects v*

def test_orthogonal_key_selects_its_value():
    g = _rng(3)
    d, N = 16, 10
    K = np.eye(d)[:N][None, None]                    # orthonormal key rows
    V = g.standard_normal((1, 1, N, 8))
    targets = g.integers(0, N, size=5)
    Q = (100.0 * math.sqrt(d) * np.eye(d)[targets])[None, None]  # scaled score 100 vs 0
    O = mha_ref.sdpa_ref(Q, K, V)
    np.testing.assert_allclose(O[0, 0], V[0, 0, targets], atol=1e-12, rtol=0)


# ----------------------------------------- masked positions cannot change earlier outputs

def check_mask_invariance():
    g = _rng(4)
    B, H, N, d = 2, 2, 9, 8
    Q, K, V = (g.standard_normal((B, H, N, d)) for _ in range(3))
    O = mha_ref.sdpa_ref(Q, K, V, "causal")
    i0 = 4
    K2, V2 = K.copy(), V.copy()
    K2[:, :, i0 + 1:] += 10 * g.standard_normal(K2[:, :, i0 + 1:].shape)
    V2[:, :, i0 + 1:] -= 7.0
    O2 = mha_ref.sdpa_ref(Q, K2, V2, "causal")
    assert np.array_equal(O[:, :, :i0 + 1], O2[:, :, :i0 + 1])
    assert not np.array_equal(O[:, :, i0 + 1:], O2[:, :, i0 + 1:])
    key_len = np.array([3, 7], np.int32)
    O = mha_ref.sdpa_ref(Q, K, V, "key_padding", key_len)
    K3, V3 = K.copy(), V.copy()
    for b in range(B):
        K3[b, :, key_len[b]:] = 5.0
        V3[b, :, key_len[b]:] = -3.0
    O3 = mha_ref.sdpa_ref(Q, K3, V3, "key_padding", key_len)
    assert np.array_equal(O, O3)


def test_mask_invariance_bitwise():
    check_mask_invariance()


def check_causal_mask_matches_pages():
    path = os.path.join(GOLDEN, "causal_mask_4x4.txt")
    rows = [ln.strip() for ln in open(path, encoding="utf-8") if ln.strip() and not ln.startswith("#")]
    want = np.array([[c == "1" for c in r] for r in rows])
    got = mha_ref.allowed_keys("causal", 4, 4)
    assert np.array_equal(got, want)


def test_causal_mask_matches_pages():
    check_causal_mask_matches_pages()


# ------------------------------------------------------------ the worked example's weights

def check_worked_example_weights():
    ex = json.load(open(os.path.join(GOLDEN, "worked_example_love.json"), encoding="utf-8"))
    w_want = np.array(ex["weights"])
    n, d = ex["n"], ex["d_head"]
    # one head: keys along e_0 with lengths ln(w_j) and a query sqrt(d)*e_0, so that the
    # scaled scores are exactly ln(w_j) and softmax returns w_j (their sum is 1).
    K = np.zeros((n, d))
    K[:, 0] = np.log(w_want)
    q = np.zeros((1, d))
    q[0, 0] = math.sqrt(d)
    w = mha_ref.attention_weights_ref(q, K, np.ones((1, n), bool))
    np.testing.assert_allclose(w[0], w_want, atol=1e-14, rtol=0)
    V = _rng(5).standard_normal((n, d))
    o = mha_ref.sdpa_ref(q[None, None], K[None, None], V[None, None])[0, 0, 0]
    np.testing.assert_allclose(o, w_want @ V, atol=1e-14, rtol=0)


def test_worked_example_weights():
    check_worked_example_weights()


def test_worked_example_shapes():
    ex = json.load(open(os.path.join(GOLDEN, "worked_example_love.json"), encoding="utf-8"))
    n, D, H, dh = ex["n"], ex["d_model"], ex["heads"], ex["d_head"]
    assert D == H * dh
    g = _rng(6)
    x = g.standard_normal((1, n, D))
    W_qkv = g.uniform(-0.07, 0.07, (3 * D, D))
    W_o = g.uniform(-0.07, 0.07, (D, D))
    y, parts = mha_ref.mha_layer_ref(x, None, W_qkv, None, W_o, None, None, None, H,
                                    return_parts=True)
    assert parts["Q"].shape == (1, H, n, dh)
    assert parts["O"].shape == (1, H, n, dh)
    assert parts["C"].shape == (1, n, D)
    assert y.shape == (1, n, D)
    shapes = json.load(open(os.path.join(GOLDEN, "model_shapes.json"), encoding="utf-8"))
    assert shapes["base"]["d_model"] == shapes["base"]["heads"] * shapes["base"]["d_k"]
    assert shapes["big"]["d_model"] // shapes["big"]["heads"] == 64


# ------------------------------------------------------------------- algebraic invariances

def test_shift_invariance_of_keys():
    g = _rng(7)
    Q, K, V = (g.standard_normal((2, 3, 8, 16)) for _ in range(3))
    c = g.standard_normal(16)
    O = mha_ref.sdpa_ref(Q, K, V)
    O2 = mha_ref.sdpa_ref(Q, K + c, V)
    np.testing.assert_allclose(O, O2, atol=1e-12, rtol=1e-12)


def test_permutation_equivariance():
    g = _rng(8)
    Q, K, V = (g.standard_normal((1, 2, 11, 8)) for _ in range(3))
    pk = g.permutation(11)
    pq = g.permutation(11)
    O = mha_ref.sdpa_ref(Q, K, V)
    np.testing.assert_allclose(mha_ref.sdpa_ref(Q, K[:, :, pk], V[:, :, pk]), O, atol=1e-12, rtol=0)
    np.testing.assert_allclose(mha_ref.sdpa_ref(Q[:, :, pq], K, V), O[:, :, pq], atol=1e-12, rtol=0)


# ------------------------------------------------------------- layer special cases, LN facts

def check_layernorm_moments():
    g = _rng(9)
    r = 3.0 * g.standard_normal((5, 64)) + 1.5
    eps = 1e-5
    y = mha_ref.layernorm_ref(r, np.ones(64), np.zeros(64), eps)
    var = r.var(axis=1)  # biased
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=1), var / (var + eps), atol=1e-12, rtol=0)


def test_layernorm_moments():
    check_layernorm_moments()


def test_zero_output_projection_gives_layernorm_of_input():
    g = _rng(10)
    B, N, D, H = 2, 5, 32, 4
    x = g.standard_normal((B, N, D))
    W_qkv = g.standard_normal((3 * D, D))
    gamma, beta = 1 + 0.1 * g.standard_normal(D), 0.1 * g.standard_normal(D)
    y = mha_ref.mha_layer_ref(x, None, W_qkv, None, np.zeros((D, D)), np.zeros(D), gamma, beta, H)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (D,), torch.from_numpy(gamma),
                                         torch.from_numpy(beta), eps=1e-5).numpy()
    np.testing.assert_allclose(y, ref, atol=1e-12, rtol=0)


def check_single_head_identity_is_plain_attention():
    """H=1, d_k=D, all projections the identity: the sublayer is LN(x + SDPA(x, x, x)).
    Checked against torch's own float64 attention and layer_norm routines."""
    g = _rng(11)
    B, N, D = 2, 7, 16
    x = g.standard_normal((B, N, D))
    I = np.eye(D)
    for mask in ["none", "causal"]:
        y = mha_ref.mha_layer_ref(x, None, np.concatenate([I, I, I]), None, I, None,
                                 None, None, 1, mask)
        xt = torch.from_numpy(x)[:, None]
        att = torch.nn.functional.scaled_dot_product_attention(xt, xt, xt,
                                                               is_causal=(mask == "causal"))
        ref = torch.nn.functional.layer_norm(torch.from_numpy(x) + att[:, 0], (D,), eps=1e-5)
        np.testing.assert_allclose(y, ref.numpy(), atol=1e-12, rtol=0)


def test_single_head_identity_is_plain_attention():
    check_single_head_identity_is_plain_attention()


# ------------------------------------------------------- library cross-check of the SDPA

def check_sdpa_against_torch():
    g = _rng(12)
    B, H, N, d = 3, 2, 13, 8
    Q, K, V = (g.standard_normal((B, H, N, d)) for _ in range(3))
    key_len = np.array([1, 5, 13], np.int32)
    for mask in ["none", "causal", "key_padding"]:
        O = mha_ref.sdpa_ref(Q, K, V, mask, key_len if mask == "key_padding" else None)
        m = torch.stack([torch.from_numpy(mha_ref.allowed_keys(
            mask, N, N, key_len[b] if mask == "key_padding" else None)) for b in range(B)])[:, None]
        # the mask fed to torch is built here from first principles, not from the oracle:
        i, j = torch.arange(N)[:, None], torch.arange(N)[None, :]
        if mask == "none":
            tm = torch.ones(B, 1, N, N, dtype=torch.bool)
        elif mask == "causal":
            tm = (j <= i).expand(B, 1, N, N)
        else:
            tm = (j < torch.from_numpy(key_len)[:, None, None, None]).expand(B, 1, N, N)
        assert torch.equal(m, tm)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(Q), torch.from_numpy(K), torch.from_numpy(V), attn_mask=tm)
        np.testing.assert_allclose(O, ref.numpy(), atol=1e-12, rtol=0)


def test_sdpa_against_torch():
    check_sdpa_against_torch()


def test_key_len_zero_row_is_zero():
    g = _rng(13)
    Q, K, V = (g.standard_normal((1, 1, 4, 8)) for _ in range(3))
    O = mha_ref.sdpa_ref(Q, K, V, "key_padding", np.array([0], np.int32))
    assert np.array_equal(O, np.zeros_like(O))


def test_causal_needs_square():
    with pytest.raises(ValueError):
        mha_ref.allowed_keys("causal", 3, 4)


# -------------------------------------------------------------- brute force on tiny shapes

def _brute_layer(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H, mask, key_len, eps):
    """Independent loops over b, i, h, j, t with math.exp; no NumPy linear algebra."""
    B, Nq, D = x_q.shape
    src = x_q if x_kv is None else x_kv
    Nk = src.shape[1]
    dk = D // H
    y = np.zeros((B, Nq, D))

    def proj(vec, row0):
        out = []
        for o in range(D):
            acc = float(b_qkv[row0 + o]) if b_qkv is not None else 0.0
            for c in range(D):
                acc += float(W_qkv[row0 + o][c]) * float(vec[c])
            out.append(acc)
        return out

    for b in range(B):
        qs = [proj(x_q[b, i], 0) for i in range(Nq)]
        ks = [proj(src[b, j], D) for j in range(Nk)]
        vs = [proj(src[b, j], 2 * D) for j in range(Nk)]
        for i in range(Nq):
            concat = []
            for h in range(H):
                if mask == "causal":
                    keys = list(range(0, i + 1))
                elif mask == "key_padding":
                    keys = list(range(0, int(key_len[b])))
                else:
                    keys = list(range(Nk))
                scores = []
                for j in keys:
                    dot = 0.0
                    for t in range(dk):
                        dot += qs[i][h * dk + t] * ks[j][h * dk + t]
                    scores.append(dot / math.sqrt(dk))
                head = [0.0] * dk
                if keys:
                    mx = max(scores)
                    ex = [math.exp(s - mx) for s in scores]
                    tot = sum(ex)
                    for jj, j in enumerate(keys):
                        for t in range(dk):
                            head[t] += ex[jj] / tot * vs[j][h * dk + t]
                concat.extend(head)
            r = []
            for o in range(D):
                acc = float(b_o[o]) if b_o is not None else 0.0
                for c in range(D):
                    acc += float(W_o[o][c]) * concat[c]
                r.append(float(x_q[b, i, o]) + acc)
            mu = sum(r) / D
            var = sum((v - mu) ** 2 for v in r) / D
            for o in range(D):
                y[b, i, o] = (r[o] - mu) / math.sqrt(var + eps) * float(gamma[o]) + float(beta[o])
    return y


def check_bruteforce_tiny():
    g = _rng(14)
    for mask, cross in [("none", False), ("causal", False), ("key_padding", True), ("none", True)]:
        B, H, D = 2, 2, 4
        Nq = 5 if mask == "causal" or not cross else 3
        Nk = Nq if not cross else 5
        x_q = g.standard_normal((B, Nq, D))
        x_kv = g.standard_normal((B, Nk, D)) if cross else None
        W_qkv = g.standard_normal((3 * D, D))
        b_qkv = g.standard_normal(3 * D)
        W_o = g.standard_normal((D, D))
        b_o = g.standard_normal(D)
        gamma, beta = g.standard_normal(D), g.standard_normal(D)
        key_len = np.array([2, 5], np.int32) if mask == "key_padding" else None
        y = mha_ref.mha_layer_ref(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H, mask, key_len)
        yb = _brute_layer(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H, mask, key_len, 1e-5)
        np.testing.assert_allclose(y, yb, atol=1e-10, rtol=1e-10)
        for b in range(B):
            rows = np.array([Nq - 1, 0])
            yr = mha_ref.mha_layer_rows_ref(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H, b,
                                           rows, mask, key_len)
            np.testing.assert_allclose(yr, yb[b, rows], atol=1e-10, rtol=1e-10)


def test_bruteforce_tiny():
    check_bruteforce_tiny()


# ----------------------------------------------- planted mistakes: each must trip some pin

def _planted(monkeypatch, name, fn):
    monkeypatch.setattr(mha_ref, name, fn)


def test_plant_dropped_scale_is_caught(monkeypatch):
    orig = mha_ref.attention_weights_ref
    _planted(monkeypatch, "attention_weights_ref",
             lambda q, k, allowed, scale=None: orig(q, k, allowed, scale=1.0))
    with pytest.raises(AssertionError):
        check_worked_example_weights()
    with pytest.raises(AssertionError):
        check_sdpa_against_torch()


def test_plant_strict_causal_is_caught(monkeypatch):
    orig = mha_ref.allowed_keys

    def wrong(mask, Nq, Nk, key_len=None, rows=None):
        a = orig(mask, Nq, Nk, key_len, rows)
        if mask == "causal":
            i = (np.arange(Nq) if rows is None else np.asarray(rows))[:, None]
            a = np.arange(Nk)[None, :] < i  # drops the diagonal
        return a

    _planted(monkeypatch, "allowed_keys", wrong)
    with pytest.raises(AssertionError):
        check_causal_mask_matches_pages()


def test_plant_unbiased_variance_is_caught(monkeypatch):
    def wrong(r, gamma=None, beta=None, eps=1e-5):
        r = np.asarray(r, np.float64)
        mu = r.mean(axis=-1, keepdims=True)
        var = r.var(axis=-1, ddof=1, keepdims=True)
        y = (r - mu) / np.sqrt(var + eps)
        return y * (1 if gamma is None else gamma) + (0 if beta is None else beta)

    _planted(monkeypatch, "layernorm_ref", wrong)
    with pytest.raises(AssertionError):
        check_layernorm_moments()
    with pytest.raises(AssertionError):
        check_single_head_identity_is_plain_attention()


def test_plant_transposed_head_split_is_caught(monkeypatch):
    def wrong(x, H, d):
        *lead, n, _ = x.shape
        return np.moveaxis(x.reshape(*lead, n, d, H), -1, -3)  # heads interleaved, not blocks

    _planted(monkeypatch, "_heads", wrong)
    with pytest.raises(AssertionError):
        check_bruteforce_tiny()


def test_plant_missing_max_subtraction_guard_is_caught(monkeypatch):
    # forgetting to exclude masked keys (adding them with weight) breaks mask invariance
    orig = mha_ref.attention_weights_ref
    _planted(monkeypatch, "attention_weights_ref",
             lambda q, k, allowed, scale=None: orig(q, k, np.ones_like(allowed), scale))
    with pytest.raises(AssertionError):
        check_mask_invariance()
    with pytest.raises(AssertionError):
        check_rows_sum_to_one()
