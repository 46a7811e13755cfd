"""Pins for the backward pass in the CPU oracle ([JY] Transformer 训练样例 > 反向传播: the chain
rule through every step of the sublayer).

The central pin is independent of the analytic formulas: central finite differences of the
FORWARD definition (``oracle.mha_ref``), in float64, on tiny shapes, for every gradient.
Invariants that the mathematics fixes (LayerNorm's input gradient sums to zero per row, key
gradients sum to zero per query block when a common shift of the keys leaves the output
unchanged, keys that no query may see get no gradient) pin the structure.  Planted mistakes
each trip a pin.
"""
import numpy as np
import pytest

from oracle import backward as BW
from oracle import mha_ref


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _fd(f, x, idx, h=1e-6):
    """Central difference of the scalar f at element idx of array x (modified in place)."""
    old = x[idx]
    x[idx] = old + h
    fp = f()
    x[idx] = old - h
    fm = f()
    x[idx] = old
    return (fp - fm) / (2 * h)


def _sample(g, shape, n):
    flat = g.choice(int(np.prod(shape)), size=min(n, int(np.prod(shape))), replace=False)
    return [np.unravel_index(i, shape) for i in flat]


def _layer_case(seed, cross, mask):
    g = _rng(seed)
    B, H, dk = 2, 2, 3
    D = H * dk
    Nq = 4
    Nk = 5 if cross else Nq
    x_q = g.standard_normal((B, Nq, D))
    x_kv = g.standard_normal((B, Nk, D)) if cross else None
    W_qkv = 0.5 * g.standard_normal((3 * D, D))
    b_qkv = 0.3 * g.standard_normal(3 * D)
    W_o = 0.5 * g.standard_normal((D, D))
    b_o = 0.3 * g.standard_normal(D)
    gamma = 1.0 + 0.2 * g.standard_normal(D)
    beta = 0.2 * g.standard_normal(D)
    key_len = np.array([Nk, 2], np.int32) if mask == "key_padding" else None
    G = g.standard_normal((B, Nq, D))  # L = sum(y * G), so dL/dy = G
    return dict(x_q=x_q, x_kv=x_kv, W_qkv=W_qkv, b_qkv=b_qkv, W_o=W_o, b_o=b_o, gamma=gamma,
                beta=beta, key_len=key_len, G=G, H=H, mask=mask)


def check_layer_gradients_match_finite_differences(case, n_per_tensor=12):
    c = case
    loss = lambda: float(np.sum(mha_ref.mha_layer_ref(  # noqa: E731
        c["x_q"], c["x_kv"], c["W_qkv"], c["b_qkv"], c["W_o"], c["b_o"], c["gamma"], c["beta"],
        c["H"], c["mask"], c["key_len"]) * c["G"]))
    grads = BW.mha_layer_bwd_ref(c["x_q"], c["x_kv"], c["W_qkv"], c["b_qkv"], c["W_o"],
                                 c["b_o"], c["gamma"], c["beta"], c["H"], c["G"], c["mask"],
                                 c["key_len"])
    g = _rng(99)
    names = [("x_q", "dx_q"), ("W_qkv", "dW_qkv"), ("b_qkv", "db_qkv"), ("W_o", "dW_o"),
             ("b_o", "db_o"), ("gamma", "dgamma"), ("beta", "dbeta")]
    if c["x_kv"] is not None:
        names.append(("x_kv", "dx_kv"))
    for tname, gname in names:
        t = c[tname]
        for idx in _sample(g, t.shape, n_per_tensor):
            num = _fd(loss, t, idx)
            ana = grads[gname][idx]
            assert abs(num - ana) <= 1e-6 * max(1.0, abs(num)), (tname, idx, num, ana)


@pytest.mark.parametrize("cross,mask", [(False, "none"), (False, "causal"),
                                        (True, "none"), (True, "key_padding")])
def test_layer_gradients_match_finite_differences(cross, mask):
    check_layer_gradients_match_finite_differences(_layer_case(7, cross, mask))


def check_attention_gradients_match_finite_differences(mask="causal", window=None):
    g = _rng(11)
    B, H, N, d = 1, 2, 5, 3
    Q, K, V = (g.standard_normal((B, H, N, d)) for _ in range(3))
    G = g.standard_normal((B, H, N, d))
    loss = lambda: float(np.sum(mha_ref.sdpa_ref(Q, K, V, mask, window=window) * G))  # noqa
    dQ, dK, dV = BW.sdpa_bwd_ref(Q, K, V, G, mask, window=window)
    for t, gt in ((Q, dQ), (K, dK), (V, dV)):
        for idx in _sample(g, t.shape, 15):
            num = _fd(loss, t, idx)
            assert abs(num - gt[idx]) <= 1e-7 * max(1.0, abs(num)), (idx, num, gt[idx])


@pytest.mark.parametrize("mask,window", [("none", None), ("causal", None), ("window", 1)])
def test_attention_gradients_match_finite_differences(mask, window):
    check_attention_gradients_match_finite_differences(mask, window)


def check_layernorm_gradient_structure():
    g = _rng(13)
    r = g.standard_normal((6, 8)) * 2 + 0.5
    gamma = 1 + 0.3 * g.standard_normal(8)
    dy = g.standard_normal((6, 8))
    dr, dgamma, dbeta = BW.layernorm_bwd_ref(r, gamma, dy)
    # LayerNorm ignores a common shift and (up to eps) a common scale of its input row
    assert np.allclose(dr.sum(axis=-1), 0.0, atol=1e-12)
    assert np.allclose((dr * r).sum(axis=-1) - (dr.sum(-1) * r.mean(-1)), 0.0, atol=1e-4)
    loss = lambda: float(np.sum(mha_ref.layernorm_ref(r, gamma, None) * dy))  # noqa: E731
    for idx in _sample(g, r.shape, 10):
        num = _fd(loss, r, idx)
        assert abs(num - dr[idx]) <= 1e-6 * max(1.0, abs(num))
    assert np.allclose(dbeta, dy.sum(axis=0))


def test_layernorm_gradient_structure():
    check_layernorm_gradient_structure()


def check_attention_gradient_invariants():
    g = _rng(17)
    B, H, N, d = 2, 1, 6, 4
    Q, K, V = (g.standard_normal((B, H, N, d)) for _ in range(3))
    dO = g.standard_normal((B, H, N, d))
    # a common shift of every key changes each row's scores by a constant: no effect, so the
    # key gradients sum to zero (no mask; every row sees every key)
    _, dK, _ = BW.sdpa_bwd_ref(Q, K, V, dO, "none")
    assert np.allclose(dK.sum(axis=2), 0.0, atol=1e-12)
    # keys past key_len are seen by no query: exactly zero gradient
    kl = np.array([4, 6], np.int32)
    dQ, dK, dV = BW.sdpa_bwd_ref(Q, K, V, dO, "key_padding", kl)
    assert np.all(dK[0, :, 4:] == 0.0) and np.all(dV[0, :, 4:] == 0.0)
    # causal: the last key is seen only by the last query, so only that query's dO reaches it
    dQc, dKc, dVc = BW.sdpa_bwd_ref(Q, K, V, dO, "causal")
    assert not np.allclose(dVc[:, :, -1], 0.0)
    dO2 = dO.copy()
    dO2[:, :, :-1] = 0.0
    _, _, dV2 = BW.sdpa_bwd_ref(Q, K, V, dO2, "causal")
    assert np.array_equal(dV2[:, :, -1], dVc[:, :, -1])


def test_attention_gradient_invariants():
    check_attention_gradient_invariants()


def test_lse_matches_direct_sum():
    g = _rng(19)
    Q, K = g.standard_normal((1, 2, 4, 3)), g.standard_normal((1, 2, 5, 3))
    lse = BW.sdpa_lse_ref(Q, K, "key_padding", np.array([3], np.int32))
    for h in range(2):
        for i in range(4):
            s = [float(np.dot(Q[0, h, i], K[0, h, j])) / np.sqrt(3) for j in range(3)]
            assert abs(lse[0, h, i] - np.log(sum(np.exp(x) for x in s))) < 1e-12
    assert np.all(np.isinf(BW.sdpa_lse_ref(Q, K, "key_padding", np.array([0], np.int32))))


# ----------------------------------------------- planted mistakes: each must trip some pin

def test_plant_missing_softmax_correction_is_caught(monkeypatch):
    def wrong(q, k, v, allowed, dO, scale=None):
        sc = 1.0 / np.sqrt(q.shape[-1]) if scale is None else float(scale)
        P = mha_ref.attention_weights_ref(q, k, allowed, sc)
        dS = P * (dO @ v.T)  # drops the rowsum(dO * O) term
        return sc * (dS @ k), sc * (dS.T @ q), P.T @ dO

    monkeypatch.setattr(BW, "attention_bwd_ref", wrong)
    with pytest.raises(AssertionError):
        check_attention_gradients_match_finite_differences()
    with pytest.raises(AssertionError):
        check_attention_gradient_invariants()


def test_plant_untransposed_value_gradient_is_caught(monkeypatch):
    orig = BW.attention_bwd_ref

    def wrong(q, k, v, allowed, dO, scale=None):
        dq, dk, _ = orig(q, k, v, allowed, dO, scale)
        sc = 1.0 / np.sqrt(q.shape[-1]) if scale is None else float(scale)
        P = mha_ref.attention_weights_ref(q, k, allowed, sc)
        return dq, dk, P @ dO  # P instead of P^T

    monkeypatch.setattr(BW, "attention_bwd_ref", wrong)
    with pytest.raises(AssertionError):
        check_attention_gradients_match_finite_differences()


def test_plant_layernorm_mean_term_dropped_is_caught(monkeypatch):
    def wrong(r, gamma, dy, eps=1e-5):
        r, dy = np.asarray(r, np.float64), np.asarray(dy, np.float64)
        mu = r.mean(-1, keepdims=True)
        sigma = np.sqrt(((r - mu) ** 2).mean(-1, keepdims=True) + eps)
        rhat = (r - mu) / sigma
        g = dy * (1.0 if gamma is None else gamma)
        dr = (g - rhat * (g * rhat).mean(-1, keepdims=True)) / sigma  # no mean(g)
        D = r.shape[-1]
        return dr, (dy * rhat).reshape(-1, D).sum(0), dy.reshape(-1, D).sum(0)

    monkeypatch.setattr(BW, "layernorm_bwd_ref", wrong)
    with pytest.raises(AssertionError):
        check_layernorm_gradient_structure()
    with pytest.raises(AssertionError):
        check_layer_gradients_match_finite_differences(_layer_case(7, False, "none"))


def test_plant_missing_residual_gradient_is_caught(monkeypatch):
    orig = BW.mha_layer_bwd_ref

    # subtract the residual path's contribution: dx_q loses dr
    def wrong2(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H, dy, mask="none",
               key_len=None, eps=1e-5, d_k=None, d_v=None):
        out = orig(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H, dy, mask, key_len, eps,
                   d_k, d_v)
        y, parts = mha_ref.mha_layer_ref(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H,
                                        mask, key_len, eps, return_parts=True)
        dr, _, _ = BW.layernorm_bwd_ref(np.asarray(x_q) + parts["A"], gamma, dy, eps)
        out["dx_q"] = out["dx_q"] - dr
        return out

    monkeypatch.setattr(BW, "mha_layer_bwd_ref", wrong2)
    with pytest.raises(AssertionError):
        check_layer_gradients_match_finite_differences(_layer_case(7, True, "none"))
