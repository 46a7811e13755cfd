"""Plain float64 backward pass of the multi-head attention sublayer (CPU, NumPy).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the bench's
CPU-baseline leg, never by the product path.  ``numpy`` matmul is the only library
primitive; every step is the chain rule applied to one step of ``oracle.mha_ref``'s forward
definition, in reverse order, with nothing fused or reordered.

Source: "Transformer：抛弃循环与卷积的序列建模" (jiashun-ye.github.io), Transformer 训练样例 >
反向传播: after the loss, back-propagation applies the chain rule backwards through every
step, so that the projections W^Q, W^K, W^V of each head, W^O and the LayerNorm parameters
all receive gradients.  The forward steps are those of ``oracle.mha_ref`` ([LT] 3.1, 3.2.1,
3.2.2).

Conventions: a gradient has the shape of its tensor; ``dy`` is dL/dy for the sublayer output
y; weights are [out, in] as in the forward (so dW = dOut^T In).  The sums over positions
(dW, db, dgamma, dbeta) run over every token of every batch element.
"""
from __future__ import annotations

import numpy as np

from .mha_ref import _heads, _split_weights, allowed_keys, attention_weights_ref, linear_ref


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def layernorm_bwd_ref(r, gamma, dy, eps: float = 1e-5):
    """Backward of y = (r - mean) / sqrt(var + eps) * gamma + beta over the last axis.

    With rhat = (r - mean) / sigma and g = dy * gamma:
    dr = (g - mean(g) - rhat * mean(g * rhat)) / sigma, dgamma = sum(dy * rhat),
    dbeta = sum(dy) (sums over all rows).  Biased variance, as in the forward.
    """
    r, dy = _f64(r), _f64(dy)
    D = r.shape[-1]
    mu = r.mean(axis=-1, keepdims=True)
    var = ((r - mu) ** 2).mean(axis=-1, keepdims=True)
    sigma = np.sqrt(var + eps)
    rhat = (r - mu) / sigma
    g = dy * (1.0 if gamma is None else _f64(gamma))
    dr = (g - g.mean(axis=-1, keepdims=True)
          - rhat * (g * rhat).mean(axis=-1, keepdims=True)) / sigma
    dgamma = (dy * rhat).reshape(-1, D).sum(axis=0)
    dbeta = dy.reshape(-1, D).sum(axis=0)
    return dr, dgamma, dbeta


def attention_bwd_ref(q, k, v, allowed, dO, scale=None):
    """Backward of one (batch, head): O = P V with P = softmax(q k^T * scale over allowed).

    dV = P^T dO; dP = dO V^T; dS = P * (dP - rowsum(dO * O)) (the softmax Jacobian row by
    row); dq = scale * dS k; dk = scale * dS^T q.  Excluded keys have P = 0, so they get no
    gradient.  Returns dq, dk, dv.
    """
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    sc = 1.0 / np.sqrt(q.shape[-1]) if scale is None else float(scale)
    P = attention_weights_ref(q, k, allowed, sc)
    O = P @ v
    dV = P.T @ dO
    dP = dO @ v.T
    Drow = (dO * O).sum(axis=1, keepdims=True)
    dS = P * (dP - Drow)
    return sc * (dS @ k), sc * (dS.T @ q), dV


def sdpa_bwd_ref(Q, K, V, dO, mask: str = "none", key_len=None, scale=None, window=None):
    """dQ, dK, dV of Attention(Q,K,V) per (batch, head) for the given mask ([LT] 3.2.1)."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, Nq, _ = Q.shape
    Nk = K.shape[2]
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for b in range(B):
        allowed = allowed_keys(mask, Nq, Nk, None if key_len is None else key_len[b],
                               window=window)
        for h in range(H):
            dQ[b, h], dK[b, h], dV[b, h] = attention_bwd_ref(Q[b, h], K[b, h], V[b, h],
                                                             allowed, dO[b, h], scale)
    return dQ, dK, dV


def sdpa_lse_ref(Q, K, mask: str = "none", key_len=None, scale=None, window=None):
    """Natural log of sum_j exp(q . k_j * scale) over each row's allowed keys (-inf-free:
    +inf for a row with no allowed key, so that exp(s - lse) = 0 there)."""
    Q, K = _f64(Q), _f64(K)
    B, H, Nq, dk = Q.shape
    Nk = K.shape[2]
    sc = 1.0 / np.sqrt(dk) if scale is None else float(scale)
    out = np.zeros((B, H, Nq))
    for b in range(B):
        allowed = allowed_keys(mask, Nq, Nk, None if key_len is None else key_len[b],
                               window=window)
        for h in range(H):
            s = np.where(allowed, Q[b, h] @ K[b, h].T * sc, -np.inf)
            m = s.max(axis=1)
            has = allowed.any(axis=1)
            m0 = np.where(has, m, 0.0)
            tot = np.exp(s - m0[:, None]).sum(axis=1)
            out[b, h] = np.where(has, m0 + np.log(np.where(has, tot, 1.0)), np.inf)
    return out


def mha_layer_bwd_ref(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H: int, dy,
                      mask: str = "none", key_len=None, eps: float = 1e-5,
                      d_k: int | None = None, d_v: int | None = None) -> dict:
    """Gradients of y = LayerNorm(x_q + MultiHead(x_q, x_kv, x_kv)) for dL/dy = dy.

    Forward steps recomputed exactly as ``oracle.mha_ref.mha_layer_ref`` takes them, then
    walked backwards: LayerNorm, residual (dx_q gets dr directly), W^O (dC = dA W^O,
    dW^O = dA^T C, db_o = sum dA), head concat (dO = split of dC), attention per head,
    head split (dQ_f = concat of dQ heads, likewise K, V), and the three projections
    (dx += dQ_f W^Q etc.; dW^Q = dQ_f^T x_q ...).  Self-attention (x_kv None) adds the
    key/value projections' input gradient to dx_q.  Returns dx_q, dx_kv (None for
    self-attention), dW_qkv, db_qkv, dW_o, db_o, dgamma, dbeta.
    """
    x_q = _f64(x_q)
    self_attn = x_kv is None
    x_kv = x_q if self_attn else _f64(x_kv)
    dy = _f64(dy)
    B, Nq, D = x_q.shape
    Nk = x_kv.shape[1]
    d_k = D // H if d_k is None else d_k
    d_v = D // H if d_v is None else d_v
    Wq, Wk, Wv, bq, bk, bv = _split_weights(W_qkv, b_qkv, H, d_k, d_v)
    W_o = _f64(W_o)
    # forward, step by step
    Qf, Kf, Vf = linear_ref(x_q, Wq, bq), linear_ref(x_kv, Wk, bk), linear_ref(x_kv, Wv, bv)
    Q, K, V = _heads(Qf, H, d_k), _heads(Kf, H, d_k), _heads(Vf, H, d_v)
    P = np.zeros((B, H, Nq, Nk))
    for b in range(B):
        allowed = allowed_keys(mask, Nq, Nk, None if key_len is None else key_len[b])
        for h in range(H):
            P[b, h] = attention_weights_ref(Q[b, h], K[b, h], allowed)
    O = P @ V
    C = np.moveaxis(O, 1, 2).reshape(B, Nq, H * d_v)
    A = linear_ref(C, W_o, b_o)
    r = x_q + A
    # backward
    dr, dgamma, dbeta = layernorm_bwd_ref(r, gamma, dy, eps)
    dA = dr
    dx_q = dr.copy()
    dC = dA @ W_o
    dW_o = dA.reshape(-1, D).T @ C.reshape(-1, H * d_v)
    db_o = dA.reshape(-1, D).sum(axis=0)
    dO = _heads(dC, H, d_v)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    for b in range(B):
        allowed = allowed_keys(mask, Nq, Nk, None if key_len is None else key_len[b])
        for h in range(H):
            dQ[b, h], dK[b, h], dV[b, h] = attention_bwd_ref(Q[b, h], K[b, h], V[b, h],
                                                             allowed, dO[b, h])
    dQf = np.moveaxis(dQ, 1, 2).reshape(B, Nq, H * d_k)
    dKf = np.moveaxis(dK, 1, 2).reshape(B, Nk, H * d_k)
    dVf = np.moveaxis(dV, 1, 2).reshape(B, Nk, H * d_v)
    dx_q = dx_q + dQf @ Wq
    dx_kv = dKf @ Wk + dVf @ Wv
    dWq = dQf.reshape(-1, H * d_k).T @ x_q.reshape(-1, D)
    dWk = dKf.reshape(-1, H * d_k).T @ x_kv.reshape(-1, D)
    dWv = dVf.reshape(-1, H * d_v).T @ x_kv.reshape(-1, D)
    db_qkv = np.concatenate([dQf.reshape(-1, H * d_k).sum(axis=0),
                             dKf.reshape(-1, H * d_k).sum(axis=0),
                             dVf.reshape(-1, H * d_v).sum(axis=0)])
    if self_attn:
        dx_q = dx_q + dx_kv
        dx_kv = None
    return dict(dx_q=dx_q, dx_kv=dx_kv, dW_qkv=np.concatenate([dWq, dWk, dWv], axis=0),
                db_qkv=db_qkv, dW_o=dW_o, db_o=db_o, dgamma=dgamma, dbeta=dbeta)
