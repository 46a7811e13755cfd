"""Plain float64 definition of the multi-head attention sublayer (CPU, NumPy).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the bench's
CPU-baseline leg, never by the product path.  Nothing here is blocked, fused or
reordered beyond what the definitions say; ``numpy`` matmul is the only library
primitive used.  Inputs of any float dtype are upcast exactly to float64.

Sources (page title, then section):

* [LT] "Attention Is All You Need" Chinese translation on lettle.cn --
  3.1 Encoder and Decoder Stacks; 3.2.1 缩放点积注意力; 3.2.2 多头注意力.
* [TC] "Transformer 为什么抛弃循环网络" on treecat.cn -- 一次注意力计算在做什么;
  为什么需要多头注意力; 编码器和解码器.
* [JY] "Transformer：抛弃循环与卷积的序列建模" on jiashun-ye.github.io --
  Scaled Dot-Product Attention; Multi-Head Attention; Transformer 中的三种 Attention;
  Residual Connection 与 LayerNorm; Transformer 翻译样例 (Encoder / Decoder);
  Transformer 训练样例 (训练样本, 反向传播).

Readings where the pages leave a step open (each one is also listed in the design notes):

* LayerNorm: mean and biased variance over the d_model features, eps added to the
  variance, then per-feature gamma and beta.  The pages name LayerNorm but never
  write its formula.
* Projection biases are optional (None means zero): the pages write the head
  projections without biases.
* Masked scores are excluded exactly (weight 0), the reading of "-inf before the
  softmax, e^-inf = 0" in [JY] 训练样本.
* A query row with no allowed key (only possible with key_len = 0) has output 0.
* Causal masking is defined only for Nq == Nk (self-attention); other shapes raise.
* Key padding keeps keys j < key_len[b] of batch element b; queries are not masked.
* Restricted self-attention ([JY] Self-Attention的优势, 总结): each position attends only
  a neighbourhood of size r; the pages give its size and its O(r n d) cost but not where it
  sits, so it is read as centred on the query: keys j with |i - j| <= w, r = 2 w + 1.
* Autoregressive decoding ([JY] Transformer 翻译样例 > Decoder, Transformer 训练样例): at each
  step the newest target positions attend every earlier position and themselves.  Keys and
  values of earlier positions never change under the causal mask, so they are read from a
  cache of the first L = key_len[b] positions; the Nq new queries are the last Nq of those L
  positions (query i sits at position L - Nq + i): the causal mask aligned bottom-right.
"""
from __future__ import annotations

import numpy as np

MASKS = ("none", "causal", "key_padding", "window", "causal_cache")


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def allowed_keys(mask: str, Nq: int, Nk: int, key_len: int | None = None,
                 rows: np.ndarray | None = None, window: int | None = None) -> np.ndarray:
    """Boolean [len(rows), Nk] table: True where query row i may attend key j.

    * "none": every key ([LT] 3.2.1: the query is compared with all keys).
    * "causal": j <= i, the current position and those before it ([JY] Transformer 中的
      三种 Attention; the 4x4 matrix M of [JY] 训练样本 has its diagonal allowed).
    * "key_padding": j < key_len ([JY] 反向传播: padded <PAD> positions are excluded by a
      padding mask; here the mask is applied to the keys).
    * "window": |i - j| <= window, the neighbourhood of restricted self-attention ([JY]
      Self-Attention的优势), self-attention only.
    * "causal_cache": decoding against a cache holding the first L = key_len positions; query
      i is position L - Nq + i and attends j <= L - Nq + i ([JY] Transformer 翻译样例 >
      Decoder: the masked self-attention of one generation step).
    """
    if mask not in MASKS:
        raise ValueError(f"unknown mask kind {mask!r}")
    i = (np.arange(Nq) if rows is None else np.asarray(rows))[:, None]
    j = np.arange(Nk)[None, :]
    if mask == "none":
        return np.ones((i.shape[0], Nk), dtype=bool)
    if mask == "causal":
        if Nq != Nk:
            raise ValueError("causal mask needs Nq == Nk")
        return j <= i
    if mask == "window":
        if Nq != Nk:
            raise ValueError("window mask needs Nq == Nk")
        if window is None or int(window) < 0:
            raise ValueError("window mask needs a radius window >= 0")
        return np.abs(j - i) <= int(window)
    if key_len is None:
        raise ValueError(f"{mask} needs key_len")
    L = min(max(int(key_len), 0), Nk)
    if mask == "causal_cache":
        if Nq > L:
            raise ValueError("causal_cache needs Nq <= key_len (the new queries are cached)")
        return j <= (L - Nq) + i
    return np.broadcast_to(j < L, (i.shape[0], Nk)).copy()


def attention_weights_ref(q, k, allowed, scale=None) -> np.ndarray:
    """softmax(q k^T / sqrt(d_k)) over the allowed keys, one (batch, head) pair.

    q [n, d_k], k [Nk, d_k], allowed bool [n, Nk].  [LT] 3.2.1 and [JY] Scaled
    Dot-Product Attention: dot products with all keys, divided by sqrt(d_k), softmax
    over the keys.  Subtracting the row maximum leaves the softmax unchanged and keeps
    exp finite.  Disallowed keys get weight exactly 0; rows with no allowed key are 0.
    """
    q, k = _f64(q), _f64(k)
    d_k = q.shape[-1]
    s = q @ k.T
    s = s / np.sqrt(d_k) if scale is None else s * float(scale)
    s = np.where(allowed, s, -np.inf)
    has_any = allowed.any(axis=1)
    m = np.where(has_any, np.max(s, axis=1), 0.0)
    e = np.exp(s - m[:, None])  # exp(-inf) = 0 for excluded keys
    tot = e.sum(axis=1)
    w = np.zeros_like(e)
    w[has_any] = e[has_any] / tot[has_any, None]
    return w


def sdpa_ref(Q, K, V, mask: str = "none", key_len=None, scale=None,
             window: int | None = None) -> np.ndarray:
    """Attention(Q,K,V) = softmax(QK^T/sqrt(d_k)) V per (batch, head).

    Q [B,H,Nq,d_k], K [B,H,Nk,d_k], V [B,H,Nk,d_v] -> O [B,H,Nq,d_v] (float64).
    [LT] 3.2.1; the output is the weight-averaged values ([JY] Scaled Dot-Product Attention).
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, Nq, _ = Q.shape
    Nk = K.shape[2]
    O = np.zeros((B, H, Nq, V.shape[3]))
    for b in range(B):
        allowed = allowed_keys(mask, Nq, Nk, None if key_len is None else key_len[b],
                               window=window)
        for h in range(H):
            w = attention_weights_ref(Q[b, h], K[b, h], allowed, scale)
            O[b, h] = w @ V[b, h]
    return O


def linear_ref(x, W, b=None) -> np.ndarray:
    """x W^T + b with W stored [out, in] ([JY] Multi-Head Attention: Q_i = X W_i^Q)."""
    y = _f64(x) @ _f64(W).T
    if b is not None:
        y = y + _f64(b)
    return y


def layernorm_ref(r, gamma=None, beta=None, eps: float = 1e-5) -> np.ndarray:
    """LayerNorm over the last axis: (r - mean) / sqrt(var + eps) * gamma + beta.

    The variance is the biased one (divide by the feature count).  [LT] 3.1 and [JY]
    Residual Connection 与 LayerNorm name the normalisation; its formula is this reading.
    """
    r = _f64(r)
    mu = r.mean(axis=-1, keepdims=True)
    var = ((r - mu) ** 2).mean(axis=-1, keepdims=True)
    y = (r - mu) / np.sqrt(var + eps)
    if gamma is not None:
        y = y * _f64(gamma)
    if beta is not None:
        y = y + _f64(beta)
    return y


def _split_weights(W_qkv, b_qkv, H, d_k, d_v):
    W_qkv = _f64(W_qkv)
    b_qkv = None if b_qkv is None else _f64(b_qkv)
    nq, nk, nv = H * d_k, H * d_k, H * d_v
    Wq, Wk, Wv = W_qkv[:nq], W_qkv[nq:nq + nk], W_qkv[nq + nk:nq + nk + nv]
    if b_qkv is None:
        bq = bk = bv = None
    else:
        bq, bk, bv = b_qkv[:nq], b_qkv[nq:nq + nk], b_qkv[nq + nk:nq + nk + nv]
    return Wq, Wk, Wv, bq, bk, bv


def _heads(x, H, d):
    """[..., n, H*d] -> [..., H, n, d]: head h takes features [h*d, (h+1)*d)."""
    *lead, n, _ = x.shape
    return np.moveaxis(x.reshape(*lead, n, H, d), -2, -3)


def mha_layer_ref(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H: int,
                  mask: str = "none", key_len=None, eps: float = 1e-5,
                  d_k: int | None = None, d_v: int | None = None,
                  return_parts: bool = False):
    """y = LayerNorm(x_q + MultiHead(x_q, x_kv, x_kv)), one post-norm attention sublayer.

    * Head projections Q_i = x_q W_i^Q, K_i = x_kv W_i^K, V_i = x_kv W_i^V, each from the full
      d_model vector ([LT] 3.2.2, [JY] Multi-Head Attention).  x_kv=None means self-attention
      (x_kv = x_q); cross-attention takes queries from the decoder side and keys/values from
      the encoder output ([JY] Transformer 中的三种 Attention, Decoder).
    * head_i = Attention(Q_i, K_i, V_i) (``sdpa_ref``).
    * MultiHead = Concat(head_1..head_h) W^O, heads in order along the features ([TC]
      为什么需要多头注意力, [JY] Encoder: 8 heads of n x 64 concatenate to n x 512).
    * Output LayerNorm(x + Sublayer(x)) with x = x_q ([LT] 3.1; [JY] Residual Connection 与
      LayerNorm; [JY] Decoder for the cross-attention residual).

    Shapes: x_q [B,Nq,D], x_kv [B,Nk,D] or None, W_qkv [H*(2 d_k + d_v), D] rows Q then K then V,
    W_o [D, H*d_v].  Returns y [B,Nq,D] in float64 (and a dict of intermediates if asked).
    """
    x_q = _f64(x_q)
    src = x_q if x_kv is None else _f64(x_kv)
    B, Nq, D = x_q.shape
    Nk = src.shape[1]
    d_k = D // H if d_k is None else d_k
    d_v = D // H if d_v is None else d_v
    Wq, Wk, Wv, bq, bk, bv = _split_weights(W_qkv, b_qkv, H, d_k, d_v)
    Q = _heads(linear_ref(x_q, Wq, bq), H, d_k)
    K = _heads(linear_ref(src, Wk, bk), H, d_k)
    V = _heads(linear_ref(src, Wv, bv), H, d_v)
    O = sdpa_ref(Q, K, V, mask, key_len)
    C = np.moveaxis(O, 1, 2).reshape(B, Nq, H * d_v)  # concat heads in order
    A = linear_ref(C, W_o, b_o)
    y = layernorm_ref(x_q + A, gamma, beta, eps)
    if return_parts:
        return y, dict(Q=Q, K=K, V=V, O=O, C=C, A=A)
    return y


def mha_layer_rows_ref(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H: int, b: int,
                       rows, mask: str = "none", key_len=None, eps: float = 1e-5,
                       d_k: int | None = None, d_v: int | None = None) -> np.ndarray:
    """The same definition as ``mha_layer_ref``, evaluated only at query rows ``rows`` of
    batch element ``b`` (keys and values of that element are projected in full).

    Returns y[b, rows] [len(rows), D] in float64.
    """
    rows = np.asarray(rows)
    xq_b = _f64(x_q[b])
    src_b = xq_b if x_kv is None else _f64(x_kv[b])
    Nq, D = xq_b.shape
    Nk = src_b.shape[0]
    d_k = D // H if d_k is None else d_k
    d_v = D // H if d_v is None else d_v
    Wq, Wk, Wv, bq, bk, bv = _split_weights(W_qkv, b_qkv, H, d_k, d_v)
    xr = xq_b[rows]
    Q = _heads(linear_ref(xr, Wq, bq), H, d_k)      # [H, n, d_k]
    K = _heads(linear_ref(src_b, Wk, bk), H, d_k)   # [H, Nk, d_k]
    V = _heads(linear_ref(src_b, Wv, bv), H, d_v)
    allowed = allowed_keys(mask, Nq, Nk, None if key_len is None else key_len[b], rows=rows)
    O = np.stack([attention_weights_ref(Q[h], K[h], allowed) @ V[h] for h in range(H)])
    C = np.moveaxis(O, 0, 1).reshape(len(rows), H * d_v)
    A = linear_ref(C, W_o, b_o)
    return layernorm_ref(xr + A, gamma, beta, eps)
