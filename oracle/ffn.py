"""Plain float64 definition of the position-wise feed-forward sublayer and of the encoder
layer it completes (CPU, NumPy).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the bench's
CPU-baseline leg, never by the product path.  ``numpy`` matmul is the only library
primitive; nothing is blocked, fused or reordered beyond the definitions.

Sources (page title, then section):

* [LT] "Attention Is All You Need" Chinese translation on lettle.cn -- 3.1 Encoder and
  Decoder Stacks: each encoder layer is a self-attention sublayer followed by a simple
  position-wise fully connected feed-forward sublayer, each wrapped as
  LayerNorm(x + Sublayer(x)).
* [TC] "Transformer 为什么抛弃循环网络" on treecat.cn -- 编码器和解码器: the same parameters
  at every position, 512 -> 2048 -> ReLU -> 512 in the base model, and the formula
  FFN(x) = max(0, x W1 + b1) W2 + b2.
* [LC] "Attention Is All You Need" on likecs.com -- 1.3 按地址的前向反馈网络: two linear maps
  with a ReLU between them, applied to each position separately and identically (like two
  convolutions of kernel size 1); d_model = 512, d_ff = 2048.
* [JY] "Transformer：抛弃循环与卷积的序列建模" on jiashun-ye.github.io -- FFN (position-wise:
  no mixing of positions), Residual Connection 与 LayerNorm, Encoder-Decoder (an encoder
  layer is Multi-Head Self-Attention then FFN), 模型变体与消融实验 (big model: d_model 1024,
  d_ff 4096, 16 heads).

Readings (also listed in the design notes): weights are stored in the [out, in] layout, so
x W1 of the pages is x @ W1.T here; biases are optional (None = 0); LayerNorm is the
biased-variance reading of ``oracle.mha_ref.layernorm_ref``.
"""
from __future__ import annotations

import numpy as np

from .mha_ref import layernorm_ref, linear_ref, mha_layer_ref


def relu_ref(z) -> np.ndarray:
    """max(0, z) elementwise ([TC] 编码器和解码器; [JY] FFN)."""
    z = np.asarray(z, dtype=np.float64)
    return np.where(z > 0.0, z, 0.0)


def ffn_ref(x, W1, b1, W2, b2) -> np.ndarray:
    """FFN(x) = max(0, x W1 + b1) W2 + b2 on every row (position) of x.

    x [..., D]; W1 [d_ff, D]; W2 [D, d_ff] (the [out, in] layout).  [TC] 编码器和解码器;
    [LC] 1.3; [JY] FFN.
    """
    hidden = relu_ref(linear_ref(x, W1, b1))
    return linear_ref(hidden, W2, b2)


def ffn_layer_ref(x, W1, b1, W2, b2, gamma=None, beta=None, eps: float = 1e-5,
                  return_parts: bool = False):
    """y = LayerNorm(x + FFN(x)), one post-norm feed-forward sublayer ([LT] 3.1; [JY]
    Residual Connection 与 LayerNorm)."""
    x = np.asarray(x, dtype=np.float64)
    f = ffn_ref(x, W1, b1, W2, b2)
    y = layernorm_ref(x + f, gamma, beta, eps)
    if return_parts:
        return y, {"ffn": f}
    return y


def encoder_layer_ref(x, W_qkv, b_qkv, W_o, b_o, gamma1, beta1, W1, b1, W2, b2, gamma2,
                      beta2, H: int, mask: str = "none", key_len=None,
                      eps: float = 1e-5, return_parts: bool = False):
    """One encoder layer ([LT] 3.1; [JY] Encoder-Decoder):
    h = LayerNorm(x + MultiHead(x, x, x)), then y = LayerNorm(h + FFN(h))."""
    h = mha_layer_ref(x, None, W_qkv, b_qkv, W_o, b_o, gamma1, beta1, H, mask, key_len, eps)
    y = ffn_layer_ref(h, W1, b1, W2, b2, gamma2, beta2, eps)
    if return_parts:
        return y, {"h": h}
    return y
