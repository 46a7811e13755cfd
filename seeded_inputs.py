"""Seeded synthetic inputs for the multi-head attention sublayer, the position-wise
feed-forward sublayer and the encoder layer workloads.

This module draws random numbers and rounds them to bf16; it holds none of the
attention method's arithmetic.  Both the CPU oracle (through the tests and the
bench's CPU leg) and the CUDA path take their inputs from here, so the two sides
always see the same values.

Shapes follow the base and big models of "Transformer：抛弃循环与卷积的序列建模"
(section "模型变体与消融实验": d_model=512, h=8, d_k=d_v=64 for the base model;
d_model=1024, h=16 for the big model).  Recipe:

* generator ``numpy.random.Generator(PCG64(seed))``;
* draw order: x (self-attention) or x_q then x_kv (cross-attention), then
  W_q, W_k, W_v, W_o, then key_len (key-padding workloads only);
* activations i.i.d. N(0, 1); each weight matrix Xavier-uniform on
  [-sqrt(6/(D+D)), +sqrt(6/(D+D))], stored as [out, in];
* key_len uniform on [64, 256] inclusive;
* biases 0, gamma 1, beta 0 unless ``affine=True`` asks for random ones
  (drawn after everything above, so the main draws do not move);
* every floating value is rounded to bf16 (round-to-nearest-even) for the bf16
  workloads; fp32 workloads keep float32 values.

Feed-forward workloads use the pages' inner sizes (d_ff = 2048 for the base model, 4096 for
the big one): x ~ N(0, 1) [B, N, D], then W1 [d_ff, D] and W2 [D, d_ff], each
Xavier-uniform on [-sqrt(6/(D+d_ff)), +sqrt(6/(D+d_ff))]; b1, b2 are 0 (or, with
``affine=True``, 0.1 N(0, 1)), gamma 1 and beta 0 (or 1 + 0.1 N(0, 1) and 0.1 N(0, 1)).
An encoder-layer workload draws the attention sublayer's inputs exactly as ``draw_layer``
does and then, from a second generator seeded with seed + 1, the feed-forward weights.
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "round_bf16",
    "draw_sdpa",
    "draw_layer",
    "draw_qkv",
    "draw_ffn",
    "draw_encoder",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str  # "sdpa", "layer", "ffn" or "encoder"
    dtype: str  # "f32" or "bf16"
    B: int
    H: int
    Nq: int
    Nk: int
    d_k: int = 64
    d_v: int = 64
    mask: str = "none"  # "none" | "causal" | "key_padding"
    cross: bool = False
    seed: int = 0
    d_ff: int = 0  # feed-forward inner size ("ffn" and "encoder" workloads)

    @property
    def D(self) -> int:
        return self.H * self.d_k

    def with_mask(self, mask: str) -> "Workload":
        return dataclasses.replace(self, mask=mask, name=f"{self.name}_{mask}")


WORKLOADS = {
    w.name: w
    for w in [
        Workload("sdpa_f32_b1_h8_n32", "sdpa", "f32", B=1, H=8, Nq=32, Nk=32, seed=20260001),
        Workload("enc_self_base_b32_n128", "layer", "bf16", B=32, H=8, Nq=128, Nk=128, seed=20260002),
        Workload("dec_causal_base_b32_n256", "layer", "bf16", B=32, H=8, Nq=256, Nk=256,
                 mask="causal", seed=20260003),
        Workload("cross_pad_base_b32_q128_k256", "layer", "bf16", B=32, H=8, Nq=128, Nk=256,
                 mask="key_padding", cross=True, seed=20260004),
        Workload("big_long_b8_n4096", "layer", "bf16", B=8, H=16, Nq=4096, Nk=4096, seed=20260005),
        # position-wise feed-forward sublayer (D = H * d_k; H only fixes D here)
        Workload("ffn_f32_b2_n50", "ffn", "f32", B=2, H=1, Nq=50, Nk=50, d_ff=256, seed=20260006),
        Workload("ffn_base_b32_n128", "ffn", "bf16", B=32, H=8, Nq=128, Nk=128, d_ff=2048,
                 seed=20260007),
        Workload("ffn_big_b8_n4096", "ffn", "bf16", B=8, H=16, Nq=4096, Nk=4096, d_ff=4096,
                 seed=20260008),
        # encoder layer: self-attention sublayer, then feed-forward sublayer
        Workload("encoder_base_b32_n128", "encoder", "bf16", B=32, H=8, Nq=128, Nk=128,
                 d_ff=2048, seed=20260009),
        Workload("encoder_base_pad_b32_n128", "encoder", "bf16", B=32, H=8, Nq=128, Nk=128,
                 d_ff=2048, mask="key_padding", seed=20260010),
    ]
}


def round_bf16(a) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even); returns float32 holding bf16 values."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).reshape(f.shape)


def _finish(a: np.ndarray, dtype: str) -> np.ndarray:
    return round_bf16(a) if dtype == "bf16" else np.asarray(a, dtype=np.float32)


def draw_sdpa(B, H, Nq, Nk, d_k=64, d_v=64, dtype="f32", seed=0, key_len_range=(64, 256),
              mask="none"):
    """Q [B,H,Nq,d_k], K [B,H,Nk,d_k], V [B,H,Nk,d_v] ~ N(0,1); key_len int32[B] if key padding."""
    g = np.random.Generator(np.random.PCG64(seed))
    Q = _finish(g.standard_normal((B, H, Nq, d_k)), dtype)
    K = _finish(g.standard_normal((B, H, Nk, d_k)), dtype)
    V = _finish(g.standard_normal((B, H, Nk, d_v)), dtype)
    key_len = None
    if mask == "key_padding":
        lo, hi = key_len_range
        key_len = g.integers(lo, hi + 1, size=B).astype(np.int32)
    return Q, K, V, key_len


def draw_qkv(w: Workload):
    """Raw per-head Q/K/V for an ``sdpa`` workload."""
    return draw_sdpa(w.B, w.H, w.Nq, w.Nk, w.d_k, w.d_v, w.dtype, w.seed, mask=w.mask)


def draw_layer(w: Workload, affine: bool = False, batch: slice | None = None):
    """All inputs of one sublayer call, as float32 arrays (bf16-exact for bf16 workloads).

    Returns a dict with x_q [B,Nq,D], x_kv [B,Nk,D] (None for self-attention),
    W_qkv [3D,D] (rows: Q heads 0..H-1, then K, then V), b_qkv [3D], W_o [D,H*d_v],
    b_o [D], gamma [D], beta [D], key_len int32[B] or None.
    ``batch`` keeps only some batch rows of x_q/x_kv/key_len after drawing all of them.
    """
    g = np.random.Generator(np.random.PCG64(w.seed))
    D, dt = w.D, w.dtype
    x_q = _finish(g.standard_normal((w.B, w.Nq, D)), dt)
    x_kv = _finish(g.standard_normal((w.B, w.Nk, D)), dt) if w.cross else None
    bound = float(np.sqrt(6.0 / (D + D)))
    W_q = _finish(g.uniform(-bound, bound, (w.H * w.d_k, D)), dt)
    W_k = _finish(g.uniform(-bound, bound, (w.H * w.d_k, D)), dt)
    W_v = _finish(g.uniform(-bound, bound, (w.H * w.d_v, D)), dt)
    bound_o = float(np.sqrt(6.0 / (w.H * w.d_v + D)))
    W_o = _finish(g.uniform(-bound_o, bound_o, (D, w.H * w.d_v)), dt)
    key_len = None
    if w.mask == "key_padding":
        key_len = g.integers(64, 257, size=w.B).astype(np.int32)
    W_qkv = np.concatenate([W_q, W_k, W_v], axis=0)
    n_qkv = W_qkv.shape[0]
    if affine:
        b_qkv = _finish(0.1 * g.standard_normal(n_qkv), dt)
        b_o = _finish(0.1 * g.standard_normal(D), dt)
        gamma = _finish(1.0 + 0.1 * g.standard_normal(D), dt)
        beta = _finish(0.1 * g.standard_normal(D), dt)
    else:
        b_qkv = np.zeros(n_qkv, np.float32)
        b_o = np.zeros(D, np.float32)
        gamma = np.ones(D, np.float32)
        beta = np.zeros(D, np.float32)
    if batch is not None:
        x_q = x_q[batch]
        x_kv = x_kv[batch] if x_kv is not None else None
        key_len = key_len[batch] if key_len is not None else None
    return dict(x_q=x_q, x_kv=x_kv, W_qkv=W_qkv, b_qkv=b_qkv, W_o=W_o, b_o=b_o,
                gamma=gamma, beta=beta, key_len=key_len)


def _ffn_weights(g, D: int, d_ff: int, dt: str, affine: bool):
    bound = float(np.sqrt(6.0 / (D + d_ff)))
    W1 = _finish(g.uniform(-bound, bound, (d_ff, D)), dt)
    W2 = _finish(g.uniform(-bound, bound, (D, d_ff)), dt)
    if affine:
        b1 = _finish(0.1 * g.standard_normal(d_ff), dt)
        b2 = _finish(0.1 * g.standard_normal(D), dt)
        gamma = _finish(1.0 + 0.1 * g.standard_normal(D), dt)
        beta = _finish(0.1 * g.standard_normal(D), dt)
    else:
        b1 = np.zeros(d_ff, np.float32)
        b2 = np.zeros(D, np.float32)
        gamma = np.ones(D, np.float32)
        beta = np.zeros(D, np.float32)
    return dict(W1=W1, b1=b1, W2=W2, b2=b2, gamma=gamma, beta=beta)


def draw_ffn(w: Workload, affine: bool = False, batch: slice | None = None):
    """Inputs of one feed-forward sublayer call: x [B,N,D], W1 [d_ff,D], b1 [d_ff],
    W2 [D,d_ff], b2 [D], gamma [D], beta [D] (float32, bf16-exact for bf16 workloads).
    ``batch`` keeps only some batch rows of x after drawing all of it."""
    g = np.random.Generator(np.random.PCG64(w.seed))
    x = _finish(g.standard_normal((w.B, w.Nq, w.D)), w.dtype)
    out = _ffn_weights(g, w.D, w.d_ff, w.dtype, affine)
    out["x"] = x[batch] if batch is not None else x
    return out


def draw_encoder(w: Workload, affine: bool = False):
    """Inputs of one encoder layer: the attention sublayer's (``draw_layer``: x_q is the
    layer input, x_kv None) plus the feed-forward weights W1, b1, W2, b2, gamma2, beta2."""
    att = draw_layer(w, affine=affine)
    g = np.random.Generator(np.random.PCG64(w.seed + 1))
    f = _ffn_weights(g, w.D, w.d_ff, w.dtype, affine)
    att.update(W1=f["W1"], b1=f["b1"], W2=f["W2"], b2=f["b2"], gamma2=f["gamma"],
               beta2=f["beta"])
    return att
