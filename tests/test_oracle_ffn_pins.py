"""Pins for the feed-forward and encoder-layer parts of the CPU oracle: facts the pages and the
mathematics fix, independent of the oracle's own code.

Each ``check_*`` raises AssertionError when the oracle breaks the fact it pins; the
planted-mistake tests at the end swap a wrong step into the oracle (on the CPU) and show that
a pin catches it.
"""
import json
import os

import numpy as np
import pytest

from oracle import ffn as F
from oracle import mha_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


# ------------------------------------------- closed form: relu(z) - relu(-z) = z

def check_identity_pair():
    # W1 = [I; -I], W2 = [I, -I]: the hidden layer holds relu(x) and relu(-x), and their
    # difference is x again, so FFN(x) = x exactly (ReLU of [TC] 编码器和解码器).
    g = _rng(1)
    D = 6
    x = g.standard_normal((5, D))
    I = np.eye(D)
    W1 = np.concatenate([I, -I], axis=0)   # [2D, D]
    W2 = np.concatenate([I, -I], axis=1)   # [D, 2D]
    f = F.ffn_ref(x, W1, None, W2, None)
    assert np.array_equal(f, x)
    # and a bias b2 is added after the second map
    b2 = g.standard_normal(D)
    assert np.allclose(F.ffn_ref(x, W1, None, W2, b2), x + b2, rtol=0, atol=1e-15)


def test_identity_pair():
    check_identity_pair()


# ------------------------------------------- ReLU switches off negative pre-activations

def check_dead_hidden_layer():
    g = _rng(2)
    x = g.standard_normal((4, 8))
    W1 = g.standard_normal((16, 8))
    W2 = g.standard_normal((8, 16))
    b2 = g.standard_normal(8)
    f = F.ffn_ref(x, W1, np.full(16, -1e6), W2, b2)   # every pre-activation < 0
    assert np.array_equal(f, np.broadcast_to(b2, f.shape))
    # all pre-activations positive: ReLU is the identity and FFN is affine
    f2 = F.ffn_ref(x, W1, np.full(16, 1e6), W2, None)
    assert np.allclose(f2, (x @ W1.T + 1e6) @ W2.T, rtol=1e-12, atol=0)


def test_dead_hidden_layer():
    check_dead_hidden_layer()


# ------------------------------------------- position-wise: rows never mix ([JY] FFN)

def check_position_wise():
    g = _rng(3)
    x = g.standard_normal((2, 7, 8))
    W1, b1 = g.standard_normal((12, 8)), g.standard_normal(12)
    W2, b2 = g.standard_normal((8, 12)), g.standard_normal(8)
    y = F.ffn_layer_ref(x, W1, b1, W2, b2)
    # one row alone gives the same output as inside the batch
    for b, i in [(0, 0), (1, 6), (0, 3)]:
        yi = F.ffn_layer_ref(x[b, i][None], W1, b1, W2, b2)[0]
        assert np.allclose(yi, y[b, i], rtol=0, atol=1e-13)
    # changing other positions leaves a position's output bitwise unchanged
    x2 = x.copy()
    x2[:, 1:] = g.standard_normal(x2[:, 1:].shape)
    y2 = F.ffn_layer_ref(x2, W1, b1, W2, b2)
    assert np.array_equal(y2[:, 0], y[:, 0])
    # permuting positions permutes outputs
    perm = g.permutation(7)
    assert np.allclose(F.ffn_layer_ref(x[:, perm], W1, b1, W2, b2), y[:, perm], rtol=0,
                       atol=1e-13)


def test_position_wise():
    check_position_wise()


# ------------------------------------------- brute force on tiny shapes (scalar loops)

def _ffn_loops(x, W1, b1, W2, b2):
    M, D = x.shape
    d_ff = W1.shape[0]
    out = np.zeros((M, D))
    for m in range(M):
        hid = []
        for j in range(d_ff):
            z = float(b1[j])
            for k in range(D):
                z += float(x[m, k]) * float(W1[j, k])
            hid.append(z if z > 0 else 0.0)
        for i in range(D):
            z = float(b2[i])
            for j in range(d_ff):
                z += hid[j] * float(W2[i, j])
            out[m, i] = z
    return out


def check_bruteforce_tiny():
    g = _rng(4)
    for M, D, d_ff in [(1, 1, 1), (3, 2, 5), (4, 3, 7)]:
        x = g.standard_normal((M, D))
        W1, b1 = g.standard_normal((d_ff, D)), g.standard_normal(d_ff)
        W2, b2 = g.standard_normal((D, d_ff)), g.standard_normal(D)
        assert np.allclose(F.ffn_ref(x, W1, b1, W2, b2), _ffn_loops(x, W1, b1, W2, b2),
                           rtol=1e-12, atol=1e-12)


def test_bruteforce_tiny():
    check_bruteforce_tiny()


# ------------------------------------------- the pages' sizes

def test_model_sizes_from_pages():
    shapes = json.load(open(os.path.join(GOLDEN, "model_shapes.json"), encoding="utf-8"))
    for key in ("base", "big"):
        D, d_ff = shapes[key]["d_model"], shapes[key]["d_ff"]
        assert d_ff == 4 * D
        x = np.zeros((3, D))
        f = F.ffn_ref(x, np.zeros((d_ff, D)), None, np.zeros((D, d_ff)), None)
        assert f.shape == (3, D)
    # base: the 512 -> 2048 -> 512 map holds 2 * 512 * 2048 weights and 2048 + 512 biases
    b = shapes["base"]
    assert 2 * b["d_model"] * b["d_ff"] + b["d_ff"] + b["d_model"] == 2_099_712


# ------------------------------------------- sublayer and layer composition

def check_zero_ffn_is_layernorm_fixed_point():
    # W2 = 0, b2 = 0: y = LayerNorm(x); on an input that is already normalised (gamma 1,
    # beta 0) LayerNorm changes nothing beyond the eps term.
    g = _rng(5)
    x = g.standard_normal((6, 32)) * 3 + 1
    W1 = g.standard_normal((64, 32))
    y = F.ffn_layer_ref(x, W1, None, np.zeros((32, 64)), None)
    # the residual carries x through: y is LayerNorm(x), zero mean and unit variance per row
    assert np.allclose(y.mean(axis=-1), 0.0, atol=1e-12)
    assert np.allclose(y.var(axis=-1), 1.0, atol=1e-4)
    yy = F.ffn_layer_ref(y, W1, None, np.zeros((32, 64)), None)
    assert np.allclose(yy, y, rtol=0, atol=1e-4)


def test_zero_ffn_is_layernorm_fixed_point():
    check_zero_ffn_is_layernorm_fixed_point()


def check_encoder_layer_order():
    # attention first, then the feed-forward sublayer ([LT] 3.1; [JY] Encoder-Decoder):
    # with the feed-forward weights zero the layer output is the attention sublayer's output
    # (already normalised), and with W_o = 0, b_o = 0 the attention sublayer is LayerNorm(x).
    g = _rng(6)
    B, N, H, dk = 2, 5, 2, 4
    D, d_ff = H * dk, 16
    x = g.standard_normal((B, N, D))
    Wqkv = g.standard_normal((3 * D, D)) * 0.3
    Wo = g.standard_normal((D, D)) * 0.3
    W1, W2 = g.standard_normal((d_ff, D)), g.standard_normal((D, d_ff))
    y, parts = F.encoder_layer_ref(x, Wqkv, None, Wo, None, None, None, W1, None,
                                   np.zeros((D, d_ff)), None, None, None, H,
                                   return_parts=True)
    assert np.allclose(y, parts["h"], rtol=0, atol=1e-4)
    assert not np.allclose(parts["h"], mha_ref.layernorm_ref(x), atol=1e-3)
    y0 = F.encoder_layer_ref(x, Wqkv, None, np.zeros((D, D)), None, None, None, W1, None, W2,
                             None, None, None, H)
    h0 = mha_ref.layernorm_ref(x)
    f0 = np.maximum(h0 @ W1.T, 0) @ W2.T
    r = h0 + f0
    expect = (r - r.mean(-1, keepdims=True)) / np.sqrt(r.var(-1, keepdims=True) + 1e-5)
    assert np.allclose(y0, expect, rtol=0, atol=1e-12)


def test_encoder_layer_order():
    check_encoder_layer_order()


# ------------------------------------------- planted mistakes: each must trip some pin

def test_plant_missing_relu_is_caught(monkeypatch):
    monkeypatch.setattr(F, "relu_ref", lambda z: np.asarray(z, np.float64))
    with pytest.raises(AssertionError):
        check_identity_pair()
    with pytest.raises(AssertionError):
        check_dead_hidden_layer()


def test_plant_relu_after_second_map_is_caught(monkeypatch):
    def wrong(x, W1, b1, W2, b2):
        return F.relu_ref(mha_ref.linear_ref(mha_ref.linear_ref(x, W1, b1), W2, b2))

    monkeypatch.setattr(F, "ffn_ref", wrong)
    with pytest.raises(AssertionError):
        check_identity_pair()


def test_plant_dropped_second_bias_is_caught(monkeypatch):
    orig = F.ffn_ref
    monkeypatch.setattr(F, "ffn_ref", lambda x, W1, b1, W2, b2: orig(x, W1, b1, W2, None))
    with pytest.raises(AssertionError):
        check_dead_hidden_layer()
    with pytest.raises(AssertionError):
        check_bruteforce_tiny()


def test_plant_transposed_first_map_is_caught(monkeypatch):
    orig = F.ffn_ref

    def wrong(x, W1, b1, W2, b2):
        if W1.shape[0] == W1.shape[1]:
            W1 = W1.T
        return orig(x, W1, b1, W2, b2)

    monkeypatch.setattr(F, "ffn_ref", wrong)
    g = _rng(7)
    x, W1 = g.standard_normal((3, 4)), g.standard_normal((4, 4))
    W2 = g.standard_normal((4, 4))
    with pytest.raises(AssertionError):
        assert np.allclose(F.ffn_ref(x, W1, None, W2, None), _ffn_loops(
            x, W1, np.zeros(4), W2, np.zeros(4)), rtol=1e-12, atol=1e-12)


def test_plant_missing_residual_is_caught(monkeypatch):
    def wrong(x, W1, b1, W2, b2, gamma=None, beta=None, eps=1e-5, return_parts=False):
        return mha_ref.layernorm_ref(F.ffn_ref(x, W1, b1, W2, b2), gamma, beta, eps)

    monkeypatch.setattr(F, "ffn_layer_ref", wrong)
    with pytest.raises(AssertionError):
        check_zero_ffn_is_layernorm_fixed_point()
