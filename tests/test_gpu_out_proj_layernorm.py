"""The sublayer's last two steps in one call, y = LayerNorm(x + C W_o^T + b_o) * gamma + beta
(mha_out_proj_layernorm_fwd), against the oracle's W^O projection followed by its residual
LayerNorm.  bf16 widths that are multiples of 256 run the fused kernel (one cluster of
d_model / 256 CTAs per 128-row tile exchanging row statistics); the other widths and fp32 run
the projection and the LayerNorm as two launches."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity_util import assert_bf16_close, assert_f32_close

import transformer_head_scaled_04_gb300 as mha


def _draw(M, D, K, dtype, affine, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    fin = si.round_bf16 if dtype == "bf16" else (lambda a: np.asarray(a, np.float32))
    c = fin(g.standard_normal((M, K)))
    bound = float(np.sqrt(6.0 / (K + D)))
    W = fin(g.uniform(-bound, bound, (D, K)))
    x = fin(g.standard_normal((M, D)))
    if affine:
        b = fin(0.1 * g.standard_normal(D))
        gamma = fin(1.0 + 0.1 * g.standard_normal(D))
        beta = fin(0.1 * g.standard_normal(D))
    else:
        b = gamma = beta = None
    return c, W, b, x, gamma, beta


def _run(c, W, b, x, gamma, beta, dtype):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dev = torch.device("cuda", 0)
    t = [None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev, tdt)
         for a in (c, W, b, x, gamma, beta)]
    y = mha.out_proj_layernorm(t[0], t[1], t[2], t[3], t[4], t[5], eps=1e-5)
    torch.cuda.synchronize()
    assert mha.device_status() == 0
    return y.float().cpu().numpy()


def _ref(c, W, b, x, gamma, beta):
    return oracle.layernorm_ref(x + oracle.linear_ref(c, W, b), gamma, beta, eps=1e-5)


@pytest.mark.gpu
@pytest.mark.parametrize("M,D,K,affine", [
    (300, 256, 256, True),     # clusters of one CTA; a ragged last row tile
    (129, 512, 512, True),     # two-CTA clusters (the base model); one row past a tile
    (1000, 768, 512, False),   # three-CTA clusters, K != D, no bias / gamma / beta
    (333, 1024, 1024, True),   # four-CTA clusters (the big model)
    (5000, 2048, 256, True),   # eight-CTA clusters; more row tiles than resident clusters
    (51200, 512, 512, True),   # several row tiles per cluster: both statistics buffers reused
    (200, 192, 128, True),     # width not a multiple of 256: projection, then LayerNorm
])
def test_out_proj_layernorm_bf16(M, D, K, affine):
    args = _draw(M, D, K, "bf16", affine, seed=M + D + K)
    y = _run(*args, "bf16")
    assert_bf16_close(y, _ref(*args), f"out-proj + LayerNorm bf16 M={M} D={D} K={K}")


@pytest.mark.gpu
def test_out_proj_layernorm_f32():
    args = _draw(77, 96, 40, "f32", True, seed=5)
    y = _run(*args, "f32")
    assert_f32_close(y, _ref(*args), "out-proj + LayerNorm f32")


@pytest.mark.gpu
def test_out_proj_layernorm_matches_the_sublayer_path_bitwise():
    """From 8192 rows on, mha_layer_fwd runs this same kernel on its head-concat buffer:
    the fused call on the sublayer's own concat (recomputed by the attention entry point)
    gives the same bits.  The big model's heads at half its batch."""
    w = dataclasses.replace(si.WORKLOADS["big_long_b8_n4096"], B=4)
    inp = si.draw_layer(w, affine=True)
    dev = torch.device("cuda", 0)
    t = {k: (None if v is None else torch.from_numpy(v).to(dev, torch.bfloat16))
         for k, v in inp.items() if k != "key_len"}
    y_layer = mha.mha_layer(t["x_q"], None, t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"],
                            t["gamma"], t["beta"], w.H, "none", None)
    D = w.D
    x2 = t["x_q"].reshape(-1, D)
    qkv = mha.linear(x2, t["W_qkv"], t["b_qkv"]).reshape(w.B, w.Nq, 3, w.H, 64)
    q, k, v = (qkv[:, :, i].permute(0, 2, 1, 3) for i in range(3))
    o = mha.sdpa(q, k, v, "none")
    concat = o.permute(0, 2, 1, 3).reshape(-1, D).contiguous()
    y_fused = mha.out_proj_layernorm(concat, t["W_o"], t["b_o"], x2, t["gamma"], t["beta"])
    torch.cuda.synchronize()
    assert torch.equal(y_fused.reshape(y_layer.shape), y_layer)
