"""Feed-forward sublayer and encoder layer: CUDA path vs the CPU oracle on the same seeded
inputs, through the C ABI.

The feed-forward network is position-wise, so the big workload (B=8, n=4096, d_model=1024,
d_ff=4096) is checked on sampled rows that the oracle evaluates on their own.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity_util import BF16_TWO_SUBLAYER_MAX_ABS, assert_bf16_close, assert_f32_close

pytestmark = pytest.mark.gpu

mha = pytest.importorskip("transformer_head_scaled_04_gb300")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from transformer_head_scaled_04_gb300 import build

    build.build()
    mha.load_library()
    torch.cuda.set_device(0)
    mha.device_status()
    yield
    assert mha.device_status() == 0, "a kernel recorded a device-side error"


def dev(a, dtype):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype)


def host(t):
    return t.float().cpu().numpy()


TORCH = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_linear_relu(dt):
    g = np.random.Generator(np.random.PCG64(61))
    M, N, K = 333, 512, 256
    fin = si.round_bf16 if dt == "bf16" else (lambda a: np.asarray(a, np.float32))
    x = fin(g.standard_normal((M, K)))
    W = fin(0.1 * g.standard_normal((N, K)))
    b = fin(0.2 * g.standard_normal(N))
    y = host(mha.linear(dev(x, TORCH[dt]), dev(W, TORCH[dt]), dev(b, TORCH[dt]), relu=True))
    ref = oracle.relu_ref(oracle.linear_ref(x, W, b))
    assert np.all(y >= 0.0)
    check = assert_bf16_close if dt == "bf16" else assert_f32_close
    check(y, ref, f"linear relu {dt}")


def _run_ffn(inp, dtype):
    t = {k: dev(v, dtype) for k, v in inp.items()}
    return host(mha.ffn(t["x"], t["W1"], t["b1"], t["W2"], t["b2"], t["gamma"], t["beta"]))


def test_ffn_f32_workload():
    w = si.WORKLOADS["ffn_f32_b2_n50"]
    for affine in (False, True):
        inp = si.draw_ffn(w, affine=affine)
        y = _run_ffn(inp, torch.float32)
        ref = oracle.ffn_layer_ref(inp["x"], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                                   inp["gamma"], inp["beta"])
        assert_f32_close(y, ref, f"ffn f32 affine={affine}")


@pytest.mark.parametrize("affine", [False, True])
def test_ffn_bf16_base_workload(affine):
    w = si.WORKLOADS["ffn_base_b32_n128"]
    inp = si.draw_ffn(w, affine=affine)
    y = _run_ffn(inp, torch.bfloat16)
    ref = oracle.ffn_layer_ref(inp["x"], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                               inp["gamma"], inp["beta"])
    assert_bf16_close(y, ref, f"ffn bf16 base affine={affine}")


def test_ffn_bf16_ragged_rows():
    # 3 x 111 = 333 positions: the last 128-row tile of both GEMMs is partial
    w = si.WORKLOADS["ffn_base_b32_n128"]
    inp = si.draw_ffn(w, affine=True)
    inp["x"] = inp["x"][:3, :111]
    y = _run_ffn(inp, torch.bfloat16)
    ref = oracle.ffn_layer_ref(inp["x"], inp["W1"], inp["b1"], inp["W2"], inp["b2"],
                               inp["gamma"], inp["beta"])
    assert_bf16_close(y, ref, "ffn bf16 ragged")


def test_ffn_bf16_big_workload_sampled_rows():
    w = si.WORKLOADS["ffn_big_b8_n4096"]
    inp = si.draw_ffn(w)
    y = _run_ffn(inp, torch.bfloat16)
    g = np.random.Generator(np.random.PCG64(71))
    for b in (0, w.B - 1):
        rows = np.unique(np.concatenate([[0, w.Nq - 1], g.integers(0, w.Nq, 62)]))
        ref = oracle.ffn_layer_ref(inp["x"][b, rows], inp["W1"], inp["b1"], inp["W2"],
                                   inp["b2"], inp["gamma"], inp["beta"])
        assert_bf16_close(y[b, rows], ref, f"ffn bf16 big b={b}")


@pytest.mark.parametrize("name", ["encoder_base_b32_n128", "encoder_base_pad_b32_n128"])
def test_encoder_layer_bf16(name):
    w = si.WORKLOADS[name]
    inp = si.draw_encoder(w, affine=True)
    t = {k: dev(v, torch.bfloat16) for k, v in inp.items() if k != "key_len"}
    key_len = None if inp["key_len"] is None else torch.from_numpy(inp["key_len"]).cuda()
    y = host(mha.encoder_layer(t["x_q"], t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"],
                               t["gamma"], t["beta"], t["W1"], t["b1"], t["W2"], t["b2"],
                               t["gamma2"], t["beta2"], w.H, w.mask, key_len))
    ref = oracle.encoder_layer_ref(inp["x_q"], inp["W_qkv"], inp["b_qkv"], inp["W_o"],
                                   inp["b_o"], inp["gamma"], inp["beta"], inp["W1"], inp["b1"],
                                   inp["W2"], inp["b2"], inp["gamma2"], inp["beta2"], w.H,
                                   w.mask, inp["key_len"])
    # two bf16-rounded sublayer outputs in a row: the derived two-sublayer bound
    assert_bf16_close(y, ref, f"encoder layer {name}", max_abs_bound=BF16_TWO_SUBLAYER_MAX_ABS)
    # the second sublayer alone, from the first sublayer's own bf16 output: one-sublayer bound
    h = host(mha.mha_layer(t["x_q"], None, t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"],
                           t["gamma"], t["beta"], w.H, w.mask, key_len))
    ref2 = oracle.ffn_layer_ref(h, inp["W1"], inp["b1"], inp["W2"], inp["b2"], inp["gamma2"],
                                inp["beta2"])
    assert_bf16_close(y, ref2, f"encoder layer {name}, feed-forward sublayer on the GPU's h")
