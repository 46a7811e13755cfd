"""Sublayer backward: every gradient of y = LayerNorm(x_q + MultiHead(x_q, x_kv, x_kv)) from the
CUDA path (``mha_layer_bwd`` through the C ABI) against the CPU oracle's chain rule
(``oracle.mha_layer_bwd_ref``) on the same seeded inputs and the same upstream gradient dy.

Per-token gradients (dx_q, dx_kv) are held to the bf16 gradient bound at each token's own
scale; parameter gradients, sums over all B*N tokens, to a bound that scales with the
tensor's RMS (both derived in ``parity_util``).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity_util import (assert_bf16_param_grad_close, assert_bf16_token_grad_close,
                         assert_f32_close)

pytestmark = pytest.mark.gpu

mha = pytest.importorskip("transformer_head_scaled_04_gb300")

PER_TOKEN = ("dx_q", "dx_kv")
PARAMS = ("dW_qkv", "db_qkv", "dW_o", "db_o", "dgamma", "dbeta")


@pytest.fixture(scope="module", autouse=True)
def _built():
    from transformer_head_scaled_04_gb300 import build

    build.build()
    mha.load_library()
    torch.cuda.set_device(0)
    mha.device_status()
    yield
    assert mha.device_status() == 0, "a kernel recorded a device-side error"


def to_dev(a, dtype):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype)


def host(t):
    return None if t is None else t.float().cpu().numpy()


def draw_dy(w, seed, dtype):
    g = np.random.Generator(np.random.PCG64(seed))
    dy = g.standard_normal((w.B, w.Nq, w.D))
    return si.round_bf16(dy) if dtype == "bf16" else dy.astype(np.float32)


def run_gpu(inp, dy, w, dtype):
    t = {k: to_dev(v, dtype) for k, v in inp.items() if k != "key_len"}
    kl = to_dev(inp["key_len"], torch.int32)
    g = mha.mha_layer_backward(t["x_q"], t["x_kv"], t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"],
                               t["gamma"], t["beta"], w.H, to_dev(dy, dtype), w.mask, kl,
                               d_k=w.d_k, d_v=w.d_v)
    return {k: host(v) for k, v in g.items()}


def run_oracle(inp, dy, w):
    return oracle.mha_layer_bwd_ref(inp["x_q"], inp["x_kv"], inp["W_qkv"], inp["b_qkv"],
                                    inp["W_o"], inp["b_o"], inp["gamma"], inp["beta"], w.H, dy,
                                    w.mask, inp["key_len"], d_k=w.d_k, d_v=w.d_v)


def compare_bf16(got, ref, what):
    for k in PER_TOKEN:
        if ref[k] is None:
            assert got[k] is None
            continue
        assert_bf16_token_grad_close(got[k], ref[k], f"{what} {k}")
    for k in PARAMS:
        assert_bf16_param_grad_close(got[k], ref[k], f"{what} {k}")


@pytest.mark.parametrize("name", ["enc_self_base_b32_n128", "dec_causal_base_b32_n256",
                                  "cross_pad_base_b32_q128_k256"])
def test_layer_backward_base_workloads(name):
    w = si.WORKLOADS[name]
    inp = si.draw_layer(w, affine=True)
    dy = draw_dy(w, w.seed + 100, "bf16")
    compare_bf16(run_gpu(inp, dy, w, torch.bfloat16), run_oracle(inp, dy, w), name)


@pytest.mark.parametrize("mask,cross,Nq,Nk", [
    ("none", False, 70, 70),
    ("causal", False, 300, 300),
    ("key_padding", True, 130, 200),
    ("none", True, 64, 257),
    ("key_padding", False, 1, 1),
    # enough tokens (3 x 700, 3 x 1500) for the split-K weight gradients, with a ragged last
    # K slice (2100 and 4500 are not multiples of 64)
    ("none", False, 700, 700),
    ("key_padding", True, 130, 1500),
])
def test_layer_backward_bf16_ragged(mask, cross, Nq, Nk):
    w = si.Workload("t", "layer", "bf16", B=3, H=4, Nq=Nq, Nk=Nk, mask=mask, cross=cross,
                    seed=79)
    inp = si.draw_layer(w, affine=True)
    if mask == "key_padding":
        inp["key_len"] = np.array([0, min(5, Nk), Nk], np.int32)
    dy = draw_dy(w, 80, "bf16")
    got = run_gpu(inp, dy, w, torch.bfloat16)
    ref = run_oracle(inp, dy, w)
    compare_bf16(got, ref, f"layer bwd bf16 {mask} cross={cross} {Nq}x{Nk}")
    if mask == "key_padding":
        # batch 0 sees no key: its attention output is 0 and nothing flows back into x_kv
        src = "dx_kv" if cross else None
        if src is not None:
            assert np.all(got[src][0] == 0.0)


@pytest.mark.parametrize("mask,cross,H,dk", [("none", False, 2, 64), ("causal", False, 3, 32),
                                             ("key_padding", True, 4, 16)])
def test_layer_backward_f32(mask, cross, H, dk):
    w = si.Workload("t", "layer", "f32", B=2, H=H, Nq=40, Nk=40 if not cross else 75, d_k=dk,
                    d_v=dk, mask=mask, cross=cross, seed=81)
    inp = si.draw_layer(w, affine=True)
    if mask == "key_padding":
        inp["key_len"] = np.array([1, 75], np.int32)
    dy = draw_dy(w, 82, "f32")
    got = run_gpu(inp, dy, w, torch.float32)
    ref = run_oracle(inp, dy, w)
    for k in PER_TOKEN + PARAMS:
        if ref[k] is None:
            assert got[k] is None
        else:
            assert_f32_close(got[k], ref[k], f"layer bwd f32 {mask} {k}")


def test_layer_backward_is_deterministic():
    w = si.WORKLOADS["dec_causal_base_b32_n256"]
    inp = si.draw_layer(w, affine=True)
    dy = draw_dy(w, 83, "bf16")
    before = mha.get_deterministic()
    mha.set_deterministic(True)
    try:
        a = run_gpu(inp, dy, w, torch.bfloat16)
        b = run_gpu(inp, dy, w, torch.bfloat16)
    finally:
        mha.set_deterministic(before)
    for k in PER_TOKEN + PARAMS:
        if a[k] is not None:
            assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_layer_backward_big_long_sampled_batches(mask):
    """B=8, n=4096, d_model=1024, 16 heads, in the bench's launch configuration.  dy is zero
    outside the first and the last batch element, so those two carry every parameter
    gradient: the oracle evaluates just them (one at a time), and every other batch element's
    input gradient must be exactly zero."""
    w = si.WORKLOADS["big_long_b8_n4096"].with_mask(mask)
    inp = si.draw_layer(w, affine=True)
    dy = draw_dy(w, 84, "bf16")
    keep = [0, w.B - 1]
    dy[[b for b in range(w.B) if b not in keep]] = 0.0
    got = run_gpu(inp, dy, w, torch.bfloat16)
    for b in range(w.B):
        if b not in keep:
            assert np.all(got["dx_q"][b] == 0.0), b
    total = None
    for b in keep:
        one = dict(inp, x_q=inp["x_q"][b:b + 1])
        wb = si.Workload("one", "layer", "bf16", B=1, H=w.H, Nq=w.Nq, Nk=w.Nk, mask=mask)
        ref = run_oracle(one, dy[b:b + 1], wb)
        assert_bf16_token_grad_close(got["dx_q"][b:b + 1], ref["dx_q"], f"big {mask} dx_q b={b}")
        total = ref if total is None else {k: total[k] + ref[k] for k in PARAMS}
    for k in PARAMS:
        assert_bf16_param_grad_close(got[k], total[k], f"big {mask} {k}")


@pytest.mark.parametrize("name", ["enc_self_base_b32_n128", "cross_pad_base_b32_q128_k256"])
def test_layer_training_split_matches(name):
    """mha_layer_fwd_train writes the forward's y bitwise, and mha_layer_bwd_saved from the
    activations it left gives the gradients of mha_layer_bwd bitwise (deterministic mode);
    in the default mode the saved backward still meets the oracle's bound."""
    w = si.WORKLOADS[name]
    inp = si.draw_layer(w, affine=True)
    dy = draw_dy(w, 86, "bf16")
    bf = torch.bfloat16
    t = {k: to_dev(v, bf) for k, v in inp.items() if k != "key_len"}
    kl = to_dev(inp["key_len"], torch.int32)
    args = (t["x_q"], t["x_kv"], t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"], t["gamma"],
            t["beta"], w.H)
    kw = dict(mask=w.mask, key_len=kl, d_k=w.d_k, d_v=w.d_v)
    tdy = to_dev(dy, bf)
    y_ref = mha.mha_layer(*args, **kw)
    before = mha.get_deterministic()
    mha.set_deterministic(True)
    try:
        y, ws = mha.mha_layer_forward_train(*args, **kw)
        assert torch.equal(y, y_ref)
        full = mha.mha_layer_backward(*args, tdy, **kw)
        saved = mha.mha_layer_backward(*args, tdy, workspace=ws, saved=True, **kw)
        for k in PER_TOKEN + PARAMS:
            if full[k] is None:
                assert saved[k] is None
            else:
                assert torch.equal(full[k], saved[k]), k
        mha.set_deterministic(False)
        y2, ws2 = mha.mha_layer_forward_train(*args, **kw)
        assert torch.equal(y2, y_ref)
        fast = mha.mha_layer_backward(*args, tdy, workspace=ws2, saved=True, **kw)
    finally:
        mha.set_deterministic(before)
    compare_bf16({k: host(v) for k, v in fast.items()}, run_oracle(inp, dy, w),
                 f"training split {name}")


def test_layer_training_split_big_model_rows():
    """The big model's heads at 16384 rows (the fused path starts at 8192), where the training
    forward computes y with the W^O projection and the LayerNorm in one kernel that also keeps
    the projection for the backward: y equals mha_layer_fwd's bitwise, and the backward from
    the saved activations
    equals the recomputing backward bitwise (deterministic mode).  The recomputing backward
    itself is held to the oracle by test_layer_backward_big_long_sampled_batches."""
    w = dataclasses.replace(si.WORKLOADS["big_long_b8_n4096"], B=4)
    inp = si.draw_layer(w, affine=True)
    dy = draw_dy(w, 87, "bf16")
    bf = torch.bfloat16
    t = {k: to_dev(v, bf) for k, v in inp.items() if k != "key_len"}
    args = (t["x_q"], t["x_kv"], t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"], t["gamma"],
            t["beta"], w.H)
    kw = dict(mask="none", key_len=None, d_k=w.d_k, d_v=w.d_v)
    tdy = to_dev(dy, bf)
    y_ref = mha.mha_layer(*args, **kw)
    before = mha.get_deterministic()
    mha.set_deterministic(True)
    try:
        y, ws = mha.mha_layer_forward_train(*args, **kw)
        assert torch.equal(y, y_ref)
        full = mha.mha_layer_backward(*args, tdy, **kw)
        saved = mha.mha_layer_backward(*args, tdy, workspace=ws, saved=True, **kw)
        for k in PER_TOKEN + PARAMS:
            if full[k] is not None:
                assert torch.equal(full[k], saved[k]), k
    finally:
        mha.set_deterministic(before)
    assert mha.device_status() == 0
