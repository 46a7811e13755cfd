"""The index-checking build (libmha_debug.so, compiled with MHA_DEBUG_BOUNDS): every plain
global load and store of the forward kernels (bf16 and fp32 attention, the projection GEMM's
epilogue, the W^O projection fused with the residual LayerNorm, the residual LayerNorm)
checks its index against the extent the kernel's size arguments give the buffer and records
MHA_ERR_DEVICE_BOUNDS instead of making the access.  Small parity cases of every mask and
shape family run through its C ABI: each result must match the oracle and the device status
word must stay clear."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity_util import assert_bf16_close, assert_f32_close

from transformer_head_scaled_04_gb300 import _capi as C
from transformer_head_scaled_04_gb300 import build as B

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg():
    B.build(debug_bounds=True)
    return C.load_debug()


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(a, dtype):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _status(lib):
    return lib.mha_debug_last_device_status(_stream())


@pytest.mark.parametrize("B_,H,Nq,Nk,mask,kl", [
    (2, 3, 300, 333, "none", None),
    (2, 2, 300, 300, "causal", None),
    (3, 2, 200, 390, "key_padding", [0, 1, 390]),
    (3, 5, 128, 256, "key_padding", [256, 0, 100]),
    (1, 1, 1, 1, "none", None),
])
def test_debug_build_attention_bf16(dbg, B_, H, Nq, Nk, mask, kl):
    Q, K, V, _ = si.draw_sdpa(B_, H, Nq, Nk, dtype="bf16", seed=900 + Nq + Nk)
    key_len = None if kl is None else np.array(kl, np.int32)
    tq, tk, tv = (_dev(a, torch.bfloat16) for a in (Q, K, V))
    tl = _dev(key_len, torch.int32)
    O = torch.empty_like(tq)
    lse = torch.empty((B_, H, Nq), dtype=torch.float32, device="cuda")
    assert dbg.mha_sdpa_fwd_lse(B_, H, Nq, Nk, 64, 64, C.MHA_BF16, C.MASKS[mask], _vp(tl), 0.0,
                                _vp(tq), _vp(tk), _vp(tv), _vp(O), None, _vp(lse),
                                _stream()) == 0
    assert _status(dbg) == 0
    assert_bf16_close(O.float().cpu().numpy(), oracle.sdpa_ref(Q, K, V, mask, key_len),
                      f"debug build sdpa bf16 {mask}")


def test_debug_build_restricted_and_short_queries(dbg):
    Q, K, V, _ = si.draw_sdpa(1, 2, 640, 640, dtype="bf16", seed=901)
    tq, tk, tv = (_dev(a, torch.bfloat16) for a in (Q, K, V))
    O = torch.empty_like(tq)
    assert dbg.mha_sdpa_window_fwd(1, 2, 640, 64, 64, C.MHA_BF16, 63, 0.0, _vp(tq), _vp(tk),
                                   _vp(tv), _vp(O), None, _stream()) == 0
    assert _status(dbg) == 0
    assert_bf16_close(O.float().cpu().numpy(), oracle.sdpa_ref(Q, K, V, "window", window=63),
                      "debug build window")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hs = sms + 5
    Q, K, V, _ = si.draw_sdpa(2, Hs, 90, 90, dtype="bf16", seed=902)
    tq, tk, tv = (_dev(a, torch.bfloat16) for a in (Q, K, V))
    O = torch.empty_like(tq)
    assert dbg.mha_sdpa_fwd(2, Hs, 90, 90, 64, 64, C.MHA_BF16, 0, None, 0.0, _vp(tq), _vp(tk),
                            _vp(tv), _vp(O), None, _stream()) == 0
    assert _status(dbg) == 0
    assert_bf16_close(O.float().cpu().numpy(), oracle.sdpa_ref(Q, K, V, "none"),
                      "debug build short queries")


@pytest.mark.parametrize("mask,kl", [("none", None), ("key_padding", [0, 32]),
                                     ("causal", None)])
def test_debug_build_attention_f32(dbg, mask, kl):
    Q, K, V, _ = si.draw_sdpa(2, 8, 32, 32, dtype="f32", seed=903)
    key_len = None if kl is None else np.array(kl, np.int32)
    tq, tk, tv = (_dev(a, torch.float32) for a in (Q, K, V))
    tl = _dev(key_len, torch.int32)
    O = torch.empty_like(tq)
    lse = torch.empty((2, 8, 32), dtype=torch.float32, device="cuda")
    assert dbg.mha_sdpa_fwd_lse(2, 8, 32, 32, 64, 64, C.MHA_F32, C.MASKS[mask], _vp(tl), 0.0,
                                _vp(tq), _vp(tk), _vp(tv), _vp(O), None, _vp(lse),
                                _stream()) == 0
    assert _status(dbg) == 0
    assert_f32_close(O.cpu().numpy(), oracle.sdpa_ref(Q, K, V, mask, key_len),
                     f"debug build sdpa f32 {mask}")


@pytest.mark.parametrize("name", ["enc_self_base_b32_n128", "dec_causal_base_b32_n256",
                                  "cross_pad_base_b32_q128_k256"])
def test_debug_build_base_sublayers(dbg, name):
    import dataclasses

    w = dataclasses.replace(si.WORKLOADS[name], B=4)
    inp = si.draw_layer(w, affine=True)
    t = {k: _dev(v, torch.bfloat16) for k, v in inp.items() if k != "key_len"}
    kl = _dev(inp["key_len"], torch.int32)
    n = ctypes.c_size_t(0)
    assert dbg.mha_layer_workspace_size(w.B, w.H, w.Nq, w.Nk, w.D, 64, 64, C.MHA_BF16,
                                        ctypes.byref(n)) == 0
    ws = torch.empty(n.value, dtype=torch.uint8, device="cuda")
    y = torch.empty_like(t["x_q"])
    assert dbg.mha_layer_fwd(w.B, w.H, w.Nq, w.Nk, w.D, 64, 64, C.MHA_BF16, C.MASKS[w.mask],
                             _vp(kl), 1e-5, _vp(t["x_q"]), _vp(t["x_kv"]), _vp(t["W_qkv"]),
                             _vp(t["b_qkv"]), _vp(t["W_o"]), _vp(t["b_o"]), _vp(t["gamma"]),
                             _vp(t["beta"]), _vp(y), _vp(ws), n.value, _stream()) == 0
    assert _status(dbg) == 0
    ref = oracle.mha_layer_ref(inp["x_q"], inp["x_kv"], inp["W_qkv"], inp["b_qkv"], inp["W_o"],
                               inp["b_o"], inp["gamma"], inp["beta"], w.H, w.mask,
                               inp["key_len"])
    assert_bf16_close(y.float().cpu().numpy(), ref, f"debug build {name}")


@pytest.mark.parametrize("M,D,K", [(300, 512, 512), (129, 256, 128)])
def test_debug_build_out_proj_layernorm(dbg, M, D, K):
    g = np.random.Generator(np.random.PCG64(M + D))
    c = si.round_bf16(g.standard_normal((M, K)))
    W = si.round_bf16(g.uniform(-0.1, 0.1, (D, K)))
    b = si.round_bf16(0.1 * g.standard_normal(D))
    x = si.round_bf16(g.standard_normal((M, D)))
    gam = si.round_bf16(1.0 + 0.1 * g.standard_normal(D))
    bet = si.round_bf16(0.1 * g.standard_normal(D))
    t = [_dev(a, torch.bfloat16) for a in (c, W, b, x, gam, bet)]
    y = torch.empty_like(t[3])
    assert dbg.mha_out_proj_layernorm_fwd(M, D, K, C.MHA_BF16, 1e-5, *[_vp(a) for a in t],
                                          _vp(y), _stream()) == 0
    assert _status(dbg) == 0
    ref = oracle.layernorm_ref(x + oracle.linear_ref(c, W, b), gam, bet, eps=1e-5)
    assert_bf16_close(y.float().cpu().numpy(), ref, f"debug build out-proj LN {M}x{D}")


def test_debug_build_residual_layernorm_f32(dbg):
    g = np.random.Generator(np.random.PCG64(904))
    x = g.standard_normal((77, 96)).astype(np.float32)
    a = g.standard_normal((77, 96)).astype(np.float32)
    tx, ta = _dev(x, torch.float32), _dev(a, torch.float32)
    y = torch.empty_like(tx)
    assert dbg.mha_residual_layernorm_fwd(77, 96, C.MHA_F32, 1e-5, _vp(tx), _vp(ta), None, None,
                                          _vp(y), _stream()) == 0
    assert _status(dbg) == 0
    assert_f32_close(y.cpu().numpy(), oracle.layernorm_ref(x + a, None, None, eps=1e-5),
                     "debug build residual LN f32")
