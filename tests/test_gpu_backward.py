"""Attention backward (and the forward's log-sum-exp): CUDA path through the C ABI vs the CPU
oracle's chain rule (``oracle.backward``) on the same seeded inputs.

The GPU gradients start from the GPU forward's own O and lse, as a training step would; the
oracle recomputes everything exactly from the same bf16 (or fp32) Q, K, V and dO.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity_util import assert_bf16_grad_close, assert_f32_close

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


@pytest.fixture(params=[False, True], ids=["fused_dq", "deterministic"])
def det_mode(request):
    """Both bf16 dQ paths: the fused accumulation (default) and the separate dQ kernel."""
    before = mha.get_deterministic()
    mha.set_deterministic(request.param)
    yield request.param
    mha.set_deterministic(before)


def dev(a, dtype):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype)


def host(t):
    return t.float().cpu().numpy()


def draw(B, H, Nq, Nk, dtype, seed, d=64):
    g = np.random.Generator(np.random.PCG64(seed))
    fin = si.round_bf16 if dtype == "bf16" else (lambda a: np.asarray(a, np.float32))
    Q = fin(g.standard_normal((B, H, Nq, d)))
    K = fin(g.standard_normal((B, H, Nk, d)))
    V = fin(g.standard_normal((B, H, Nk, d)))
    dO = fin(g.standard_normal((B, H, Nq, d)))
    return Q, K, V, dO


def run(Q, K, V, dO, mask, kl, dtype):
    t = torch.bfloat16 if dtype == "bf16" else torch.float32
    tq, tk, tv, tg = (dev(a, t) for a in (Q, K, V, dO))
    tkl = None if kl is None else dev(np.asarray(kl, np.int32), torch.int32)
    O, lse = mha.sdpa_with_lse(tq, tk, tv, mask, tkl)
    dq, dk, dv = mha.sdpa_backward(tq, tk, tv, O, tg, lse, mask, tkl)
    return host(O), host(lse), host(dq), host(dk), host(dv)


CASES = [  # B, H, Nq, Nk, mask, key_len
    (1, 2, 128, 128, "none", None),
    (2, 2, 300, 300, "causal", None),
    (1, 1, 640, 640, "none", None),
    (2, 3, 333, 333, "causal", None),
    (3, 1, 200, 390, "key_padding", [0, 1, 390]),
    (2, 1, 100, 900, "none", None),
    (1, 2, 1, 1, "none", None),
]


@pytest.mark.parametrize("B,H,Nq,Nk,mask,kl", CASES)
def test_sdpa_backward_bf16(B, H, Nq, Nk, mask, kl, det_mode):
    Q, K, V, dO = draw(B, H, Nq, Nk, "bf16", seed=500 + Nq + Nk)
    O, lse, dq, dk, dv = run(Q, K, V, dO, mask, kl, "bf16")
    key_len = None if kl is None else np.asarray(kl, np.int32)
    rq, rk, rv = oracle.sdpa_bwd_ref(Q, K, V, dO, mask, key_len)
    what = f"sdpa bwd bf16 {B}x{H} {Nq}x{Nk} {mask}"
    assert_bf16_grad_close(dq, rq, what + " dQ")
    assert_bf16_grad_close(dk, rk, what + " dK")
    assert_bf16_grad_close(dv, rv, what + " dV")
    lse_ref = oracle.sdpa_lse_ref(Q, K, mask, key_len)
    finite = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), finite)
    assert np.allclose(lse[finite], lse_ref[finite], rtol=0, atol=2e-3)
    if key_len is not None:
        for b, L in enumerate(kl):
            assert np.all(dk[b, :, L:] == 0.0) and np.all(dv[b, :, L:] == 0.0)
            if L == 0:
                assert np.all(dq[b] == 0.0)


@pytest.mark.parametrize("mask,kl", [("none", None), ("causal", None),
                                     ("key_padding", [40, 77])])
def test_sdpa_backward_f32(mask, kl):
    Q, K, V, dO = draw(2, 2, 77, 77, "f32", seed=541, d=48)
    O, lse, dq, dk, dv = run(Q, K, V, dO, mask, kl, "f32")
    key_len = None if kl is None else np.asarray(kl, np.int32)
    rq, rk, rv = oracle.sdpa_bwd_ref(Q, K, V, dO, mask, key_len)
    assert_f32_close(dq, rq, f"sdpa bwd f32 {mask} dQ")
    assert_f32_close(dk, rk, f"sdpa bwd f32 {mask} dK")
    assert_f32_close(dv, rv, f"sdpa bwd f32 {mask} dV")
    lse_ref = oracle.sdpa_lse_ref(Q, K, mask, key_len)
    assert np.allclose(lse, lse_ref, rtol=1e-6, atol=1e-5)


def test_sdpa_backward_bf16_strided_projection_layout():
    # Q|K|V and their gradients inside packed [B, N, 3, H, 64] buffers, O/dO as [B, N, H*64]
    B, H, N = 2, 4, 260
    g = np.random.Generator(np.random.PCG64(551))
    buf = si.round_bf16(g.standard_normal((B, N, 3, H, 64)))
    dObuf = si.round_bf16(g.standard_normal((B, N, H * 64)))
    tb = dev(buf, torch.bfloat16)
    q, k, v = (tb[:, :, i].permute(0, 2, 1, 3) for i in range(3))
    tg = dev(dObuf, torch.bfloat16).view(B, N, H, 64).permute(0, 2, 1, 3)
    O, lse = mha.sdpa_with_lse(q, k, v, "causal")
    dq, dk, dv = mha.sdpa_backward(q, k, v, O, tg, lse, "causal")
    Q, K, V = (np.moveaxis(buf[:, :, i], 1, 2) for i in range(3))
    dO = np.moveaxis(dObuf.reshape(B, N, H, 64), 1, 2)
    rq, rk, rv = oracle.sdpa_bwd_ref(Q, K, V, dO, "causal")
    assert_bf16_grad_close(host(dq), rq, "strided dQ")
    assert_bf16_grad_close(host(dk), rk, "strided dK")
    assert_bf16_grad_close(host(dv), rv, "strided dV")


def test_sdpa_backward_bf16_big_heads():
    # the big model's heads at n = 4096: two (b, h) pairs compared in full
    w = si.WORKLOADS["big_long_b8_n4096"]
    Q, K, V, _ = si.draw_sdpa(w.B, w.H, w.Nq, w.Nk, dtype="bf16", seed=w.seed)
    g = np.random.Generator(np.random.PCG64(561))
    dO = si.round_bf16(g.standard_normal(Q.shape))
    O, lse, dq, dk, dv = run(Q, K, V, dO, "none", None, "bf16")
    for b, h in [(0, 0), (w.B - 1, w.H - 1)]:
        sl = (slice(b, b + 1), slice(h, h + 1))
        rq, rk, rv = oracle.sdpa_bwd_ref(Q[sl], K[sl], V[sl], dO[sl], "none")
        assert_bf16_grad_close(dq[sl], rq, f"big dQ b={b} h={h}")
        assert_bf16_grad_close(dk[sl], rk, f"big dK b={b} h={h}")
        assert_bf16_grad_close(dv[sl], rv, f"big dV b={b} h={h}")


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_sdpa_backward_bf16_modes(mask):
    """The deterministic path repeats bitwise; the fused one repeats dK and dV bitwise (each
    key tile's own accumulators) and dQ up to the order of its fp32 additions; the two paths'
    gradients agree to bf16 rounding."""
    Q, K, V, dO = draw(2, 4, 1000, 1000, "bf16", seed=571)
    before = mha.get_deterministic()
    try:
        mha.set_deterministic(True)
        assert mha.get_deterministic()
        a = run(Q, K, V, dO, mask, None, "bf16")
        b = run(Q, K, V, dO, mask, None, "bf16")
        for x, y in zip(a, b):
            assert np.array_equal(x, y)
        mha.set_deterministic(False)
        assert not mha.get_deterministic()
        c = run(Q, K, V, dO, mask, None, "bf16")
        e = run(Q, K, V, dO, mask, None, "bf16")
    finally:
        mha.set_deterministic(before)
    for i in (3, 4):  # dK, dV
        assert np.array_equal(c[i], e[i])
    for i in (2, 3, 4):
        scale = np.abs(a[i]).max()
        assert np.abs(c[i] - a[i]).max() <= 2 ** -7 * scale
    assert np.abs(c[2] - e[2]).max() <= 2 ** -7 * np.abs(a[2]).max()
