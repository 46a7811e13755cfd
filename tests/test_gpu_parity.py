"""CUDA path vs the CPU oracle, element by element, on the same seeded inputs.

Every call goes through the C ABI (libmha.so via the thin torch binding).  Sizes span
several 128-row tiles with ragged tails; the five workloads of the sublayer are covered,
the largest (B=8, n=4096, d_model=1024) on sampled rows the oracle evaluates one by one.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity_util import assert_bf16_close, assert_f32_close

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


def to_dev(a, dtype):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype)


def host(t):
    return t.float().cpu().numpy()


# ------------------------------------------------------------------------ attention, fp32

def test_sdpa_f32_small_workload():
    w = si.WORKLOADS["sdpa_f32_b1_h8_n32"]
    Q, K, V, _ = si.draw_qkv(w)
    O = mha.sdpa(to_dev(Q, torch.float32), to_dev(K, torch.float32), to_dev(V, torch.float32))
    assert_f32_close(host(O), oracle.sdpa_ref(Q, K, V), "sdpa f32 B1 H8 N32")


@pytest.mark.parametrize("mask,Nq,Nk,dk,dv", [
    ("causal", 77, 77, 64, 64),
    ("key_padding", 40, 97, 32, 48),
    ("none", 5, 300, 128, 16),
])
def test_sdpa_f32_masks(mask, Nq, Nk, dk, dv):
    Q, K, V, _ = si.draw_sdpa(3, 2, Nq, Nk, dk, dv, "f32", seed=11)
    key_len = np.array([0, 1, Nk], np.int32) if mask == "key_padding" else None
    O = mha.sdpa(to_dev(Q, torch.float32), to_dev(K, torch.float32), to_dev(V, torch.float32),
                 mask, to_dev(key_len, torch.int32))
    assert_f32_close(host(O), oracle.sdpa_ref(Q, K, V, mask, key_len), f"sdpa f32 {mask}")


# ------------------------------------------------------------------------ attention, bf16

SDPA_CASES = [
    (1, 1, 1, 1, "none", None),
    (1, 2, 128, 128, "none", None),
    (2, 3, 300, 333, "none", None),
    (1, 1, 512, 1000, "none", None),
    (2, 2, 300, 300, "causal", None),
    (2, 1, 257, 257, "causal", None),
    (1, 2, 640, 640, "causal", None),
    (3, 5, 1000, 1000, "causal", None),   # heaviest query tiles of all 15 heads launch first
    (3, 2, 200, 390, "key_padding", [0, 1, 390]),
    (4, 1, 129, 256, "key_padding", [64, 127, 128, 129]),
    # more key tiles than K/V ring slots while a block's second query tile is empty
    (1, 2, 640, 1000, "none", None),
    (2, 1, 100, 900, "key_padding", [900, 700]),
]


@pytest.mark.parametrize("B,H,Nq,Nk,mask,kl", SDPA_CASES)
def test_sdpa_bf16(B, H, Nq, Nk, mask, kl):
    Q, K, V, _ = si.draw_sdpa(B, H, Nq, Nk, dtype="bf16", seed=100 + Nq + Nk)
    key_len = np.array(kl, np.int32) if kl is not None else None
    O = mha.sdpa(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16), to_dev(V, torch.bfloat16),
                 mask, to_dev(key_len, torch.int32))
    ref = oracle.sdpa_ref(Q, K, V, mask, key_len)
    assert_bf16_close(host(O), ref, f"sdpa bf16 {B}x{H} {Nq}x{Nk} {mask}")
    if key_len is not None:
        for b, L in enumerate(kl):
            if L == 0:
                assert np.all(host(O)[b] == 0.0)


# Query sequences of at most 128 rows (a single query tile per head; the base model's encoder
# and cross-attention shapes), over odd numbers of heads, with every mask; with key padding
# some batch elements see no key at all next to ones that see many, and the log-sum-exp is
# checked too (+inf exactly where a row sees no key).
SHORT_Q_CASES = [
    (3, 5, 128, 128, "none", None),
    (1, 7, 128, 128, "causal", None),
    (5, 3, 128, 256, "key_padding", [0, 256, 1, 129, 0]),
    (2, 3, 77, 300, "none", None),
    (3, 1, 100, 100, "causal", None),
    (4, 1, 1, 5, "key_padding", [5, 0, 3, 1]),
]


@pytest.mark.parametrize("B,H,Nq,Nk,mask,kl", SHORT_Q_CASES)
def test_sdpa_bf16_short_queries(B, H, Nq, Nk, mask, kl):
    Q, K, V, _ = si.draw_sdpa(B, H, Nq, Nk, dtype="bf16", seed=500 + B * H + Nq + Nk)
    key_len = np.array(kl, np.int32) if kl is not None else None
    O, lse = mha.sdpa_with_lse(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                               to_dev(V, torch.bfloat16), mask, to_dev(key_len, torch.int32))
    ref = oracle.sdpa_ref(Q, K, V, mask, key_len)
    assert_bf16_close(host(O), ref, f"sdpa bf16 short queries {B}x{H} {Nq}x{Nk} {mask}")
    lse_ref = oracle.sdpa_lse_ref(Q, K, mask, key_len)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(host(lse)), fin)
    assert np.allclose(host(lse)[fin], lse_ref[fin], rtol=0, atol=2e-3)
    if key_len is not None:
        for b, L in enumerate(kl):
            if L == 0:
                assert np.all(host(O)[b] == 0.0)


def test_sdpa_bf16_short_queries_more_heads_than_sms():
    """More (b, h) than SMs with a single ragged query tile each (persistent blocks take over
    blocks that have not started)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, H, N = 2, sms + 5, 90
    Q, K, V, _ = si.draw_sdpa(B, H, N, N, dtype="bf16", seed=4343)
    O = mha.sdpa(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16), to_dev(V, torch.bfloat16),
                 "none")
    assert_bf16_close(host(O), oracle.sdpa_ref(Q, K, V, "none"), f"sdpa bf16 short queries {H} heads")


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_sdpa_bf16_more_blocks_than_sms(mask):
    """More 256-row query blocks than SMs, with a short last round, so that persistent blocks
    take over blocks that have not started: every row of O and of the log-sum-exp against
    the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, H, N = 1, sms + 3, 512  # 2 blocks per head: one full round and 6 blocks more
    Q, K, V, _ = si.draw_sdpa(B, H, N, N, dtype="bf16", seed=4242)
    O, lse = mha.sdpa_with_lse(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                               to_dev(V, torch.bfloat16), mask)
    ref = oracle.sdpa_ref(Q, K, V, mask)
    assert_bf16_close(host(O), ref, f"sdpa bf16 {H} heads {mask}")
    lse_ref = oracle.sdpa_lse_ref(Q, K, mask)
    assert np.allclose(host(lse), lse_ref, rtol=0, atol=2e-3)


def test_sdpa_bf16_large_scores_stay_finite():
    # scores of +-40 whose tile maxima grow along the keys: later tiles are exponentiated
    # against the smaller first-tile max (large but finite exponentials)
    g = np.random.Generator(np.random.PCG64(5))
    B, H, N = 1, 2, 700
    Q = si.round_bf16(2.5 * g.standard_normal((B, H, N, 64)))
    K = si.round_bf16(2.5 * g.standard_normal((B, H, N, 64)) * np.linspace(0.2, 1.5, N)[:, None])
    V = si.round_bf16(g.standard_normal((B, H, N, 64)))
    for mask in ["none", "causal"]:
        O = mha.sdpa(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                     to_dev(V, torch.bfloat16), mask)
        assert_bf16_close(host(O), oracle.sdpa_ref(Q, K, V, mask), f"sdpa bf16 large {mask}")


def test_sdpa_bf16_later_tiles_overflowing_the_first_tile_max():
    # Key tile k has its keys scaled by 0.05 * 3^k, so a row's scores jump by far more than
    # 64 / (scale * log2 e) between tiles: the exponentials taken against an earlier tile's
    # max would overflow, and the kernel must rebuild those tiles with the larger max
    # (thousands of such tiles over these rows, several per row, with every mask).  The
    # rows end up nearly one-hot, so O is close to a single value row: V is drawn at half
    # scale to keep |O| below ~2.5, where a bf16 output's own rounding stays well inside the
    # absolute tolerance.
    g = np.random.Generator(np.random.PCG64(7))
    B, H, N = 2, 2, 900
    Q = si.round_bf16(4.0 * g.standard_normal((B, H, N, 64)))
    ramp = 0.05 * 3.0 ** (np.arange(N) // 128)
    K = si.round_bf16(g.standard_normal((B, H, N, 64)) * ramp[:, None])
    V = si.round_bf16(0.5 * g.standard_normal((B, H, N, 64)))
    key_len = np.array([900, 650], dtype=np.int32)
    for mask in ["none", "causal", "key_padding", "window"]:
        kl = key_len if mask == "key_padding" else None
        win = 300 if mask == "window" else None
        O = mha.sdpa(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                     to_dev(V, torch.bfloat16), mask,
                     key_len=None if kl is None else torch.from_numpy(kl).cuda(), window=win)
        got = host(O)
        assert np.all(np.isfinite(got))
        assert_bf16_close(got, oracle.sdpa_ref(Q, K, V, mask, kl, window=win),
                          f"sdpa bf16 overflow {mask}")


WINDOW_CASES = [
    (1, 2, 640, 0), (1, 2, 640, 1), (1, 1, 640, 63), (2, 1, 700, 128), (1, 2, 1000, 300),
    (1, 1, 129, 5), (1, 1, 1, 3), (1, 1, 300, 299), (1, 1, 300, 5000),
]


@pytest.mark.parametrize("B,H,N,win", WINDOW_CASES)
def test_sdpa_bf16_window(B, H, N, win):
    Q, K, V, _ = si.draw_sdpa(B, H, N, N, dtype="bf16", seed=300 + N + win)
    O = mha.sdpa(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16), to_dev(V, torch.bfloat16),
                 "window", window=win)
    assert_bf16_close(host(O), oracle.sdpa_ref(Q, K, V, "window", window=win),
                      f"sdpa bf16 window {B}x{H} N={N} w={win}")


@pytest.mark.parametrize("N,win,dk,dv", [(77, 3, 64, 64), (50, 0, 32, 48), (40, 100, 128, 16)])
def test_sdpa_f32_window(N, win, dk, dv):
    Q, K, V, _ = si.draw_sdpa(2, 2, N, N, dk, dv, "f32", seed=17)
    O = mha.sdpa(to_dev(Q, torch.float32), to_dev(K, torch.float32), to_dev(V, torch.float32),
                 "window", window=win)
    assert_f32_close(host(O), oracle.sdpa_ref(Q, K, V, "window", window=win),
                     f"sdpa f32 window N={N} w={win}")


def test_sdpa_bf16_window_keys_outside_band_cannot_change_outputs_bitwise():
    B, H, N, win = 1, 2, 900, 100
    Q, K, V, _ = si.draw_sdpa(B, H, N, N, dtype="bf16", seed=33)
    tq = to_dev(Q, torch.bfloat16)
    O = host(mha.sdpa(tq, to_dev(K, torch.bfloat16), to_dev(V, torch.bfloat16), "window",
                      window=win))
    rows = slice(400, 500)   # their bands cover keys 300..599
    K2, V2 = K.copy(), V.copy()
    K2[:, :, :300] = si.round_bf16(K2[:, :, :300] * -2.0 + 1.0)
    K2[:, :, 600:] = 3.0
    V2[:, :, :300] = -6.0
    V2[:, :, 600:] = 6.0
    O2 = host(mha.sdpa(tq, to_dev(K2, torch.bfloat16), to_dev(V2, torch.bfloat16), "window",
                       window=win))
    assert np.array_equal(O[:, :, rows], O2[:, :, rows])
    assert not np.array_equal(O[:, :, :200], O2[:, :, :200])


def test_sdpa_bf16_window_big_workload_sampled_rows():
    # the big model's heads at n = 4096 with a 513-key neighbourhood, rows sampled per (b, h)
    w = si.WORKLOADS["big_long_b8_n4096"]
    win = 256
    Q, K, V, _ = si.draw_sdpa(w.B, w.H, w.Nq, w.Nk, dtype="bf16", seed=w.seed)
    O = host(mha.sdpa(to_dev(Q, torch.bfloat16), to_dev(K, torch.bfloat16),
                      to_dev(V, torch.bfloat16), "window", window=win))
    g = np.random.Generator(np.random.PCG64(81))
    for b, h in [(0, 0), (w.B - 1, w.H - 1), (3, 7)]:
        rows = np.unique(np.concatenate([[0, 255, 256, w.Nq - 1], g.integers(0, w.Nq, 28)]))
        allowed = oracle.allowed_keys("window", w.Nq, w.Nk, rows=rows, window=win)
        ref = oracle.attention_weights_ref(Q[b, h, rows], K[b, h], allowed) @ \
            np.asarray(V[b, h], np.float64)
        assert_bf16_close(O[b, h, rows], ref, f"sdpa bf16 window big b={b} h={h}")


def test_sdpa_bf16_packed_qkv_and_concat_layout():
    # Q|K|V read straight from a projection buffer [B, N, 3, H, 64]; O written as [B, N, H*64]
    B, H, N = 2, 4, 333
    g = np.random.Generator(np.random.PCG64(21))
    buf = si.round_bf16(g.standard_normal((B, N, 3, H, 64)))
    tb = to_dev(buf, torch.bfloat16)
    q, k, v = (tb[:, :, i].permute(0, 2, 1, 3) for i in range(3))
    out = torch.zeros((B, N, H * 64), dtype=torch.bfloat16, device="cuda")
    o_view = out.view(B, N, H, 64).permute(0, 2, 1, 3)
    mha.sdpa(q, k, v, "causal", out=o_view)
    Q, K, V = (np.moveaxis(buf[:, :, i], 1, 2) for i in range(3))
    ref = np.moveaxis(oracle.sdpa_ref(Q, K, V, "causal"), 1, 2).reshape(B, N, H * 64)
    assert_bf16_close(host(out), ref, "sdpa bf16 packed/concat")


def test_sdpa_bf16_masked_keys_cannot_change_outputs_bitwise():
    B, H, N = 2, 2, 390
    Q, K, V, _ = si.draw_sdpa(B, H, N, N, dtype="bf16", seed=31)
    tq = to_dev(Q, torch.bfloat16)
    O = host(mha.sdpa(tq, to_dev(K, torch.bfloat16), to_dev(V, torch.bfloat16), "causal"))
    i0 = 200
    K2, V2 = K.copy(), V.copy()
    K2[:, :, i0 + 1:] = si.round_bf16(K2[:, :, i0 + 1:] * -3.0 + 1.0)
    V2[:, :, i0 + 1:] = 7.0
    O2 = host(mha.sdpa(tq, to_dev(K2, torch.bfloat16), to_dev(V2, torch.bfloat16), "causal"))
    assert np.array_equal(O[:, :, :i0 + 1], O2[:, :, :i0 + 1])
    assert not np.array_equal(O[:, :, i0 + 1:], O2[:, :, i0 + 1:])
    kl = np.array([150, 300], np.int32)
    tkl = to_dev(kl, torch.int32)
    O = host(mha.sdpa(tq, to_dev(K, torch.bfloat16), to_dev(V, torch.bfloat16), "key_padding", tkl))
    K3, V3 = K.copy(), V.copy()
    for b in range(B):
        K3[b, :, kl[b]:] = 3.0
        V3[b, :, kl[b]:] = -5.0
    O3 = host(mha.sdpa(tq, to_dev(K3, torch.bfloat16), to_dev(V3, torch.bfloat16),
                       "key_padding", tkl))
    assert np.array_equal(O, O3)


def test_sdpa_bf16_deterministic():
    Q, K, V, _ = si.draw_sdpa(2, 4, 600, 600, dtype="bf16", seed=41)
    args = [to_dev(a, torch.bfloat16) for a in (Q, K, V)]
    a = mha.sdpa(*args, "causal")
    b = mha.sdpa(*args, "causal")
    assert torch.equal(a, b)


# ------------------------------------------------------------------------ projection GEMM

@pytest.mark.parametrize("M,N,K,bias", [
    (1, 64, 64, False),
    (300, 192, 128, True),
    (1000, 1536, 512, True),     # 128-wide tiles
    (9800, 512, 512, True),      # enough tiles for the 256-wide variant
    (4096, 1024, 1024, False),
    (8192, 3072, 256, True),
])
def test_linear_bf16(M, N, K, bias):
    g = np.random.Generator(np.random.PCG64(M + N + K))
    X = si.round_bf16(g.standard_normal((M, K)))
    W = si.round_bf16(g.uniform(-0.08, 0.08, (N, K)))
    b = si.round_bf16(0.1 * g.standard_normal(N)) if bias else None
    Y = mha.linear(to_dev(X, torch.bfloat16), to_dev(W, torch.bfloat16), to_dev(b, torch.bfloat16))
    assert_bf16_close(host(Y), oracle.linear_ref(X, W, b), f"linear bf16 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K,bias,relu", [
    (9800, 2048, 512, True, False),   # last row band: the odd CTA of the pair has no rows
    (9900, 2112, 448, True, True),    # ragged N: the odd CTA's W rows of the last band past N
    (16384, 2048, 1024, False, False),
])
def test_linear_bf16_pair_tiles(M, N, K, bias, relu):
    """Shapes with at least four rounds of 256 x 256 tiles run on pairs of SMs.  Weights in
    [-0.04, 0.04] keep every |y| below 8, where half a bf16 ulp of the rounded output stays
    under the 2e-2 bound (tens of millions of outputs with the wider weights of the other cases
    reach |y| > 8, whose half-ulp is 0.031)."""
    g = np.random.Generator(np.random.PCG64(M * 7 + N + K))
    X = si.round_bf16(g.standard_normal((M, K)))
    W = si.round_bf16(g.uniform(-0.04, 0.04, (N, K)))
    b = si.round_bf16(0.1 * g.standard_normal(N)) if bias else None
    Y = mha.linear(to_dev(X, torch.bfloat16), to_dev(W, torch.bfloat16),
                   to_dev(b, torch.bfloat16), relu=relu)
    ref = oracle.linear_ref(X, W, b)
    if relu:
        ref = np.maximum(ref, 0.0)
    assert_bf16_close(host(Y), ref, f"linear bf16 pair tiles {M}x{N}x{K}")


@pytest.mark.parametrize("M1, N1, M2, N2, K", [(4096, 512, 8192, 1024, 512),
                                               (300, 128, 1000, 192, 64),
                                               (8192, 1024, 16384, 2048, 1024)])
def test_linear2_bf16(M1, N1, M2, N2, K):
    """The two projections of encoder-decoder attention in one launch: each output equals its
    own mha_linear_fwd call bit for bit and the oracle within the bf16 bound (the last case
    is large enough that each problem alone would take the pair-SM form: two launches)."""
    g = np.random.Generator(np.random.PCG64(M1 + N2 * 3 + K))
    X1 = si.round_bf16(g.standard_normal((M1, K)))
    X2 = si.round_bf16(g.standard_normal((M2, K)))
    W1 = si.round_bf16(g.uniform(-0.04, 0.04, (N1, K)))
    W2 = si.round_bf16(g.uniform(-0.04, 0.04, (N2, K)))
    b1 = si.round_bf16(0.1 * g.standard_normal(N1))
    b2 = si.round_bf16(0.1 * g.standard_normal(N2))
    d = [to_dev(a, torch.bfloat16) for a in (X1, W1, b1, X2, W2, b2)]
    y1, y2 = mha.linear2(*d)
    assert torch.equal(y1, mha.linear(d[0], d[1], d[2]))
    assert torch.equal(y2, mha.linear(d[3], d[4], d[5]))
    assert_bf16_close(host(y1), oracle.linear_ref(X1, W1, b1), f"linear2 first {M1}x{N1}x{K}")
    assert_bf16_close(host(y2), oracle.linear_ref(X2, W2, b2), f"linear2 second {M2}x{N2}x{K}")


def test_linear_bf16_row_pitch():
    g = np.random.Generator(np.random.PCG64(3))
    X = si.round_bf16(g.standard_normal((257, 320)))
    W = si.round_bf16(g.uniform(-0.08, 0.08, (128, 256)))
    tx = to_dev(X, torch.bfloat16)[:, :256]                      # row pitch 320
    wide = torch.zeros((257, 200), dtype=torch.bfloat16, device="cuda")
    Y = mha.linear(tx, to_dev(W, torch.bfloat16), out=wide[:, :128])  # row pitch 200
    assert_bf16_close(host(Y), oracle.linear_ref(X[:, :256], W), "linear bf16 pitch")
    assert torch.count_nonzero(wide[:, 128:]) == 0                # nothing past column N
    with pytest.raises(ValueError):
        mha.linear(tx, to_dev(W, torch.bfloat16), out=wide[:, :120])


def test_linear_f32():
    g = np.random.Generator(np.random.PCG64(4))
    X = g.standard_normal((130, 96)).astype(np.float32)
    W = g.uniform(-0.1, 0.1, (70, 96)).astype(np.float32)
    b = g.standard_normal(70).astype(np.float32)
    Y = mha.linear(to_dev(X, torch.float32), to_dev(W, torch.float32), to_dev(b, torch.float32))
    assert_f32_close(host(Y), oracle.linear_ref(X, W, b), "linear f32")


# ------------------------------------------------------------------------ residual LayerNorm

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,D", [(1, 8), (333, 512), (65, 1024), (10, 200), (7, 2048),
                                 (4099, 1024)])
def test_residual_layernorm(dtype, M, D):
    g = np.random.Generator(np.random.PCG64(M * D))
    rnd = si.round_bf16 if dtype == torch.bfloat16 else (lambda a: a.astype(np.float32))
    x = rnd(g.standard_normal((M, D)) * 2 + 0.5)
    a = rnd(0.3 * g.standard_normal((M, D)))
    gm = rnd(1 + 0.1 * g.standard_normal(D))
    bt = rnd(0.1 * g.standard_normal(D))
    y = mha.residual_layernorm(to_dev(x, dtype), to_dev(a, dtype), to_dev(gm, dtype),
                               to_dev(bt, dtype), 1e-5)
    ref = oracle.layernorm_ref(x.astype(np.float64) + a, gm, bt, 1e-5)
    check = assert_bf16_close if dtype == torch.bfloat16 else assert_f32_close
    check(host(y), ref, f"residual LN {dtype} {M}x{D}")


# ------------------------------------------------------------------------ the whole sublayer

def run_layer(inp, w, dtype=torch.bfloat16):
    t = {k: to_dev(v, dtype) for k, v in inp.items() if k != "key_len"}
    key_len = to_dev(inp["key_len"], torch.int32)
    return mha.mha_layer(t["x_q"], t["x_kv"], t["W_qkv"], t["b_qkv"], t["W_o"], t["b_o"],
                         t["gamma"], t["beta"], w.H, w.mask, key_len)


def ref_layer(inp, w):
    return oracle.mha_layer_ref(inp["x_q"], inp["x_kv"], inp["W_qkv"], inp["b_qkv"], inp["W_o"],
                                inp["b_o"], inp["gamma"], inp["beta"], w.H, w.mask,
                                inp["key_len"])


@pytest.mark.parametrize("name", ["enc_self_base_b32_n128", "dec_causal_base_b32_n256",
                                  "cross_pad_base_b32_q128_k256"])
def test_layer_base_workloads(name):
    w = si.WORKLOADS[name]
    inp = si.draw_layer(w)
    y = run_layer(inp, w)
    assert_bf16_close(host(y), ref_layer(inp, w), name)


@pytest.mark.parametrize("mask,cross,Nq,Nk", [
    ("none", False, 70, 70),
    ("causal", False, 300, 300),
    ("key_padding", True, 130, 200),
    ("none", True, 64, 257),
])
def test_layer_bf16_with_biases_and_affine(mask, cross, Nq, Nk):
    w = si.Workload("t", "layer", "bf16", B=3, H=4, Nq=Nq, Nk=Nk, mask=mask, cross=cross, seed=77)
    inp = si.draw_layer(w, affine=True)
    if mask == "key_padding":
        inp["key_len"] = np.array([0, 5, Nk], np.int32)
    y = run_layer(inp, w)
    assert_bf16_close(host(y), ref_layer(inp, w), f"layer bf16 affine {mask} cross={cross}")


@pytest.mark.parametrize("cross", [False, True])
def test_layer_bf16_more_attention_units_than_sms(cross):
    """More attention units (256-row query blocks) than SMs and a last round that fills at
    most half of them, self- and cross-attention: the whole output against the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B = (sms + 8) // 4 + 1  # 2 heads x 2 query blocks per batch element
    units = 4 * B
    assert units > sms and 0 < units % sms <= sms // 2
    w = si.Workload("t", "layer", "bf16", B=B, H=2, Nq=512, Nk=512 if not cross else 700,
                    cross=cross, seed=91)
    inp = si.draw_layer(w, affine=True)
    y = run_layer(inp, w)
    assert_bf16_close(host(y), ref_layer(inp, w), f"layer bf16 {B}x512 cross={cross}")


@pytest.mark.parametrize("mask,cross,H,dk", [("none", False, 2, 64), ("causal", False, 3, 32),
                                             ("key_padding", True, 4, 16)])
def test_layer_f32(mask, cross, H, dk):
    w = si.Workload("t", "layer", "f32", B=2, H=H, Nq=40, Nk=40 if not cross else 75, d_k=dk,
                    d_v=dk, mask=mask, cross=cross, seed=78)
    inp = si.draw_layer(w, affine=True)
    if mask == "key_padding":
        inp["key_len"] = np.array([1, 75], np.int32)
    y = run_layer(inp, w, torch.float32)
    assert_f32_close(host(y), ref_layer(inp, w), f"layer f32 {mask}")


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_layer_big_long_sampled_rows(mask):
    """B=8, n=4096, d_model=1024, 16 heads, in the bench's launch configuration; the oracle
    evaluates 64 rows of the first and the last batch element one by one."""
    w = si.WORKLOADS["big_long_b8_n4096"].with_mask(mask)
    inp = si.draw_layer(w)
    y = host(run_layer(inp, w))
    g = np.random.Generator(np.random.PCG64(99))
    rows = np.concatenate([[0, 1, 127, 128, 4095], g.choice(np.arange(2, 4095), 59, replace=False)])
    for b in (0, w.B - 1):
        ref = oracle.mha_layer_rows_ref(inp["x_q"], None, inp["W_qkv"], inp["b_qkv"], inp["W_o"],
                                        inp["b_o"], inp["gamma"], inp["beta"], w.H, b, rows, mask)
        assert_bf16_close(y[b, rows], ref, f"big layer {mask} b={b}")
    assert np.all(np.isfinite(y))


# ------------------------------------------------------------------------ failure detection

def test_bounded_wait_reports_timeout_and_context_survives():
    assert mha.wait_selftest(200_000) == -6
    assert mha.device_status() == 0
    Q, K, V, _ = si.draw_sdpa(1, 1, 130, 130, dtype="bf16", seed=1)
    O = mha.sdpa(*(to_dev(a, torch.bfloat16) for a in (Q, K, V)))
    assert_bf16_close(host(O), oracle.sdpa_ref(Q, K, V), "sdpa after self test")
