"""One generation step against a key/value cache: CUDA path (mha_sdpa_decode_fwd through the C
ABI) vs the CPU oracle on the same seeded inputs.

Cache lengths are ragged per batch element and span several 256-key chunks, so the split-K
merge is exercised with partial and empty chunks.
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


def dev(a, dtype):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to("cuda", dtype)


def host(t):
    return t.float().cpu().numpy()


def draw(B, H, Nq, Lmax, dtype, seed, d=64):
    g = np.random.Generator(np.random.PCG64(seed))
    fin = si.round_bf16 if dtype == "bf16" else (lambda a: np.asarray(a, np.float32))
    Q = fin(g.standard_normal((B, H, Nq, d)))
    K = fin(g.standard_normal((B, H, Lmax, d)))
    V = fin(g.standard_normal((B, H, Lmax, d)))
    return Q, K, V


def ref_decode(Q, K, V, cache_len, causal):
    """The oracle's definition, with rows that have no allowed key set to zero."""
    B, H, Nq, _ = Q.shape
    Lmax = K.shape[2]
    out = np.zeros((B, H, Nq, V.shape[3]))
    for b in range(B):
        L = int(np.clip(cache_len[b], 0, Lmax))
        if causal and L >= Nq:
            out[b] = oracle.sdpa_ref(Q[b:b + 1], K[b:b + 1], V[b:b + 1], "causal_cache",
                                     np.array([L], np.int32))[0]
        elif not causal:
            out[b] = oracle.sdpa_ref(Q[b:b + 1], K[b:b + 1], V[b:b + 1], "key_padding",
                                     np.array([L], np.int32))[0]
        else:  # fewer cached positions than queries: only the last L rows see keys
            i = np.arange(Nq)[:, None]
            j = np.arange(Lmax)[None, :]
            allowed = (j <= L - Nq + i) & (j < L)
            for h in range(H):
                w = oracle.attention_weights_ref(Q[b, h], K[b, h], allowed)
                out[b, h] = w @ np.asarray(V[b, h], np.float64)
    return out


CASES = [  # B, H, Nq, Lmax, cache_len, causal
    (3, 2, 1, 700, [700, 300, 129], True),
    (3, 2, 4, 700, [700, 300, 129], True),
    (2, 2, 16, 1000, [1000, 517], True),
    (3, 2, 1, 1000, [1000, 1, 517], False),
    (2, 1, 5, 1000, [0, 777], False),
    (2, 2, 8, 300, [3, 256], True),          # 3 cached positions for 8 queries: 5 empty rows
    (1, 1, 1, 1, [1], True),
    (2, 1, 2, 513, [2, 999], True),          # cache_len past Lmax is clamped to Lmax
]


@pytest.mark.parametrize("B,H,Nq,Lmax,cl,causal", CASES)
def test_decode_bf16(B, H, Nq, Lmax, cl, causal):
    Q, K, V = draw(B, H, Nq, Lmax, "bf16", seed=400 + Nq + Lmax)
    cache_len = np.array(cl, np.int32)
    O = mha.sdpa_decode(dev(Q, torch.bfloat16), dev(K, torch.bfloat16), dev(V, torch.bfloat16),
                        dev(cache_len, torch.int32), causal=causal)
    got = host(O)
    ref = ref_decode(Q, K, V, cache_len, causal)
    assert_bf16_close(got, ref, f"decode bf16 B{B} H{H} Nq{Nq} L{cl} causal={causal}")
    zero_rows = np.all(ref == 0.0, axis=-1)
    assert np.all(got[zero_rows] == 0.0)


@pytest.mark.parametrize("Nq,causal", [(1, True), (3, True), (2, False)])
def test_decode_f32(Nq, causal):
    Q, K, V = draw(2, 2, Nq, 300, "f32", seed=450 + Nq, d=48)
    cache_len = np.array([300, 97], np.int32)
    O = mha.sdpa_decode(dev(Q, torch.float32), dev(K, torch.float32), dev(V, torch.float32),
                        dev(cache_len, torch.int32), causal=causal)
    assert_f32_close(host(O), ref_decode(Q, K, V, cache_len, causal), f"decode f32 Nq{Nq}")


def test_decode_stale_cache_entries_cannot_change_outputs_bitwise():
    B, H, Nq, Lmax = 2, 2, 3, 900
    Q, K, V = draw(B, H, Nq, Lmax, "bf16", seed=461)
    cl = np.array([400, 650], np.int32)
    args = [dev(Q, torch.bfloat16)]
    O = host(mha.sdpa_decode(*args, dev(K, torch.bfloat16), dev(V, torch.bfloat16),
                             dev(cl, torch.int32)))
    K2, V2 = K.copy(), V.copy()
    for b in range(B):
        K2[b, :, cl[b]:] = 9.0
        V2[b, :, cl[b]:] = -7.0
    O2 = host(mha.sdpa_decode(*args, dev(K2, torch.bfloat16), dev(V2, torch.bfloat16),
                              dev(cl, torch.int32)))
    assert np.array_equal(O, O2)


def test_decode_from_token_major_cache():
    # the cache kept token-major [B, Lmax, H, 64] (as a projection buffer writes it): strided views
    B, H, Nq, Lmax = 2, 4, 2, 600
    g = np.random.Generator(np.random.PCG64(471))
    Kt = si.round_bf16(g.standard_normal((B, Lmax, H, 64)))
    Vt = si.round_bf16(g.standard_normal((B, Lmax, H, 64)))
    Q = si.round_bf16(g.standard_normal((B, H, Nq, 64)))
    cl = np.array([600, 333], np.int32)
    tk, tv = dev(Kt, torch.bfloat16), dev(Vt, torch.bfloat16)
    O = mha.sdpa_decode(dev(Q, torch.bfloat16), tk.permute(0, 2, 1, 3), tv.permute(0, 2, 1, 3),
                        dev(cl, torch.int32))
    K, V = np.moveaxis(Kt, 1, 2), np.moveaxis(Vt, 1, 2)
    assert_bf16_close(host(O), ref_decode(Q, K, V, cl, True), "decode token-major cache")


def test_decode_step_matches_row_of_full_causal_attention():
    # generating position t from the cache of positions 0..t gives row t of the training-time
    # causal attention over the whole sequence (both on the GPU, both against the oracle)
    H, T = 2, 777
    Q, K, V, _ = si.draw_sdpa(1, H, T, T, dtype="bf16", seed=481)
    tq, tk, tv = (dev(a, torch.bfloat16) for a in (Q, K, V))
    full = host(mha.sdpa(tq, tk, tv, "causal"))
    for t in (0, 255, 256, 600, T - 1):
        o = host(mha.sdpa_decode(tq[:, :, t:t + 1], tk, tv,
                                 torch.tensor([t + 1], dtype=torch.int32, device="cuda")))
        assert_bf16_close(o[:, :, 0], full[:, :, t], f"decode step t={t} vs full causal row")


def test_decode_big_workload_sampled_heads():
    # one generation step for 64 sequences of the big model (h = 16) with up to 4096 cached
    # positions each
    B, H, Lmax = 64, 16, 4096
    g = np.random.Generator(np.random.PCG64(491))
    Q = si.round_bf16(g.standard_normal((B, H, 1, 64)))
    K = si.round_bf16(g.standard_normal((B, H, Lmax, 64)))
    V = si.round_bf16(g.standard_normal((B, H, Lmax, 64)))
    cl = g.integers(1, Lmax + 1, B).astype(np.int32)
    cl[0], cl[1] = Lmax, 1
    O = host(mha.sdpa_decode(dev(Q, torch.bfloat16), dev(K, torch.bfloat16),
                             dev(V, torch.bfloat16), dev(cl, torch.int32)))
    for b, h in [(0, 0), (1, 5), (17, 15), (63, 7)]:
        ref = ref_decode(Q[b:b + 1, h:h + 1], K[b:b + 1, h:h + 1], V[b:b + 1, h:h + 1],
                         cl[b:b + 1], True)
        assert_bf16_close(O[b:b + 1, h:h + 1], ref, f"decode big b={b} h={h} L={cl[b]}")
