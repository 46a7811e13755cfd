"""The C ABI on the host: the library builds, loads and exports every symbol include/mha.h
declares, and argument validation returns its status codes before anything is launched.
No call here reaches a GPU (they all fail validation first), so this runs without one."""
import ctypes
import os
import re

import pytest

from transformer_head_scaled_04_gb300 import _capi as C
from transformer_head_scaled_04_gb300 import build as B

HEADER = os.path.join(B.INCLUDE, "mha.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return C.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mha_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for need in ["mha_sdpa_fwd", "mha_layer_fwd", "mha_layer_workspace_size", "mha_status_string",
                 "mha_debug_last_device_status"]:
        assert need in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libmha.so does not export {name}"
    assert set(C.PROTOTYPES) == set(declared_functions())


def test_abi_version_and_status_strings(lib):
    assert lib.mha_abi_version() == 100
    for code in range(0, -8, -1):
        s = C.status_string(code)
        assert s.startswith("MHA_")
    assert C.status_string(-99) == "unknown mha status"


FAKE = ctypes.c_void_p(0x10000)       # never dereferenced: validation fails before any launch
ODD = ctypes.c_void_p(0x10002)        # 2-byte aligned only


def sdpa(lib, B=1, H=1, Nq=4, Nk=4, dk=64, dv=64, dt=1, mask=0, key_len=None, scale=0.0,
         q=FAKE, k=FAKE, v=FAKE, o=FAKE, strides=None):
    return lib.mha_sdpa_fwd(B, H, Nq, Nk, dk, dv, dt, mask, key_len, scale, q, k, v, o, strides,
                            None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), C.MHA_ERR_INVALID),
    (dict(H=-1), C.MHA_ERR_INVALID),
    (dict(Nq=0), C.MHA_ERR_INVALID),
    (dict(dt=7), C.MHA_ERR_INVALID),
    (dict(mask=3), C.MHA_ERR_INVALID),
    (dict(mask=1, Nq=4, Nk=5), C.MHA_ERR_INVALID),          # causal needs Nq == Nk
    (dict(mask=2), C.MHA_ERR_INVALID),                       # key padding needs key_len
    (dict(q=None), C.MHA_ERR_INVALID),
    (dict(scale=float("nan")), C.MHA_ERR_INVALID),
    (dict(dk=32), C.MHA_ERR_UNSUPPORTED),                    # bf16 path is d = 64
    (dict(dt=0, dk=256), C.MHA_ERR_UNSUPPORTED),             # fp32 path d <= 128
    (dict(q=ODD), C.MHA_ERR_ALIGN),
    (dict(dt=0, o=ODD), C.MHA_ERR_ALIGN),
])
def test_sdpa_validation(lib, kw, code):
    assert sdpa(lib, **kw) == code


def test_sdpa_stride_validation(lib):
    bad = (ctypes.c_int64 * 16)(*([256, 256, 64, 2] + [256, 256, 64, 1] * 3))
    assert sdpa(lib, strides=ctypes.cast(bad, ctypes.c_void_p)) == C.MHA_ERR_UNSUPPORTED
    bad = (ctypes.c_int64 * 16)(*([256, 256, 60, 1] + [256, 256, 64, 1] * 3))
    assert sdpa(lib, strides=ctypes.cast(bad, ctypes.c_void_p)) == C.MHA_ERR_ALIGN
    neg = (ctypes.c_int64 * 16)(*([256, -256, 64, 1] + [256, 256, 64, 1] * 3))
    assert sdpa(lib, strides=ctypes.cast(neg, ctypes.c_void_p)) == C.MHA_ERR_INVALID


def layer(lib, B=2, H=8, Nq=16, Nk=16, D=512, dk=64, dv=64, dt=1, mask=0, key_len=None,
          eps=1e-5, x_q=FAKE, x_kv=None, W_qkv=FAKE, W_o=FAKE, y=FAKE, ws=FAKE, ws_bytes=1 << 30):
    return lib.mha_layer_fwd(B, H, Nq, Nk, D, dk, dv, dt, mask, key_len, eps, x_q, x_kv, W_qkv,
                             None, W_o, None, None, None, y, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), C.MHA_ERR_INVALID),
    (dict(Nk=32), C.MHA_ERR_INVALID),                        # self-attention needs Nq == Nk
    (dict(x_kv=FAKE, Nk=32, mask=1), C.MHA_ERR_INVALID),     # causal needs Nq == Nk
    (dict(mask=2), C.MHA_ERR_INVALID),
    (dict(W_o=None), C.MHA_ERR_INVALID),
    (dict(eps=-1.0), C.MHA_ERR_INVALID),
    (dict(dk=32, D=256), C.MHA_ERR_UNSUPPORTED),
    (dict(D=520), C.MHA_ERR_UNSUPPORTED),
    (dict(ws=None), C.MHA_ERR_WORKSPACE),
    (dict(ws_bytes=1024), C.MHA_ERR_WORKSPACE),
    (dict(x_q=ODD), C.MHA_ERR_ALIGN),
])
def test_layer_validation(lib, kw, code):
    assert layer(lib, **kw) == code


def test_workspace_size(lib):
    n = ctypes.c_size_t(0)
    assert lib.mha_layer_workspace_size(8, 16, 4096, 4096, 1024, 64, 64, 1, ctypes.byref(n)) == 0
    M = 8 * 4096
    # Q|K|V + concat + W^O output, bf16
    assert n.value == 2 * (M * 3 * 1024 + M * 1024 + M * 1024)
    assert lib.mha_layer_workspace_size(8, 16, 4096, 4096, 1024, 64, 64, 1, None) == \
        C.MHA_ERR_INVALID
    n2 = ctypes.c_size_t(0)
    assert lib.mha_layer_workspace_size(32, 8, 128, 256, 512, 64, 64, 1, ctypes.byref(n2)) == 0
    assert n2.value == 2 * (32 * 128 * 512 + 32 * 256 * 1024 + 2 * 32 * 128 * 512)


@pytest.mark.parametrize("args,code", [
    ((0, 64, 64, 1), C.MHA_ERR_INVALID),
    ((8, 64, 60, 1), C.MHA_ERR_UNSUPPORTED),   # bf16 K multiple of 64
    ((8, 96, 64, 1), C.MHA_ERR_UNSUPPORTED),   # bf16 N multiple of 64
])
def test_linear_validation(lib, args, code):
    M, N, K, dt = args
    assert lib.mha_linear_fwd(M, N, K, dt, FAKE, K, FAKE, None, FAKE, N, None) == code


def test_linear_pitch_and_alignment(lib):
    assert lib.mha_linear_fwd(8, 64, 64, 1, FAKE, 32, FAKE, None, FAKE, 64, None) == \
        C.MHA_ERR_INVALID
    assert lib.mha_linear_fwd(8, 64, 64, 1, FAKE, 68, FAKE, None, FAKE, 64, None) == \
        C.MHA_ERR_ALIGN
    assert lib.mha_linear_fwd(8, 64, 64, 1, ODD, 64, FAKE, None, FAKE, 64, None) == \
        C.MHA_ERR_ALIGN


def test_layernorm_validation(lib):
    f = lib.mha_residual_layernorm_fwd
    assert f(0, 64, 1, 1e-5, FAKE, FAKE, None, None, FAKE, None) == C.MHA_ERR_INVALID
    assert f(4, 60, 1, 1e-5, FAKE, FAKE, None, None, FAKE, None) == C.MHA_ERR_UNSUPPORTED
    assert f(4, 4096, 1, 1e-5, FAKE, FAKE, None, None, FAKE, None) == C.MHA_ERR_UNSUPPORTED
    assert f(4, 64, 1, 1e-5, FAKE, ODD, None, None, FAKE, None) == C.MHA_ERR_ALIGN
    assert f(4, 64, 1, float("nan"), FAKE, FAKE, None, None, FAKE, None) == C.MHA_ERR_INVALID


def test_linear_relu_validation_matches_linear(lib):
    for (M, N, K, dt), code in [((0, 64, 64, 1), C.MHA_ERR_INVALID),
                                ((8, 64, 60, 1), C.MHA_ERR_UNSUPPORTED),
                                ((8, 96, 64, 1), C.MHA_ERR_UNSUPPORTED)]:
        assert lib.mha_linear_relu_fwd(M, N, K, dt, FAKE, K, FAKE, None, FAKE, N, None) == code
    assert lib.mha_linear_relu_fwd(8, 64, 64, 1, ODD, 64, FAKE, None, FAKE, 64, None) == \
        C.MHA_ERR_ALIGN


def ffn(lib, M=64, D=512, d_ff=2048, dt=1, eps=1e-5, x=FAKE, W1=FAKE, W2=FAKE, y=FAKE, ws=FAKE,
        ws_bytes=1 << 30):
    return lib.mha_ffn_fwd(M, D, d_ff, dt, eps, x, W1, None, W2, None, None, None, y, ws,
                           ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=0), C.MHA_ERR_INVALID),
    (dict(d_ff=0), C.MHA_ERR_INVALID),
    (dict(dt=7), C.MHA_ERR_INVALID),
    (dict(x=None), C.MHA_ERR_INVALID),
    (dict(W2=None), C.MHA_ERR_INVALID),
    (dict(eps=float("nan")), C.MHA_ERR_INVALID),
    (dict(D=520), C.MHA_ERR_UNSUPPORTED),          # bf16: D multiple of 64
    (dict(d_ff=2000), C.MHA_ERR_UNSUPPORTED),      # bf16: d_ff multiple of 64
    (dict(D=4096, d_ff=4096), C.MHA_ERR_UNSUPPORTED),  # LayerNorm rows up to 2048
    (dict(dt=0, D=36), C.MHA_ERR_UNSUPPORTED),     # LayerNorm rows a multiple of 8
    (dict(ws=None), C.MHA_ERR_WORKSPACE),
    (dict(ws_bytes=1024), C.MHA_ERR_WORKSPACE),
    (dict(x=ODD), C.MHA_ERR_ALIGN),
    (dict(ws=ctypes.c_void_p(0x10010)), C.MHA_ERR_ALIGN),  # workspace 256-byte aligned
])
def test_ffn_validation(lib, kw, code):
    assert ffn(lib, **kw) == code


def test_ffn_workspace_and_timed_marks(lib):
    n = ctypes.c_size_t(0)
    assert lib.mha_ffn_workspace_size(32768, 1024, 4096, 1, ctypes.byref(n)) == 0
    assert n.value == 2 * (32768 * 4096 + 32768 * 1024)   # hidden + second map, bf16
    assert lib.mha_ffn_workspace_size(100, 64, 256, 0, ctypes.byref(n)) == 0
    assert n.value == 102400 + 25600                      # f32, each region 256-byte padded
    assert lib.mha_ffn_workspace_size(0, 64, 256, 0, ctypes.byref(n)) == C.MHA_ERR_INVALID
    assert lib.mha_ffn_fwd_timed(64, 512, 2048, 1, 1e-5, FAKE, FAKE, None, FAKE, None, None,
                                 None, FAKE, FAKE, 1 << 30, None, None, 4) == C.MHA_ERR_INVALID
    ev = (ctypes.c_void_p * 4)(FAKE, FAKE, None, FAKE)
    assert lib.mha_ffn_fwd_timed(64, 512, 2048, 1, 1e-5, FAKE, FAKE, None, FAKE, None, None,
                                 None, FAKE, FAKE, 1 << 30, None,
                                 ctypes.cast(ev, ctypes.c_void_p), 4) == C.MHA_ERR_INVALID


def test_encoder_layer_workspace_and_validation(lib):
    n = ctypes.c_size_t(0)
    assert lib.mha_encoder_layer_workspace_size(8, 4096, 16, 1024, 4096, 1,
                                                ctypes.byref(n)) == 0
    M = 8 * 4096
    h = 2 * M * 1024
    attention = 2 * (M * 3 * 1024 + M * 1024 + M * 1024)
    feed_forward = 2 * (M * 4096 + M * 1024)
    assert n.value == h + max(attention, feed_forward)
    assert lib.mha_encoder_layer_workspace_size(8, 4096, 16, 1000, 4096, 1,
                                                ctypes.byref(n)) == C.MHA_ERR_INVALID  # D % H
    assert lib.mha_encoder_layer_workspace_size(8, 4096, 16, 1024, 4000, 1,
                                                ctypes.byref(n)) == C.MHA_ERR_UNSUPPORTED

    def enc(**kw):
        a = dict(B=2, N=16, H=8, D=512, d_ff=2048, dt=1, mask=0, x=FAKE, y=ctypes.c_void_p(0x20000),
                 ws=FAKE, ws_bytes=1 << 30)
        a.update(kw)
        return lib.mha_encoder_layer_fwd(a["B"], a["N"], a["H"], a["D"], a["d_ff"], a["dt"],
                                         a["mask"], None, 1e-5, a["x"], FAKE, None, FAKE, None,
                                         None, None, FAKE, None, FAKE, None, None, None, a["y"],
                                         a["ws"], a["ws_bytes"], None)

    assert enc(B=0) == C.MHA_ERR_INVALID
    assert enc(ws_bytes=4096) == C.MHA_ERR_WORKSPACE
    assert enc(ws=None) == C.MHA_ERR_WORKSPACE
    assert enc(y=FAKE) == C.MHA_ERR_INVALID          # y aliases x
    assert enc(mask=2) == C.MHA_ERR_INVALID          # key padding without key_len
    assert enc(x=ODD) == C.MHA_ERR_ALIGN


def test_product_path_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(C, "_lib", None)
    monkeypatch.setattr(C, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        C.load()


def test_sdpa_window_validation(lib):
    f = lib.mha_sdpa_window_fwd
    assert f(1, 1, 8, 64, 64, 1, -1, 0.0, FAKE, FAKE, FAKE, FAKE, None, None) == C.MHA_ERR_INVALID
    assert f(0, 1, 8, 64, 64, 1, 2, 0.0, FAKE, FAKE, FAKE, FAKE, None, None) == C.MHA_ERR_INVALID
    assert f(1, 1, 8, 32, 64, 1, 2, 0.0, FAKE, FAKE, FAKE, FAKE, None, None) == \
        C.MHA_ERR_UNSUPPORTED
    assert f(1, 1, 8, 64, 64, 1, 2, 0.0, ODD, FAKE, FAKE, FAKE, None, None) == C.MHA_ERR_ALIGN
    assert f(1, 1, 8, 64, 64, 1, 2, 0.0, FAKE, FAKE, FAKE, None, None, None) == C.MHA_ERR_INVALID
    # the window is not one of mha_sdpa_fwd's mask kinds
    assert lib.mha_sdpa_fwd(1, 1, 8, 8, 64, 64, 1, 3, None, 0.0, FAKE, FAKE, FAKE, FAKE, None,
                            None) == C.MHA_ERR_INVALID


def test_decode_workspace_and_validation(lib):
    n = ctypes.c_size_t(0)
    assert lib.mha_decode_workspace_size(64, 16, 1, 4096, 1, ctypes.byref(n)) == 0
    assert n.value == 64 * 16 * 16 * 1 * 66 * 4           # 16 chunks of 256 keys, fp32 partials
    assert lib.mha_decode_workspace_size(2, 2, 3, 300, 1, ctypes.byref(n)) == 0
    assert n.value == (2 * 2 * 2 * 3 * 66 * 4 + 255) // 256 * 256
    assert lib.mha_decode_workspace_size(1, 1, 17, 300, 1, ctypes.byref(n)) == \
        C.MHA_ERR_UNSUPPORTED
    assert lib.mha_decode_workspace_size(1, 1, 17, 300, 0, ctypes.byref(n)) == 0   # fp32: any Nq

    def dec(**kw):
        a = dict(B=2, H=2, Nq=1, L=300, dk=64, dv=64, dt=1, causal=1, cl=FAKE, Q=FAKE, ws=FAKE,
                 ws_bytes=1 << 20)
        a.update(kw)
        return lib.mha_sdpa_decode_fwd(a["B"], a["H"], a["Nq"], a["L"], a["dk"], a["dv"], a["dt"],
                                       a["causal"], a["cl"], 0.0, a["Q"], FAKE, FAKE, FAKE, None,
                                       a["ws"], a["ws_bytes"], None)

    assert dec(B=0) == C.MHA_ERR_INVALID
    assert dec(causal=2) == C.MHA_ERR_INVALID
    assert dec(Nq=301) == C.MHA_ERR_INVALID            # more queries than cache slots
    assert dec(cl=None) == C.MHA_ERR_INVALID
    assert dec(Nq=17) == C.MHA_ERR_UNSUPPORTED
    assert dec(dk=32) == C.MHA_ERR_UNSUPPORTED
    assert dec(ws=None) == C.MHA_ERR_WORKSPACE
    assert dec(ws_bytes=64) == C.MHA_ERR_WORKSPACE
    assert dec(Q=ODD) == C.MHA_ERR_ALIGN
    assert dec(cl=ctypes.c_void_p(0x10002)) == C.MHA_ERR_ALIGN


def test_sdpa_backward_validation(lib):
    n = ctypes.c_size_t(0)
    assert lib.mha_sdpa_bwd_workspace_size(8, 16, 4096, 1, ctypes.byref(n)) == 0
    # per 128-row tile: lse and D (1 KB), the dK/dV kernel's extra-K-step operand (8 KB),
    # then the fp32 dQ accumulator's 128 x 64 values
    assert n.value == 8 * 16 * 32 * (1024 + 8192 + 128 * 64 * 4)
    assert lib.mha_sdpa_bwd_workspace_size(8, 16, 4096, 0, ctypes.byref(n)) == 0
    assert n.value == 8 * 16 * 4096 * 4            # fp32 path: D per row
    assert lib.mha_sdpa_bwd_workspace_size(0, 16, 4096, 1, ctypes.byref(n)) == C.MHA_ERR_INVALID

    def bwd(**kw):
        a = dict(B=1, H=2, Nq=200, Nk=200, dk=64, dv=64, dt=1, mask=0, kl=None, lse=FAKE,
                 dQ=FAKE, ws=FAKE, ws_bytes=1 << 20)
        a.update(kw)
        return lib.mha_sdpa_bwd(a["B"], a["H"], a["Nq"], a["Nk"], a["dk"], a["dv"], a["dt"],
                                a["mask"], a["kl"], 0.0, FAKE, FAKE, FAKE, FAKE, FAKE, a["lse"],
                                a["dQ"], FAKE, FAKE, None, a["ws"], a["ws_bytes"], None)

    assert bwd(B=0) == C.MHA_ERR_INVALID
    assert bwd(mask=3) == C.MHA_ERR_INVALID
    assert bwd(mask=1, Nk=300) == C.MHA_ERR_INVALID     # causal needs Nq == Nk
    assert bwd(mask=2) == C.MHA_ERR_INVALID             # key padding needs key_len
    assert bwd(lse=None) == C.MHA_ERR_INVALID
    assert bwd(dQ=None) == C.MHA_ERR_INVALID
    assert bwd(dk=32) == C.MHA_ERR_UNSUPPORTED
    assert bwd(ws=None) == C.MHA_ERR_WORKSPACE
    assert bwd(ws_bytes=16) == C.MHA_ERR_WORKSPACE
    assert bwd(dQ=ODD) == C.MHA_ERR_ALIGN
    assert bwd(lse=ctypes.c_void_p(0x10002)) == C.MHA_ERR_ALIGN
    f = lib.mha_sdpa_fwd_lse
    assert f(1, 1, 8, 8, 64, 64, 1, 0, None, 0.0, FAKE, FAKE, FAKE, FAKE, None, None, None) == \
        C.MHA_ERR_INVALID
    assert f(1, 1, 8, 8, 64, 64, 1, 0, None, 0.0, FAKE, FAKE, FAKE, FAKE, None,
             ctypes.c_void_p(0x10002), None) == C.MHA_ERR_ALIGN


def test_deterministic_switch(lib):
    before = lib.mha_get_deterministic()
    try:
        assert lib.mha_set_deterministic(1) == C.MHA_OK and lib.mha_get_deterministic() == 1
        assert lib.mha_set_deterministic(0) == C.MHA_OK and lib.mha_get_deterministic() == 0
        assert lib.mha_set_deterministic(2) == C.MHA_ERR_INVALID
        assert lib.mha_set_deterministic(-1) == C.MHA_ERR_INVALID
        assert lib.mha_get_deterministic() == 0
    finally:
        lib.mha_set_deterministic(before)


def test_layer_backward_validation(lib):
    n = ctypes.c_size_t(0)
    assert lib.mha_layer_bwd_workspace_size(2, 2, 100, 100, 128, 64, 64, 1, 1,
                                            ctypes.byref(n)) == 0
    self_bytes = n.value
    assert lib.mha_layer_bwd_workspace_size(2, 2, 100, 100, 128, 64, 64, 1, 0,
                                            ctypes.byref(n)) == 0
    assert n.value > 0
    # cross-attention keeps separate key/value buffers (fp32: no split-K scratch, whose size
    # follows the largest weight gradient and is smaller for cross-attention)
    assert lib.mha_layer_bwd_workspace_size(2, 2, 100, 100, 128, 64, 64, 0, 1,
                                            ctypes.byref(n)) == 0
    self_f32 = n.value
    assert lib.mha_layer_bwd_workspace_size(2, 2, 100, 100, 128, 64, 64, 0, 0,
                                            ctypes.byref(n)) == 0
    assert n.value > self_f32
    assert self_bytes > 0
    assert lib.mha_layer_bwd_workspace_size(2, 2, 100, 90, 128, 64, 64, 1, 1,
                                            ctypes.byref(n)) == C.MHA_ERR_INVALID
    assert lib.mha_layer_bwd_workspace_size(2, 2, 100, 100, 96, 64, 64, 1, 1,
                                            ctypes.byref(n)) == C.MHA_ERR_UNSUPPORTED

    def bwd(**kw):
        a = dict(B=2, H=2, Nq=100, Nk=100, D=128, dk=64, dv=64, dt=1, mask=0, kl=None, eps=1e-5,
                 x_kv=None, dy=FAKE, dx_q=FAKE, dx_kv=None, dW_qkv=FAKE, dgamma=FAKE,
                 ws=FAKE, ws_bytes=self_bytes)
        a.update(kw)
        return lib.mha_layer_bwd(a["B"], a["H"], a["Nq"], a["Nk"], a["D"], a["dk"], a["dv"],
                                 a["dt"], a["mask"], a["kl"], a["eps"], FAKE, a["x_kv"], FAKE,
                                 None, FAKE, None, None, None, a["dy"], a["dx_q"], a["dx_kv"],
                                 a["dW_qkv"], FAKE, FAKE, FAKE, a["dgamma"], FAKE, a["ws"],
                                 a["ws_bytes"], None)

    assert bwd(B=0) == C.MHA_ERR_INVALID
    assert bwd(mask=3) == C.MHA_ERR_INVALID              # no window mask in the sublayer
    assert bwd(Nk=90) == C.MHA_ERR_INVALID               # self-attention needs Nq == Nk
    assert bwd(mask=2) == C.MHA_ERR_INVALID              # key padding needs key_len
    assert bwd(dy=None) == C.MHA_ERR_INVALID
    assert bwd(dW_qkv=None) == C.MHA_ERR_INVALID
    assert bwd(dgamma=None) == C.MHA_ERR_INVALID
    assert bwd(x_kv=FAKE, Nk=90) == C.MHA_ERR_INVALID     # cross-attention needs dx_kv
    assert bwd(eps=-1.0) == C.MHA_ERR_INVALID
    assert bwd(D=96) == C.MHA_ERR_UNSUPPORTED
    assert bwd(ws=None) == C.MHA_ERR_WORKSPACE
    assert bwd(ws_bytes=self_bytes - 1) == C.MHA_ERR_WORKSPACE
    assert bwd(dx_q=ODD) == C.MHA_ERR_ALIGN
    assert bwd(ws=ctypes.c_void_p(0x10010)) == C.MHA_ERR_ALIGN


def test_layer_training_split_validation(lib):
    n = ctypes.c_size_t(0)
    assert lib.mha_layer_bwd_workspace_size(2, 2, 100, 100, 128, 64, 64, 1, 1,
                                            ctypes.byref(n)) == 0
    need = n.value

    def fwd(**kw):
        a = dict(y=FAKE, ws=FAKE, ws_bytes=need, x_q=FAKE, D=128)
        a.update(kw)
        return lib.mha_layer_fwd_train(2, 2, 100, 100, a["D"], 64, 64, 1, 0, None, 1e-5,
                                       a["x_q"], None, FAKE, None, FAKE, None, None, None,
                                       a["y"], a["ws"], a["ws_bytes"], None)

    def bwd(**kw):
        a = dict(dy=FAKE, ws=FAKE, ws_bytes=need)
        a.update(kw)
        return lib.mha_layer_bwd_saved(2, 2, 100, 100, 128, 64, 64, 1, 0, None, 1e-5, FAKE,
                                       None, FAKE, None, FAKE, None, None, None, a["dy"], FAKE,
                                       None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, a["ws"],
                                       a["ws_bytes"], None)

    assert fwd(y=None) == C.MHA_ERR_INVALID
    assert fwd(x_q=None) == C.MHA_ERR_INVALID
    assert fwd(D=96) == C.MHA_ERR_UNSUPPORTED
    assert fwd(ws_bytes=need - 1) == C.MHA_ERR_WORKSPACE   # the backward's workspace size
    assert fwd(ws=None) == C.MHA_ERR_WORKSPACE
    assert fwd(y=ODD) == C.MHA_ERR_ALIGN
    assert bwd(dy=None) == C.MHA_ERR_INVALID
    assert bwd(ws_bytes=need - 1) == C.MHA_ERR_WORKSPACE
    assert bwd(dy=ODD) == C.MHA_ERR_ALIGN


def out_proj_ln(lib, M=4, D=256, K=256, dt=1, eps=1e-5, c=FAKE, w=FAKE, b=None, x=FAKE, y=FAKE):
    return lib.mha_out_proj_layernorm_fwd(M, D, K, dt, eps, c, w, b, x, None, None, y, None)


@pytest.mark.parametrize("kw,code", [
    (dict(M=0), C.MHA_ERR_INVALID),
    (dict(K=-1), C.MHA_ERR_INVALID),
    (dict(dt=5), C.MHA_ERR_INVALID),
    (dict(c=None), C.MHA_ERR_INVALID),
    (dict(x=None), C.MHA_ERR_INVALID),
    (dict(eps=float("nan")), C.MHA_ERR_INVALID),
    (dict(D=2304), C.MHA_ERR_UNSUPPORTED),          # wider than 2048
    (dict(D=100, dt=0), C.MHA_ERR_UNSUPPORTED),      # not a multiple of 8
    (dict(K=96), C.MHA_ERR_UNSUPPORTED),             # bf16 K multiple of 64
    (dict(b=ODD), C.MHA_ERR_ALIGN),
])
def test_out_proj_layernorm_validation(lib, kw, code):
    assert out_proj_ln(lib, **kw) == code


def layer_host(lib, B=2, H=8, N=16, D=512, dt=1, mask=0, x=FAKE, y=FAKE, chunks=2, ws=FAKE,
               ws_bytes=1 << 30, W_qkv=FAKE, W_o=FAKE):
    return lib.mha_layer_fwd_host(B, H, N, D, 64, 64, dt, mask, None, 1e-5, x, W_qkv, None,
                                  W_o, None, None, None, y, chunks, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=None), C.MHA_ERR_INVALID),
    (dict(y=None), C.MHA_ERR_INVALID),
    (dict(chunks=0), C.MHA_ERR_INVALID),
    (dict(B=0), C.MHA_ERR_INVALID),
    (dict(mask=2), C.MHA_ERR_INVALID),            # key padding needs key_len
    (dict(W_o=None), C.MHA_ERR_INVALID),
    (dict(D=520), C.MHA_ERR_UNSUPPORTED),
    (dict(ws=None), C.MHA_ERR_WORKSPACE),
    (dict(ws_bytes=1024), C.MHA_ERR_WORKSPACE),
    (dict(ws=ctypes.c_void_p(0x10010)), C.MHA_ERR_ALIGN),   # 16- but not 256-byte aligned
])
def test_layer_host_validation(lib, kw, code):
    assert layer_host(lib, **kw) == code


def test_layer_host_workspace_size(lib):
    n = ctypes.c_size_t(0)
    # 8 sequences in 3 slices of 3: four slice buffers of 3 x 4096 x 1024 bf16 + the layer
    # workspace of 3 sequences
    assert lib.mha_layer_host_workspace_size(8, 16, 4096, 1024, 64, 64, 1, 3,
                                             ctypes.byref(n)) == 0
    slot = 3 * 4096 * 1024 * 2
    m = ctypes.c_size_t(0)
    assert lib.mha_layer_workspace_size(3, 16, 4096, 4096, 1024, 64, 64, 1, ctypes.byref(m)) == 0
    assert n.value == 4 * slot + m.value
    assert lib.mha_layer_host_workspace_size(8, 16, 4096, 1024, 64, 64, 1, 0,
                                             ctypes.byref(n)) == C.MHA_ERR_INVALID
