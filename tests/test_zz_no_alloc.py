"""mha_layer_fwd_noalloc: the sublayer forward for callers that cannot allocate.

Such a caller (a plugin whose host framework owns all device memory, or a path that cannot
afford cudaMalloc's device synchronisation) gets the same results as mha_layer_fwd, with the
intermediates kept in the library's built-in 48 MiB scratch area instead of a workspace it
would have to allocate.  These tests call both entry points through the C ABI on the same
inputs and compare the outputs, for two different sublayer calls in a row (the second call
finds the first call's intermediates still in the scratch area).  Both entry points run the
same kernels on the same inputs with the same workspace layout, so their outputs must agree
bit for bit; the no-alloc output is also held to the oracle at the bf16 tolerance.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from parity_util import assert_bf16_close

from transformer_head_scaled_04_gb300 import _capi as C
from transformer_head_scaled_04_gb300 import build as B

SCRATCH_BYTES = 48 << 20


def _lib():
    B.build()
    return C.load()


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_both(lib, w, inp):
    dev = torch.device("cuda", 0)
    bf = torch.bfloat16
    t = {k: (None if v is None else torch.from_numpy(v).to(dev, bf))
         for k, v in inp.items() if k != "key_len"}
    key_len = None if inp["key_len"] is None else torch.from_numpy(inp["key_len"]).to(dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    common = (w.B, w.H, w.Nq, w.Nk, w.D, w.d_k, w.d_v, C.MHA_BF16, C.MASKS[w.mask],
              _vp(key_len), 1e-5, _vp(t["x_q"]), _vp(t["x_kv"]), _vp(t["W_qkv"]),
              _vp(t["b_qkv"]), _vp(t["W_o"]), _vp(t["b_o"]), _vp(t["gamma"]), _vp(t["beta"]))
    n = ctypes.c_size_t(0)
    assert lib.mha_layer_workspace_size(w.B, w.H, w.Nq, w.Nk, w.D, w.d_k, w.d_v, C.MHA_BF16,
                                        ctypes.byref(n)) == 0
    assert n.value <= SCRATCH_BYTES
    ws = torch.empty(n.value, dtype=torch.uint8, device=dev)
    y_ws = torch.full_like(t["x_q"], float("nan"))
    y_na = torch.full_like(t["x_q"], float("nan"))
    assert lib.mha_layer_fwd(*common, _vp(y_ws), _vp(ws), n.value, stream) == 0
    assert lib.mha_layer_fwd_noalloc(*common, _vp(y_na), stream) == 0
    torch.cuda.synchronize(dev)
    return y_ws.float().cpu().numpy(), y_na.float().cpu().numpy()


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    lib = _lib()
    torch.cuda.set_device(0)
    stream = ctypes.c_void_p(torch.cuda.current_stream(0).cuda_stream)
    assert lib.mha_debug_last_device_status(stream) in (0, C.MHA_ERR_DEVICE_TIMEOUT)
    calls = [si.WORKLOADS["dec_causal_base_b32_n256"],
             si.WORKLOADS["cross_pad_base_b32_q128_k256"]]
    for w in calls:
        inp = si.draw_layer(w, affine=True)
        y_ws, y_na = _call_both(lib, w, inp)
        assert np.all(np.isfinite(y_na))
        # identical kernels, inputs and workspace layout: bitwise equal, so a stale or
        # unwritten scratch region read by the no-alloc call cannot hide inside a tolerance
        assert np.array_equal(y_na, y_ws), f"no-alloc vs workspace entry point, {w.name}: " \
            f"{int((y_na != y_ws).sum())} elements differ"
        ref = oracle.mha_layer_ref(inp["x_q"], inp["x_kv"], inp["W_qkv"], inp["b_qkv"],
                                   inp["W_o"], inp["b_o"], inp["gamma"], inp["beta"], H=w.H,
                                   mask=w.mask, key_len=inp["key_len"], eps=1e-5)
        assert_bf16_close(y_na, ref, f"no-alloc entry point vs oracle, {w.name}")
    assert lib.mha_debug_last_device_status(stream) == 0


@pytest.mark.gpu
def test_noalloc_allocates_nothing_after_set_up():
    lib = _lib()
    torch.cuda.set_device(0)
    w = si.WORKLOADS["enc_self_base_b32_n128"]
    inp = si.draw_layer(w)
    _call_both(lib, w, inp)  # first call on this device: address look-up done
    dev = torch.device("cuda", 0)
    t = {k: (None if v is None else torch.from_numpy(v).to(dev, torch.bfloat16))
         for k, v in inp.items() if k != "key_len"}
    y = torch.empty_like(t["x_q"])
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    # Free device memory is a device-wide reading: another process on the same GPU can move
    # it between two readings.  So take up to five before/after pairs and require one in
    # which it did not change.
    pairs = []
    for _ in range(5):
        torch.cuda.synchronize(dev)
        free0, _ = torch.cuda.mem_get_info(dev)
        for _ in range(3):
            assert lib.mha_layer_fwd_noalloc(
                w.B, w.H, w.Nq, w.Nk, w.D, w.d_k, w.d_v, C.MHA_BF16, C.MASKS[w.mask], None,
                1e-5, _vp(t["x_q"]), None, _vp(t["W_qkv"]), _vp(t["b_qkv"]), _vp(t["W_o"]),
                _vp(t["b_o"]), _vp(t["gamma"]), _vp(t["beta"]), _vp(y), stream) == 0
        torch.cuda.synchronize(dev)
        free1, _ = torch.cuda.mem_get_info(dev)
        pairs.append((free0, free1))
        if free1 == free0:
            break
    assert any(a == b for a, b in pairs), f"free device memory changed on every try: {pairs}"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = _lib()
    fake = ctypes.c_void_p(0x10000)  # never touched: the size check fails first
    # big-model long sequence needs 320 MiB of intermediates > 48 MiB
    st = lib.mha_layer_fwd_noalloc(8, 16, 4096, 4096, 1024, 64, 64, C.MHA_BF16, 0, None, 1e-5,
                                   fake, None, fake, None, fake, None, None, None, fake, None)
    assert st == C.MHA_ERR_WORKSPACE
    st = lib.mha_layer_fwd_noalloc(0, 16, 4096, 4096, 1024, 64, 64, C.MHA_BF16, 0, None, 1e-5,
                                   fake, None, fake, None, fake, None, None, None, fake, None)
    assert st == C.MHA_ERR_INVALID


FAKE = ctypes.c_void_p(0x10000)   # never dereferenced: every case fails a check first
ODD = ctypes.c_void_p(0x10002)


@pytest.mark.parametrize("kw", [
    dict(B=0), dict(Nk=32), dict(mask=2), dict(W_o=None), dict(eps=-1.0), dict(D=520),
    dict(x_q=ODD), dict(B=8, H=16, Nq=4096, Nk=4096, D=1024),
])
def test_noalloc_returns_the_codes_of_the_workspace_entry_point(kw):
    """Without a GPU call: every argument error comes back as mha_layer_fwd reports it with a
    48 MiB workspace (the last case is too big for the built-in scratch)."""
    lib = _lib()
    a = dict(B=2, H=8, Nq=16, Nk=16, D=512, mask=0, eps=1e-5, x_q=FAKE, W_o=FAKE)
    a.update(kw)
    args = (a["B"], a["H"], a["Nq"], a["Nk"], a["D"], 64, 64, C.MHA_BF16, a["mask"], None,
            a["eps"], a["x_q"], None, FAKE, None, a["W_o"], None, None, None, FAKE)
    st_ws = lib.mha_layer_fwd(*args, FAKE, SCRATCH_BYTES, None)
    st_na = lib.mha_layer_fwd_noalloc(*args, None)
    assert st_ws != C.MHA_OK and st_na == st_ws


def test_noalloc_reports_the_device_error_of_the_workspace_entry_point():
    """Valid arguments on a machine with no usable CUDA device: the device check comes before
    the scratch symbol is touched, so both entry points report the same device error."""
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: valid arguments with placeholder pointers would launch")
    lib = _lib()
    args = (2, 8, 16, 16, 512, 64, 64, C.MHA_BF16, 0, None, 1e-5, FAKE, None, FAKE, None, FAKE,
            None, None, None, FAKE)
    st_ws = lib.mha_layer_fwd(*args, FAKE, SCRATCH_BYTES, None)
    st_na = lib.mha_layer_fwd_noalloc(*args, None)
    assert st_ws in (C.MHA_ERR_CUDA, C.MHA_ERR_UNSUPPORTED)
    assert st_na == st_ws
