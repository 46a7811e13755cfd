"""torch-facing wrappers of the C ABI.

Argument marshalling only: torch supplies device memory (outputs and workspace are
allocated with torch when the caller does not pass them) and the current CUDA stream;
every step of the computation runs in libmha.so's kernels.  There is no CPU fallback: a
missing library raises, and so does any non-OK status.
"""
from __future__ import annotations

import ctypes

import torch

from . import _capi as C

_DTYPES = {torch.float32: C.MHA_F32, torch.bfloat16: C.MHA_BF16}


def _dt(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}; use torch.bfloat16 or torch.float32")
    return _DTYPES[t.dtype]


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")


def _stream(dev) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _mask(mask) -> int:
    if isinstance(mask, int):
        return mask
    return C.MASKS[mask]


def sdpa(q, k, v, mask="none", key_len=None, scale=None, out=None, window=None):
    """O = softmax(q k^T * scale) v per (batch, head) via ``mha_sdpa_fwd``
    (``mha_sdpa_window_fwd`` for mask="window": keys within ``window`` positions of the query).

    q [B,H,Nq,d_k], k [B,H,Nk,d_k], v [B,H,Nk,d_v] (any strides the kernel accepts);
    out [B,H,Nq,d_v] is allocated if not given and may be a strided view.
    key_len: int32 CUDA tensor [B] for mask="key_padding".
    """
    _cuda(q, k, v, key_len, out)
    B, H, Nq, d_k = q.shape
    Nk, d_v = k.shape[2], v.shape[3]
    if out is None:
        out = torch.empty((B, H, Nq, d_v), dtype=q.dtype, device=q.device)
    strides = (ctypes.c_int64 * 16)(*(list(q.stride()) + list(k.stride()) + list(v.stride())
                                      + list(out.stride())))
    if mask == "window":
        if window is None or Nq != Nk:
            raise ValueError("mask='window' needs self-attention shapes and a window radius")
        with torch.cuda.device(q.device):
            code = C.load().mha_sdpa_window_fwd(B, H, Nq, d_k, d_v, _dt(q), int(window),
                                                float(scale or 0.0), _ptr(q), _ptr(k), _ptr(v),
                                                _ptr(out), ctypes.cast(strides, ctypes.c_void_p),
                                                _stream(q.device))
        C.check(code, "mha_sdpa_window_fwd")
        return out
    with torch.cuda.device(q.device):
        code = C.load().mha_sdpa_fwd(B, H, Nq, Nk, d_k, d_v, _dt(q), _mask(mask), _ptr(key_len),
                                     float(scale or 0.0), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                     ctypes.cast(strides, ctypes.c_void_p), _stream(q.device))
    C.check(code, "mha_sdpa_fwd")
    return out


def _strides(*ts):
    return (ctypes.c_int64 * (4 * len(ts)))(*[x for t in ts for x in t.stride()])


def sdpa_with_lse(q, k, v, mask="none", key_len=None, scale=None, out=None):
    """``sdpa`` via ``mha_sdpa_fwd_lse``: returns (O, lse) with lse [B,H,Nq] fp32, the natural
    log of each row's softmax denominator (what ``sdpa_backward`` needs)."""
    _cuda(q, k, v, key_len, out)
    B, H, Nq, d_k = q.shape
    Nk, d_v = k.shape[2], v.shape[3]
    if out is None:
        out = torch.empty((B, H, Nq, d_v), dtype=q.dtype, device=q.device)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        code = C.load().mha_sdpa_fwd_lse(
            B, H, Nq, Nk, d_k, d_v, _dt(q), _mask(mask), _ptr(key_len), float(scale or 0.0),
            _ptr(q), _ptr(k), _ptr(v), _ptr(out), ctypes.cast(_strides(q, k, v, out),
                                                              ctypes.c_void_p),
            _ptr(lse), _stream(q.device))
    C.check(code, "mha_sdpa_fwd_lse")
    return out, lse


def sdpa_backward(q, k, v, o, do, lse, mask="none", key_len=None, scale=None, workspace=None):
    """dQ, dK, dV of attention via ``mha_sdpa_bwd`` (o, lse from ``sdpa_with_lse``)."""
    _cuda(q, k, v, o, do, lse, key_len, workspace)
    B, H, Nq, d_k = q.shape
    Nk, d_v = k.shape[2], v.shape[3]
    dq = torch.empty((B, H, Nq, d_k), dtype=q.dtype, device=q.device)
    dk = torch.empty((B, H, Nk, d_k), dtype=q.dtype, device=q.device)
    dv = torch.empty((B, H, Nk, d_v), dtype=q.dtype, device=q.device)
    n = ctypes.c_size_t(0)
    C.check(C.load().mha_sdpa_bwd_workspace_size(B, H, Nq, _dt(q), ctypes.byref(n)),
            "mha_sdpa_bwd_workspace_size")
    if workspace is None:
        workspace = torch.empty(n.value, dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        code = C.load().mha_sdpa_bwd(
            B, H, Nq, Nk, d_k, d_v, _dt(q), _mask(mask), _ptr(key_len), float(scale or 0.0),
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
            _ptr(dv), ctypes.cast(_strides(q, k, v, o, do, dq, dk, dv), ctypes.c_void_p),
            _ptr(workspace), workspace.numel(), _stream(q.device))
    C.check(code, "mha_sdpa_bwd")
    return dq, dk, dv


def decode_workspace_size(B, H, Nq, Lmax, dtype) -> int:
    n = ctypes.c_size_t(0)
    dt = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    C.check(C.load().mha_decode_workspace_size(B, H, Nq, Lmax, dt, ctypes.byref(n)),
            "mha_decode_workspace_size")
    return n.value


def sdpa_decode(q, k_cache, v_cache, cache_len, causal=True, scale=None, workspace=None,
                out=None):
    """One generation step against a key/value cache via ``mha_sdpa_decode_fwd``.

    q [B,H,Nq,d] (the new positions), k_cache / v_cache [B,H,Lmax,d] (any strides the kernel
    accepts), cache_len int32 CUDA tensor [B] (valid positions, the new ones included).
    causal: the queries are the newest Nq of the cached positions (bottom-right causal mask);
    otherwise every cached position j < cache_len is attended (cross-attention to Z).
    """
    _cuda(q, k_cache, v_cache, cache_len, workspace, out)
    B, H, Nq, d_k = q.shape
    Lmax, d_v = k_cache.shape[2], v_cache.shape[3]
    if out is None:
        out = torch.empty((B, H, Nq, d_v), dtype=q.dtype, device=q.device)
    ws = decode_workspace_size(B, H, Nq, Lmax, q.dtype)
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=q.device)
    strides = (ctypes.c_int64 * 16)(*(list(q.stride()) + list(k_cache.stride())
                                      + list(v_cache.stride()) + list(out.stride())))
    with torch.cuda.device(q.device):
        code = C.load().mha_sdpa_decode_fwd(
            B, H, Nq, Lmax, d_k, d_v, _dt(q), 1 if causal else 0, _ptr(cache_len),
            float(scale or 0.0), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out),
            ctypes.cast(strides, ctypes.c_void_p), _ptr(workspace), workspace.numel(),
            _stream(q.device))
    C.check(code, "mha_sdpa_decode_fwd")
    return out


def layer_workspace_size(B, H, Nq, Nk, D, d_k, d_v, dtype) -> int:
    n = ctypes.c_size_t(0)
    dt = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    C.check(C.load().mha_layer_workspace_size(B, H, Nq, Nk, D, d_k, d_v, dt, ctypes.byref(n)),
            "mha_layer_workspace_size")
    return n.value


def mha_layer(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H, mask="none", key_len=None,
              eps=1e-5, d_k=None, d_v=None, workspace=None, out=None):
    """y = LayerNorm(x_q + MultiHead(x_q, x_kv, x_kv)) via ``mha_layer_fwd``.

    x_q [B,Nq,D]; x_kv [B,Nk,D] or None (self-attention); W_qkv [H*(2d_k+d_v), D];
    W_o [D, H*d_v]; biases, gamma, beta optional.  workspace: uint8 CUDA tensor of at least
    ``layer_workspace_size(...)`` bytes (allocated here if None).
    """
    _cuda(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, key_len, workspace, out)
    B, Nq, D = x_q.shape
    Nk = Nq if x_kv is None else x_kv.shape[1]
    d_k = D // H if d_k is None else d_k
    d_v = D // H if d_v is None else d_v
    for t in (x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta):
        if t is not None and not t.is_contiguous():
            raise ValueError("mha_layer takes contiguous tensors")
    ws = layer_workspace_size(B, H, Nq, Nk, D, d_k, d_v, x_q.dtype)
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=x_q.device)
    if out is None:
        out = torch.empty_like(x_q)
    with torch.cuda.device(x_q.device):
        code = C.load().mha_layer_fwd(
            B, H, Nq, Nk, D, d_k, d_v, _dt(x_q), _mask(mask), _ptr(key_len), float(eps),
            _ptr(x_q), _ptr(x_kv), _ptr(W_qkv), _ptr(b_qkv), _ptr(W_o), _ptr(b_o), _ptr(gamma),
            _ptr(beta), _ptr(out), _ptr(workspace), workspace.numel(), _stream(x_q.device))
    C.check(code, "mha_layer_fwd")
    return out


def layer_bwd_workspace_size(B, H, Nq, Nk, D, d_k, d_v, dtype, self_attention) -> int:
    n = ctypes.c_size_t(0)
    dt = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    C.check(C.load().mha_layer_bwd_workspace_size(B, H, Nq, Nk, D, d_k, d_v, dt,
                                                  int(bool(self_attention)), ctypes.byref(n)),
            "mha_layer_bwd_workspace_size")
    return n.value


def mha_layer_forward_train(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H, mask="none",
                            key_len=None, eps=1e-5, d_k=None, d_v=None, workspace=None,
                            out=None):
    """The training forward (``mha_layer_fwd_train``): y as ``mha_layer`` computes it, with the
    activations the backward needs left in ``workspace`` (``layer_bwd_workspace_size`` bytes,
    allocated here if None).  Returns (y, workspace); pass both on to ``mha_layer_backward(...,
    workspace=workspace, saved=True)``."""
    _cuda(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, key_len, workspace, out)
    _contiguous("mha_layer_forward_train", x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta)
    B, Nq, D = x_q.shape
    Nk = Nq if x_kv is None else x_kv.shape[1]
    d_k = D // H if d_k is None else d_k
    d_v = D // H if d_v is None else d_v
    ws = layer_bwd_workspace_size(B, H, Nq, Nk, D, d_k, d_v, x_q.dtype, x_kv is None)
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=x_q.device)
    if out is None:
        out = torch.empty_like(x_q)
    with torch.cuda.device(x_q.device):
        code = C.load().mha_layer_fwd_train(
            B, H, Nq, Nk, D, d_k, d_v, _dt(x_q), _mask(mask), _ptr(key_len), float(eps),
            _ptr(x_q), _ptr(x_kv), _ptr(W_qkv), _ptr(b_qkv), _ptr(W_o), _ptr(b_o), _ptr(gamma),
            _ptr(beta), _ptr(out), _ptr(workspace), workspace.numel(), _stream(x_q.device))
    C.check(code, "mha_layer_fwd_train")
    return out, workspace


def mha_layer_backward(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, H, dy, mask="none",
                       key_len=None, eps=1e-5, d_k=None, d_v=None, workspace=None, saved=False):
    """Gradients of ``mha_layer`` with respect to every input and parameter, given dy = dL/dy,
    via ``mha_layer_bwd`` (``mha_layer_bwd_saved`` when ``saved``: the workspace then comes
    from ``mha_layer_forward_train`` with the same arguments, and the forward is not computed
    again).  Returns a dict with dx_q, dx_kv (None for self-attention), dW_qkv, db_qkv, dW_o,
    db_o, dgamma, dbeta -- each shaped like its tensor (the bias, gamma and beta gradients are
    [D] / [H*(2d_k+d_v)] even where the forward passed None).
    """
    _cuda(x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, dy, key_len, workspace)
    _contiguous("mha_layer_backward", x_q, x_kv, W_qkv, b_qkv, W_o, b_o, gamma, beta, dy)
    B, Nq, D = x_q.shape
    Nk = Nq if x_kv is None else x_kv.shape[1]
    d_k = D // H if d_k is None else d_k
    d_v = D // H if d_v is None else d_v
    if tuple(dy.shape) != (B, Nq, D):
        raise ValueError(f"dy must be [{B},{Nq},{D}]")
    ws = layer_bwd_workspace_size(B, H, Nq, Nk, D, d_k, d_v, x_q.dtype, x_kv is None)
    if saved and workspace is None:
        raise ValueError("saved=True needs the workspace mha_layer_forward_train filled")
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=x_q.device)
    e = lambda *shape: torch.empty(shape, dtype=x_q.dtype, device=x_q.device)  # noqa: E731
    g = {"dx_q": torch.empty_like(x_q),
         "dx_kv": None if x_kv is None else torch.empty_like(x_kv),
         "dW_qkv": torch.empty_like(W_qkv), "db_qkv": e(W_qkv.shape[0]),
         "dW_o": torch.empty_like(W_o), "db_o": e(D), "dgamma": e(D), "dbeta": e(D)}
    fn = C.load().mha_layer_bwd_saved if saved else C.load().mha_layer_bwd
    with torch.cuda.device(x_q.device):
        code = fn(
            B, H, Nq, Nk, D, d_k, d_v, _dt(x_q), _mask(mask), _ptr(key_len), float(eps),
            _ptr(x_q), _ptr(x_kv), _ptr(W_qkv), _ptr(b_qkv), _ptr(W_o), _ptr(b_o), _ptr(gamma),
            _ptr(beta), _ptr(dy), _ptr(g["dx_q"]), _ptr(g["dx_kv"]), _ptr(g["dW_qkv"]),
            _ptr(g["db_qkv"]), _ptr(g["dW_o"]), _ptr(g["db_o"]), _ptr(g["dgamma"]),
            _ptr(g["dbeta"]), _ptr(workspace), workspace.numel(), _stream(x_q.device))
    C.check(code, "mha_layer_bwd_saved" if saved else "mha_layer_bwd")
    return g


def linear(x, W, bias=None, out=None, relu=False):
    """Y = x W^T + bias via ``mha_linear_fwd`` (``mha_linear_relu_fwd``: max(0, .) when relu);
    x [M,K] (row pitch = x.stride(0)), W [N,K]."""
    _cuda(x, W, bias, out)
    M, K = x.shape
    N = W.shape[0]
    if W.shape[1] != K or not W.is_contiguous() or x.stride(1) != 1:
        raise ValueError("linear: x [M,K] with unit column stride and dense W [N,K] expected")
    if out is None:
        out = torch.empty((M, N), dtype=x.dtype, device=x.device)
    if tuple(out.shape) != (M, N) or out.stride(1) != 1:
        raise ValueError(f"linear: out must be [{M},{N}] with unit column stride")
    fn = C.load().mha_linear_relu_fwd if relu else C.load().mha_linear_fwd
    with torch.cuda.device(x.device):
        code = fn(M, N, K, _dt(x), _ptr(x), x.stride(0), _ptr(W), _ptr(bias), _ptr(out),
                  out.stride(0), _stream(x.device))
    C.check(code, "mha_linear_relu_fwd" if relu else "mha_linear_fwd")
    return out


def linear2(x1, W1, b1, x2, W2, b2):
    """(x1 W1^T + b1, x2 W2^T + b2) in one launch via ``mha_linear2_fwd``; dense x1 [M1,K],
    W1 [N1,K], x2 [M2,K], W2 [N2,K] (the two projections of encoder-decoder attention)."""
    _cuda(x1, W1, b1, x2, W2, b2)
    _contiguous("linear2", x1, W1, b1, x2, W2, b2)
    (M1, K), (M2, K2) = x1.shape, x2.shape
    N1, N2 = W1.shape[0], W2.shape[0]
    if K2 != K or W1.shape[1] != K or W2.shape[1] != K:
        raise ValueError("linear2: x1, W1, x2, W2 must share K")
    y1 = torch.empty((M1, N1), dtype=x1.dtype, device=x1.device)
    y2 = torch.empty((M2, N2), dtype=x1.dtype, device=x1.device)
    with torch.cuda.device(x1.device):
        code = C.load().mha_linear2_fwd(M1, N1, _ptr(x1), _ptr(W1), _ptr(b1), _ptr(y1), M2, N2,
                                        _ptr(x2), _ptr(W2), _ptr(b2), _ptr(y2), K, _dt(x1),
                                        _stream(x1.device))
    C.check(code, "mha_linear2_fwd")
    return y1, y2


def ffn_workspace_size(M, D, d_ff, dtype) -> int:
    n = ctypes.c_size_t(0)
    dt = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    C.check(C.load().mha_ffn_workspace_size(M, D, d_ff, dt, ctypes.byref(n)),
            "mha_ffn_workspace_size")
    return n.value


def _contiguous(name, *ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} takes contiguous tensors")


def ffn(x, W1, b1, W2, b2, gamma=None, beta=None, eps=1e-5, workspace=None, out=None):
    """y = LayerNorm(x + max(0, x W1^T + b1) W2^T + b2) over the last axis via ``mha_ffn_fwd``.

    x [..., D] (every row is a position); W1 [d_ff, D]; W2 [D, d_ff]; biases, gamma, beta
    optional.  workspace: uint8 CUDA tensor of at least ``ffn_workspace_size(...)`` bytes.
    """
    _cuda(x, W1, b1, W2, b2, gamma, beta, workspace, out)
    _contiguous("ffn", x, W1, b1, W2, b2, gamma, beta)
    D = x.shape[-1]
    M = x.numel() // D
    d_ff = W1.shape[0]
    if tuple(W1.shape) != (d_ff, D) or tuple(W2.shape) != (D, d_ff):
        raise ValueError(f"ffn: W1 [d_ff, {D}] and W2 [{D}, d_ff] expected")
    ws = ffn_workspace_size(M, D, d_ff, x.dtype)
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty_like(x)
    with torch.cuda.device(x.device):
        code = C.load().mha_ffn_fwd(M, D, d_ff, _dt(x), float(eps), _ptr(x), _ptr(W1), _ptr(b1),
                                    _ptr(W2), _ptr(b2), _ptr(gamma), _ptr(beta), _ptr(out),
                                    _ptr(workspace), workspace.numel(), _stream(x.device))
    C.check(code, "mha_ffn_fwd")
    return out


def encoder_layer_workspace_size(B, N, H, D, d_ff, dtype) -> int:
    n = ctypes.c_size_t(0)
    dt = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    C.check(C.load().mha_encoder_layer_workspace_size(B, N, H, D, d_ff, dt, ctypes.byref(n)),
            "mha_encoder_layer_workspace_size")
    return n.value


def encoder_layer(x, W_qkv, b_qkv, W_o, b_o, gamma1, beta1, W1, b1, W2, b2, gamma2, beta2, H,
                  mask="none", key_len=None, eps=1e-5, workspace=None, out=None):
    """One encoder layer via ``mha_encoder_layer_fwd``:
    h = LayerNorm(x + MultiHead(x, x, x)), y = LayerNorm(h + FFN(h)).  x [B,N,D]."""
    _cuda(x, W_qkv, b_qkv, W_o, b_o, gamma1, beta1, W1, b1, W2, b2, gamma2, beta2, key_len,
          workspace, out)
    _contiguous("encoder_layer", x, W_qkv, b_qkv, W_o, b_o, gamma1, beta1, W1, b1, W2, b2,
                gamma2, beta2)
    B, N, D = x.shape
    d_ff = W1.shape[0]
    ws = encoder_layer_workspace_size(B, N, H, D, d_ff, x.dtype)
    if workspace is None:
        workspace = torch.empty(ws, dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty_like(x)
    with torch.cuda.device(x.device):
        code = C.load().mha_encoder_layer_fwd(
            B, N, H, D, d_ff, _dt(x), _mask(mask), _ptr(key_len), float(eps), _ptr(x),
            _ptr(W_qkv), _ptr(b_qkv), _ptr(W_o), _ptr(b_o), _ptr(gamma1), _ptr(beta1), _ptr(W1),
            _ptr(b1), _ptr(W2), _ptr(b2), _ptr(gamma2), _ptr(beta2), _ptr(out),
            _ptr(workspace), workspace.numel(), _stream(x.device))
    C.check(code, "mha_encoder_layer_fwd")
    return out


def residual_layernorm(x, a, gamma=None, beta=None, eps=1e-5, out=None):
    """y = LayerNorm(x + a) * gamma + beta over the last axis via ``mha_residual_layernorm_fwd``."""
    _cuda(x, a, gamma, beta, out)
    D = x.shape[-1]
    M = x.numel() // D
    if out is None:
        out = torch.empty_like(x)
    with torch.cuda.device(x.device):
        code = C.load().mha_residual_layernorm_fwd(M, D, _dt(x), float(eps), _ptr(x), _ptr(a),
                                                   _ptr(gamma), _ptr(beta), _ptr(out),
                                                   _stream(x.device))
    C.check(code, "mha_residual_layernorm_fwd")
    return out


def set_deterministic(on: bool) -> None:
    """Process-wide switch of the bf16 attention backward (``mha_set_deterministic``): True
    computes dQ by its own kernel, bitwise reproducible; False (the default) adds each key
    tile's part of dQ into an fp32 accumulator, faster, reproducible up to fp32 rounding."""
    C.check(C.load().mha_set_deterministic(1 if on else 0), "mha_set_deterministic")


def get_deterministic() -> bool:
    """The current ``mha_set_deterministic`` setting."""
    return bool(C.load().mha_get_deterministic())


def device_status(stream=None) -> int:
    """First device-side error since the last call on the current device (0 = none); syncs."""
    s = _stream(torch.cuda.current_device()) if stream is None else stream
    return C.load().mha_debug_last_device_status(s)


def wait_selftest(timeout_ns: int = 1_000_000) -> int:
    """Run the bounded-wait self test and return the device status it left (expect -6)."""
    device_status()  # clear anything older
    C.check(C.load().mha_debug_wait_selftest(int(timeout_ns), _stream(torch.cuda.current_device())),
            "mha_debug_wait_selftest")
    return device_status()


def out_proj_layernorm(c, W_o, b_o, x, gamma=None, beta=None, eps=1e-5, out=None):
    """y = LayerNorm(x + c W_o^T + b_o) * gamma + beta over the last axis via
    ``mha_out_proj_layernorm_fwd`` (c [..., K], W_o [D, K], x [..., D])."""
    _cuda(c, W_o, b_o, x, gamma, beta, out)
    D, K = W_o.shape
    M = x.numel() // D
    if out is None:
        out = torch.empty_like(x)
    with torch.cuda.device(x.device):
        code = C.load().mha_out_proj_layernorm_fwd(M, D, K, _dt(x), float(eps), _ptr(c),
                                                   _ptr(W_o), _ptr(b_o), _ptr(x), _ptr(gamma),
                                                   _ptr(beta), _ptr(out), _stream(x.device))
    C.check(code, "mha_out_proj_layernorm_fwd")
    return out


def mha_layer_host(x_host, W_qkv, b_qkv, W_o, b_o, gamma, beta, H, mask="none", key_len=None,
                   eps=1e-5, chunks=4, workspace=None, out=None, device=None):
    """Self-attention sublayer on host tensors via ``mha_layer_fwd_host``: x_host [B,N,D] (CPU,
    ideally pinned), weights on the CUDA device; returns y on the host (``out``, pinned, is
    allocated if not given).  The copies in and out overlap the computation slice by slice;
    the call returns once y is complete."""
    _cuda(W_qkv, b_qkv, W_o, b_o, gamma, beta, key_len, workspace)
    if x_host.is_cuda:
        raise ValueError("x_host must be a host tensor")
    dev = W_qkv.device if device is None else device
    B, N, D = x_host.shape
    x_host = x_host.contiguous()
    if out is None:
        out = torch.empty_like(x_host).pin_memory()
    dt = _dt(x_host)
    lib = C.load()
    if workspace is None:
        n = ctypes.c_size_t(0)
        C.check(lib.mha_layer_host_workspace_size(B, H, N, D, D // H, D // H, dt, chunks,
                                                  ctypes.byref(n)), "mha_layer_host_workspace_size")
        workspace = torch.empty(max(n.value, 256), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        code = lib.mha_layer_fwd_host(B, H, N, D, D // H, D // H, dt, C.MASKS[mask],
                                      _ptr(key_len), float(eps), _ptr(x_host), _ptr(W_qkv),
                                      _ptr(b_qkv), _ptr(W_o), _ptr(b_o), _ptr(gamma), _ptr(beta),
                                      _ptr(out), int(chunks), _ptr(workspace), workspace.numel(),
                                      _stream(dev))
        C.check(code, "mha_layer_fwd_host")
        torch.cuda.current_stream(dev).synchronize()
    return out
