"""ctypes view of libmha.so: the C ABI declared in include/mha.h, nothing more."""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmha.so")
# the same ABI with the kernels' index checks compiled in (built by build(debug_bounds=True))
DEBUG_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmha_debug.so")

# mirrors of the enums in include/mha.h
MHA_OK = 0
MHA_ERR_INVALID = -1
MHA_ERR_UNSUPPORTED = -2
MHA_ERR_ALIGN = -3
MHA_ERR_WORKSPACE = -4
MHA_ERR_CUDA = -5
MHA_ERR_DEVICE_TIMEOUT = -6
MHA_ERR_DEVICE_BOUNDS = -7
MHA_F32 = 0
MHA_BF16 = 1
MASKS = {"none": 0, "causal": 1, "key_padding": 2}

_c_int, _c_float, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
_i64, _size = ctypes.c_int64, ctypes.c_size_t

PROTOTYPES = {
    "mha_sdpa_fwd": (_c_int, [_c_int] * 8 + [_vp, _c_float, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mha_sdpa_fwd_lse": (_c_int, [_c_int] * 8 + [_vp, _c_float, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mha_sdpa_bwd_workspace_size": (_c_int, [_c_int] * 4 + [ctypes.POINTER(_size)]),
    "mha_sdpa_bwd": (_c_int, [_c_int] * 8 + [_vp, _c_float] + [_vp] * 9 + [_vp, _vp, _size, _vp]),
    "mha_sdpa_window_fwd": (_c_int, [_c_int] * 7 + [_c_float, _vp, _vp, _vp, _vp, _vp, _vp]),
    "mha_decode_workspace_size": (_c_int, [_c_int] * 5 + [ctypes.POINTER(_size)]),
    "mha_sdpa_decode_fwd": (_c_int, [_c_int] * 8 + [_vp, _c_float] + [_vp] * 5
                            + [_vp, _size, _vp]),
    "mha_layer_workspace_size": (_c_int, [_c_int] * 8 + [ctypes.POINTER(_size)]),
    "mha_layer_fwd": (_c_int, [_c_int] * 9 + [_vp, _c_float] + [_vp] * 10 + [_size, _vp]),
    "mha_layer_bwd_workspace_size": (_c_int, [_c_int] * 9 + [ctypes.POINTER(_size)]),
    "mha_layer_bwd": (_c_int, [_c_int] * 9 + [_vp, _c_float] + [_vp] * 18 + [_size, _vp]),
    "mha_layer_fwd_train": (_c_int, [_c_int] * 9 + [_vp, _c_float] + [_vp] * 10 + [_size, _vp]),
    "mha_layer_bwd_saved": (_c_int, [_c_int] * 9 + [_vp, _c_float] + [_vp] * 18 + [_size, _vp]),
    "mha_layer_fwd_timed": (_c_int, [_c_int] * 9 + [_vp, _c_float] + [_vp] * 10
                            + [_size, _vp, _vp, _c_int]),
    "mha_layer_fwd_noalloc": (_c_int, [_c_int] * 9 + [_vp, _c_float] + [_vp] * 9 + [_vp]),
    "mha_layer_host_workspace_size": (_c_int, [_c_int] * 8 + [ctypes.POINTER(_size)]),
    "mha_layer_fwd_host": (_c_int, [_c_int] * 8 + [_vp, _c_float] + [_vp] * 8 + [_c_int, _vp,
                                                                                  _size, _vp]),
    "mha_linear_fwd": (_c_int, [_c_int] * 4 + [_vp, _i64, _vp, _vp, _vp, _i64, _vp]),
    "mha_linear2_fwd": (_c_int, [_c_int] * 2 + [_vp] * 4 + [_c_int] * 2 + [_vp] * 4
                        + [_c_int] * 2 + [_vp]),
    "mha_linear_relu_fwd": (_c_int, [_c_int] * 4 + [_vp, _i64, _vp, _vp, _vp, _i64, _vp]),
    "mha_ffn_workspace_size": (_c_int, [_c_int] * 4 + [ctypes.POINTER(_size)]),
    "mha_ffn_fwd": (_c_int, [_c_int] * 4 + [_c_float] + [_vp] * 9 + [_size, _vp]),
    "mha_ffn_fwd_timed": (_c_int, [_c_int] * 4 + [_c_float] + [_vp] * 9
                          + [_size, _vp, _vp, _c_int]),
    "mha_encoder_layer_workspace_size": (_c_int, [_c_int] * 6 + [ctypes.POINTER(_size)]),
    "mha_encoder_layer_fwd": (_c_int, [_c_int] * 7 + [_vp, _c_float] + [_vp] * 15
                              + [_size, _vp]),
    "mha_residual_layernorm_fwd": (_c_int, [_c_int] * 3 + [_c_float] + [_vp] * 6),
    "mha_out_proj_layernorm_fwd": (_c_int, [_c_int] * 4 + [_c_float] + [_vp] * 8),
    "mha_status_string": (ctypes.c_char_p, [_c_int]),
    "mha_set_deterministic": (_c_int, [_c_int]),
    "mha_get_deterministic": (_c_int, []),
    "mha_debug_last_device_status": (_c_int, [_vp]),
    "mha_debug_wait_selftest": (_c_int, [_i64, _vp]),
    "mha_abi_version": (_c_int, []),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load libmha.so from this package directory (fails loudly if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "or `python -m transformer_head_scaled_04_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


_debug_lib = None


def load_debug() -> ctypes.CDLL:
    """Load libmha_debug.so, the index-checking build of the same ABI (fails loudly if it was
    never built)."""
    global _debug_lib
    if _debug_lib is None:
        if not os.path.exists(DEBUG_LIB_PATH):
            raise RuntimeError(f"{DEBUG_LIB_PATH} is missing: build it first with "
                               "`python -m transformer_head_scaled_04_gb300.build --debug-bounds`")
        lib = ctypes.CDLL(DEBUG_LIB_PATH)
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _debug_lib = lib
    return _debug_lib


def status_string(code: int) -> str:
    return load().mha_status_string(code).decode()


class MhaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


def check(code: int, where: str) -> None:
    if code != MHA_OK:
        raise MhaError(code, where)
