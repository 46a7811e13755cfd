"""GB300 (sm_103a) multi-head attention sublayer forward and backward, with the position-wise
feed-forward sublayer and the encoder layer they form: a C-ABI CUDA library (libmha.so,
declared in include/mha.h) and a thin torch binding of it.

The library itself is loaded lazily on first use; ``build.build()`` compiles it in-tree.
"""
from ._capi import (  # noqa: F401
    LIB_PATH,
    MASKS,
    MhaError,
    load as load_library,
    status_string,
)
from .api import (  # noqa: F401
    decode_workspace_size,
    device_status,
    encoder_layer,
    encoder_layer_workspace_size,
    ffn,
    ffn_workspace_size,
    get_deterministic,
    layer_bwd_workspace_size,
    layer_workspace_size,
    linear,
    linear2,
    mha_layer,
    mha_layer_backward,
    mha_layer_forward_train,
    mha_layer_host,
    out_proj_layernorm,
    residual_layernorm,
    sdpa,
    sdpa_backward,
    sdpa_decode,
    sdpa_with_lse,
    set_deterministic,
    wait_selftest,
)
