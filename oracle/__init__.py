"""CPU oracle for the multi-head attention sublayer forward pass, the position-wise
feed-forward sublayer and the encoder layer they form.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of ``__graft_entry__``
and the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (the CUDA library and its Python binding) never calls it and shares no code
with it.

Every function computes in float64 with NumPy, following the definitions on the
pages one step at a time (the backward: the chain rule through those steps).  See
``oracle.mha_ref``, ``oracle.ffn`` and ``oracle.backward`` for the citations.
"""
from .mha_ref import (  # noqa: F401
    allowed_keys,
    attention_weights_ref,
    sdpa_ref,
    linear_ref,
    layernorm_ref,
    mha_layer_ref,
    mha_layer_rows_ref,
)
from .ffn import (  # noqa: F401
    relu_ref,
    ffn_ref,
    ffn_layer_ref,
    encoder_layer_ref,
)
from .backward import (  # noqa: F401
    layernorm_bwd_ref,
    attention_bwd_ref,
    sdpa_bwd_ref,
    sdpa_lse_ref,
    mha_layer_bwd_ref,
)
