"""GB300 (sm_103a) attention forward/backward over packed variable-length sequences.

The compute lives in ``lib/libteattn.so`` (C ABI in ``include/te_attn.h``); this
package marshals torch tensors into that ABI and nothing more. There is no CPU
path: every function raises if the library is missing or a tensor is not on a
CUDA device.
"""

from ._binding import (  # noqa: F401
    MASK_PADDING,
    MASK_PADDING_CAUSAL,
    MASK_PADDING_CAUSAL_BOTTOM_RIGHT,
    TeAttnError,
    bwd,
    bwd_noalloc,
    fwd,
    fwd_e4m3,
    fwd_sbhd,
    bwd_sbhd,
    fwd_workspace_size,
    KERNELS,
    profile_enable,
    profile_read,
    bwd_workspace_size,
    library,
    library_path,
    read_status,
    version,
)
from .autograd import (  # noqa: F401
    DotProductAttention,
    SBHDAttentionFunction,
    THDAttentionFunction,
    dot_product_attention,
)
