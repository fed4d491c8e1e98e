"""GB300 (sm_103a) attention forward/backward over packed variable-length sequences.

The compute lives in ``lib/libteattn.so`` (C ABI in ``include/te_attn.h``); this
package marshals torch tensors into that ABI and nothing more. There is no CPU
path: every function raises if the library is missing or a tensor is not on a
CUDA device.

Entry points: ``fwd`` / ``bwd`` (packed THD layout, real and padded cu_seqlens),
``fwd_sbhd`` / ``bwd_sbhd`` (sequence-major ``[S, B, h, d]``), ``fwd_e4m3`` (e4m3
inputs with per-tensor descale factors, forward only), ``bwd_noalloc`` (backward
without a workspace); ``read_status`` / ``read_status_noalloc`` read a call's device
status word, ``selftest_wait_timeout`` runs the bounded-wait unwind path on purpose and
``debug_build()`` routes calls to the bounds-checking build; masks ``padding``, ``padding_causal`` (upper-left) and
``padding_causal_bottom_right``. ``dot_product_attention`` / ``DotProductAttention``
wrap them for autograd (``thd``, ``bshd``, ``sbhd``).
"""

from ._binding import (  # noqa: F401
    MASK_PADDING,
    MASK_PADDING_CAUSAL,
    MASK_PADDING_CAUSAL_BOTTOM_RIGHT,
    TeAttnError,
    bwd,
    bwd_noalloc,
    debug_build,
    fwd,
    fwd_e4m3,
    fwd_sbhd,
    bwd_sbhd,
    fwd_workspace_size,
    KERNELS,
    profile_enable,
    profile_read,
    bwd_workspace_size,
    bwd_fused_workspace_size,
    library,
    library_path,
    read_status,
    read_status_noalloc,
    selftest_wait_timeout,
    version,
)
from .autograd import (  # noqa: F401
    DotProductAttention,
    SBHDAttentionFunction,
    THDAttentionFunction,
    dot_product_attention,
)
