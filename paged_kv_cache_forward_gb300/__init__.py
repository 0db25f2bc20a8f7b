"""libpagedattn: unified paged-attention forward for GB300 (sm_103a).

``forward`` computes softmax(Q K^T * scale) V over a paged bf16 KV cache read
through a block table, for a batch that mixes decode and causal chunked-prefill
sequences (see include/pagedattn.h for the exact contract).  The compute runs
in hand-written CUDA kernels in ``libpagedattn.so``; this package only
marshals arguments.  Build the library with ``paged_kv_cache_forward_gb300.build.build()``.
"""

from .binding import (  # noqa: F401
    DEVICE_ERRORS,
    EXPORTED,
    Dims,
    PagedAttnError,
    device_error,
    forward,
    forward_noalloc,
    cache_write,
    CacheDims,
    load,
    make_dims,
    plan,
    plan_for,
    prepare,
    release_workspaces,
    version,
)
