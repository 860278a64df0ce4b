"""GB300 (sm_103a) routed mixture-of-experts FFN over block-quantized experts.

The layer runs in hand-written CUDA kernels behind a C ABI
(``include/moe_route.h``, ``libmoe_route.so``); this package is the thin
Python binding. Import is cheap: the library is loaded on first use, and a
missing library raises instead of falling back to anything else.
"""
from ._lib import (  # noqa: F401
    BLOCK_BYTES, BLOCK_ELEMS, EXPORTED, FLAG_BAD_ID, FLAG_DUPLICATE_ID, FLAG_NONFINITE_LOGIT,
    FLAG_WAIT_TIMEOUT, GEMV_STREAMING, GEMV_TILED, MOE_TABLE_PREPARED, MXFP4, PATH_AUTO, PATH_FUSED, PATH_GEMV, PATH_TENSOR, Q4_K, Q6_K, Q8_0,
    IQ4_NL, IQ4_XS, IQ3_XXS, T5_G128,
    MoeError, NOALLOC_SCRATCH_BYTES, Options, WeightTable, Workspace, bucket, ffn_forward,
    ffn_forward_noalloc, ffn_path, gemv_kernels, load, make_options, noalloc_read_status, route_topk, set_wait_timeout_ns, sum_partials,
)
from .shard import ShardedLayer, expert_shard, gather_partials  # noqa: F401
