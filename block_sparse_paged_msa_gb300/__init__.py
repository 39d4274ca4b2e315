"""Block-sparse attention over a paged KV cache (MiniMax-M3 style MSA) for GB300.

The compute path is libmsa.so (hand-written CUDA for sm_103a, C ABI in
include/msa.h); ``ops`` is its thin binding and ``workloads`` draws seeded
synthetic inputs.  The library is loaded on first use and every op raises if it
is missing: there is no CPU fallback.
"""
from . import workloads  # noqa: F401
from .ops import (MsaConfig, MsaError, SparseAttention, cache_write,  # noqa: F401
                  check_device_error, compact_selected, index_attention,
                  index_attention_scratch_bytes, index_score_topk, paged_decode,
                  combine, config_for, index_score, make_config, num_splits, plan,
                  plan_from_req_to_token, selected_width, sparse_decode, topk_select,
                  workspace_bytes)
