"""Feeds a seeded Workload to the fp64 oracle (test-side glue: dtype conversion only)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from block_sparse_paged_msa_gb300.workloads import Workload


def to_np(t: torch.Tensor) -> np.ndarray:
    """Exact host copy: bf16/fp32 -> float64, e4m3 -> raw uint8 codes, ints -> int64."""
    t = t.detach().cpu()
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    if t.is_floating_point():
        return t.to(torch.float64).numpy()
    return t.to(torch.int64).numpy()


def oracle_local_blocks(w: Workload) -> int:
    return oracle.local_blocks_from_tokens(w.spec.local_tokens, w.spec.block_size)


def run_oracle(w: Workload, tokens=None, kv_heads=None, scale=None):
    s = w.spec
    return oracle.sparse_attention(
        seq_lens=to_np(w.seq_lens), q_lens=to_np(w.q_lens),
        block_table=to_np(w.block_table), idx_q=to_np(w.idx_q),
        idx_k_pages=to_np(w.idx_k_pages), q=to_np(w.q), k_pages=to_np(w.k_pages),
        v_pages=to_np(w.v_pages), num_kv_heads=s.num_kv_heads,
        block_size=s.block_size, init_blocks=s.init_blocks,
        local_blocks=oracle_local_blocks(w), topk_blocks=s.topk_blocks,
        softmax_scale=s.softmax_scale if scale is None else scale,
        k_scale=s.kv_scale, v_scale=s.kv_scale,
        kv_is_e4m3=(s.kv_dtype == "fp8_e4m3"), kv_is_nvfp4=(s.kv_dtype == "nvfp4"),
        tokens=tokens, kv_heads=kv_heads)


def selected_array(res, T, H, S) -> np.ndarray:
    """Oracle selections as the [T, H, S] int array (ascending, -1 padded)."""
    out = np.full((T, H, S), -1, dtype=np.int64)
    for (t, h), sel in res["selected"].items():
        out[t, h, :len(sel)] = sel
    return out
