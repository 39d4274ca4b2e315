"""Thin Python binding of libmsa's C ABI (argument marshalling only).

Every step of the path runs in the CUDA kernels of libmsa.so; this module
checks dtypes / shapes / devices, passes ``data_ptr()`` and the current CUDA
stream, and turns a non-OK status into an exception.  There is no fallback:
if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmsa.so")
_lib = None

MSA_KV_BF16, MSA_KV_FP8_E4M3, MSA_KV_NVFP4 = 0, 1, 2
KV_DTYPES = {"bf16": MSA_KV_BF16, "fp8_e4m3": MSA_KV_FP8_E4M3, "nvfp4": MSA_KV_NVFP4}
MSA_MODE_DECODE, MSA_MODE_PREFILL = 0, 1
STATUS = {0: "MSA_OK", 1: "MSA_ERR_INVALID_ARG", 2: "MSA_ERR_UNSUPPORTED",
          3: "MSA_ERR_CUDA", 4: "MSA_ERR_DEVICE_FLAG"}
DEVERR_BITS = {1: "PAGE_RANGE", 2: "SEQ_LEN", 4: "SLOT_ALIGN", 8: "TIMEOUT", 16: "FP16_RANGE"}


class MsaError(RuntimeError):
    def __init__(self, fn: str, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)} {detail}".strip())


class MsaConfig(ctypes.Structure):
    """Mirror of ``msa_config`` in include/msa.h (field order matters)."""
    _fields_ = [
        ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("init_blocks", ctypes.c_int32), ("local_blocks", ctypes.c_int32),
        ("topk_blocks", ctypes.c_int32), ("index_dim", ctypes.c_int32),
        ("q_len", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float), ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float), ("max_batch", ctypes.c_int32),
        ("max_q_tokens", ctypes.c_int32), ("max_blocks_per_req", ctypes.c_int32),
        ("num_pages", ctypes.c_int32), ("blocks_per_split", ctypes.c_int32),
        ("mode", ctypes.c_int32),
    ]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


_P = ctypes.c_void_p
_CFG = ctypes.POINTER(MsaConfig)
_SIGNATURES = {
    "msa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "msa_init_blocks_from_tokens": (ctypes.c_int32, [ctypes.c_int32, ctypes.c_int32]),
    "msa_local_blocks_from_tokens": (ctypes.c_int32, [ctypes.c_int32, ctypes.c_int32]),
    "msa_noalloc_check_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32), _P]),
    "msa_validate_config": (ctypes.c_int, [_CFG]),
    "msa_selected_width": (ctypes.c_int32, [_CFG]),
    "msa_num_splits": (ctypes.c_int32, [_CFG]),
    "msa_workspace_bytes": (ctypes.c_size_t, [_CFG]),
    "msa_plan": (ctypes.c_int, [_CFG, ctypes.c_int32, _P, _P, _P, ctypes.c_int32, _P, _P]),
    "msa_plan_from_req_to_token": (ctypes.c_int, [_CFG, ctypes.c_int32, _P, _P, _P,
                                                  ctypes.c_int32, _P, _P, _P]),
    "msa_index_score": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P]),
    "msa_cache_write": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "msa_index_attention_scratch_bytes": (ctypes.c_size_t, [_CFG]),
    "msa_index_attention": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P]),
    "msa_topk_select": (ctypes.c_int, [_CFG, _P, _P, _P, _P]),
    "msa_index_score_topk": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P]),
    "msa_sparse_decode": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P]),
    "msa_combine": (ctypes.c_int, [_CFG, _P, _P, _P, _P]),
    "msa_compact_selected": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P]),
    "msa_paged_decode": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P]),
    "msa_check_device_error": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_int32), _P]),
    "msa_selftest_wait_timeout": (ctypes.c_int, [_CFG, _P, _P]),
    "msa_sparse_decode_noalloc": (ctypes.c_int, [_CFG, ctypes.c_int32, _P, _P, ctypes.c_int32,
                                                 _P, _P, _P, _P, _P, _P, _P]),
    "msa_decode_step": (ctypes.c_int, [_CFG, _P, ctypes.c_int32, _P, _P, ctypes.c_int32, _P, _P,
                                       _P, _P, _P, _P, _P, _P, _P, _P]),
    "msa_k2q_rows": (ctypes.c_int64, [_CFG]),
    "msa_k2q_capacity": (ctypes.c_int64, [_CFG]),
    "msa_build_k2q_csr": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P]),
    "msa_sparse_prefill": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _P, _P, _P]),
}
NOALLOC_SCRATCH_BYTES = 16 << 20


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """Load libmsa.so once; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with block_sparse_paged_msa_gb300.build.build()")
        L = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def _check(fn: str, status: int, detail: str = ""):
    if status != 0:
        raise MsaError(fn, status, detail)


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype=None, dim=None, rows=None, tail=None):
    """dtype / rank / contiguity, at least `rows` entries on dim 0, and the
    trailing dims equal to `tail` (None entries are not checked)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dims, has {t.dim()}")
    if rows is not None and t.shape[0] < rows:
        raise ValueError(f"{name} has {t.shape[0]} rows on dim 0, the config needs {rows}")
    if tail is not None:
        got = tuple(t.shape[t.dim() - len(tail):])
        if any(w is not None and g != w for g, w in zip(got, tail)):
            raise ValueError(f"{name} has trailing dims {got}, the config needs {tuple(tail)}")


def _kv_dtypes(cfg):
    if cfg.kv_dtype == MSA_KV_BF16:
        return (torch.bfloat16,)
    if cfg.kv_dtype == MSA_KV_FP8_E4M3:
        return (torch.float8_e4m3fn, torch.uint8)
    return (torch.uint8,)


def max_tokens(cfg) -> int:
    """Largest number of query tokens a step of `cfg` may hold."""
    return cfg.max_q_tokens or cfg.max_batch * cfg.q_len


def _need_pools(cfg, k_pages=None, v_pages=None, idx_k_pages=None):
    """The pools must hold cfg.num_pages pages of [H_kv, 128, D | d]: the
    kernels' TMA maps and page checks are built from cfg.num_pages."""
    shape = (cfg.num_kv_heads, cfg.block_size, cfg.head_dim)
    if cfg.kv_dtype == MSA_KV_NVFP4:    # K and V slots per head, 72-byte rows
        shape = (2 * cfg.num_kv_heads, cfg.block_size, cfg.head_dim // 2 + cfg.head_dim // 16)
    if k_pages is not None:
        _need(k_pages, "k_pages", _kv_dtypes(cfg), 4, cfg.num_pages, shape)
    if v_pages is not None:
        _need(v_pages, "v_pages", _kv_dtypes(cfg), 4, cfg.num_pages, shape)
    if idx_k_pages is not None:
        _need(idx_k_pages, "idx_k_pages", torch.bfloat16, 4, cfg.num_pages,
              (cfg.num_kv_heads, cfg.block_size, cfg.index_dim))


def _need_batch(cfg, seq_lens, block_table=None, cu_seqlens_q=None):
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B = seq_lens.shape[0]
    if B > cfg.max_batch:
        raise ValueError(f"batch {B} exceeds max_batch {cfg.max_batch}")
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, 2, B, (cfg.max_blocks_per_req,))
    if cu_seqlens_q is not None:
        _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1, B + 1)
    return B


# ---------------------------------------------------------------- config
def local_blocks_from_tokens(local_tokens: int, block_size: int = 128) -> int:
    """sglang MiniMaxSparseAttnBackend.__init__: sparse_local_tokens -> blocks
    (resolved by libmsa, msa_local_blocks_from_tokens)."""
    n = lib().msa_local_blocks_from_tokens(local_tokens, block_size)
    if n < 0:
        raise ValueError(f"local_tokens {local_tokens}, block_size {block_size}")
    return n


def init_blocks_from_tokens(init_tokens: int, block_size: int = 128) -> int:
    """sglang MiniMaxSparseAttnBackend.__init__: sparse_init_tokens -> blocks
    (resolved by libmsa, msa_init_blocks_from_tokens)."""
    n = lib().msa_init_blocks_from_tokens(init_tokens, block_size)
    if n < 0:
        raise ValueError(f"init_tokens {init_tokens}, block_size {block_size}")
    return n


def make_config(*, num_q_heads, num_kv_heads, init_blocks, local_blocks, topk_blocks,
                index_dim, max_batch, max_blocks_per_req, num_pages, q_len=1,
                kv_dtype="bf16", softmax_scale=None, k_scale=1.0, v_scale=1.0,
                max_q_tokens=0, blocks_per_split=0, head_dim=128,
                block_size=128, mode="decode") -> MsaConfig:
    c = MsaConfig()
    c.num_q_heads, c.num_kv_heads = num_q_heads, num_kv_heads
    c.head_dim, c.block_size = head_dim, block_size
    c.init_blocks, c.local_blocks, c.topk_blocks = init_blocks, local_blocks, topk_blocks
    c.index_dim, c.q_len = index_dim, q_len
    c.kv_dtype = KV_DTYPES[kv_dtype]
    c.softmax_scale = 1.0 / math.sqrt(head_dim) if softmax_scale is None else softmax_scale
    c.k_scale, c.v_scale = k_scale, v_scale
    c.max_batch, c.max_q_tokens = max_batch, max_q_tokens
    c.max_blocks_per_req, c.num_pages = max_blocks_per_req, num_pages
    c.blocks_per_split = blocks_per_split
    c.mode = {"decode": MSA_MODE_DECODE, "prefill": MSA_MODE_PREFILL}[mode]
    return c


def config_for(spec, **overrides) -> MsaConfig:
    """Config of a WorkloadSpec (block counts resolved here, by the library).
    Chunks of more than 4 query tokens per request run in prefill mode."""
    prefill = spec.q_len > 4
    kw = dict(num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
              init_blocks=spec.init_blocks,
              local_blocks=local_blocks_from_tokens(spec.local_tokens, spec.block_size),
              topk_blocks=spec.topk_blocks, index_dim=spec.index_dim,
              max_batch=spec.batch, max_blocks_per_req=spec.max_blocks,
              num_pages=spec.num_pages, q_len=1 if prefill else spec.q_len,
              kv_dtype=spec.kv_dtype, mode="prefill" if prefill else "decode",
              max_q_tokens=spec.batch * spec.q_len if prefill else 0,
              softmax_scale=spec.softmax_scale, k_scale=spec.kv_scale,
              v_scale=spec.kv_scale, head_dim=spec.head_dim, block_size=spec.block_size)
    kw.update(overrides)
    return make_config(**kw)


def validate_config(cfg: MsaConfig) -> int:
    return lib().msa_validate_config(ctypes.byref(cfg))


def workspace_bytes(cfg: MsaConfig) -> int:
    n = lib().msa_workspace_bytes(ctypes.byref(cfg))
    if n == 0:
        _check("msa_workspace_bytes", validate_config(cfg) or 1)
    return n


def selected_width(cfg: MsaConfig) -> int:
    return lib().msa_selected_width(ctypes.byref(cfg))


def num_splits(cfg: MsaConfig) -> int:
    return lib().msa_num_splits(ctypes.byref(cfg))


def status_string(status: int) -> str:
    return lib().msa_status_string(status).decode()


# ---------------------------------------------------------------- calls
# Every wrapper checks the tensors against the config before the C ABI sees a
# pointer: dtypes, contiguity, trailing dims, and enough rows for what the
# kernels may touch.  Calls that take the step's batch check against that
# batch; calls that only take the workspace (whose plan may describe any step
# up to the config's maxima) check against max_tokens(cfg).
_SIZES = {}


def _sizes(cfg):
    """(workspace bytes, selected width, CSR rows, CSR capacity) of a config,
    asked of the library once per distinct config."""
    key = bytes(cfg)
    v = _SIZES.get(key)
    if v is None:
        v = (workspace_bytes(cfg), selected_width(cfg), k2q_rows(cfg), k2q_capacity(cfg))
        _SIZES[key] = v
    return v


def _need_ws(cfg, ws):
    _need(ws, "ws", torch.uint8)
    n = _sizes(cfg)[0]
    if ws.numel() < n:
        raise ValueError(f"ws has {ws.numel()} bytes, the config needs {n}")


def _need_block_table(cfg, block_table, B):
    _need(block_table, "block_table", torch.int32, 2, B)
    if block_table.shape[1] < cfg.max_blocks_per_req:
        raise ValueError(f"block_table has {block_table.shape[1]} columns, the config needs "
                         f"{cfg.max_blocks_per_req}")


def _need_tokens(cfg, T, *, q=None, idx_q=None, block_scores=None, selected=None, out=None,
                 lse=None):
    if q is not None:
        _need(q, "q", torch.bfloat16, 3, T, (cfg.num_q_heads, cfg.head_dim))
    if idx_q is not None:
        _need(idx_q, "idx_q", torch.bfloat16, 3, T, (cfg.num_kv_heads, cfg.index_dim))
    if block_scores is not None:
        _need(block_scores, "block_scores", torch.float32, 3, T,
              (cfg.num_kv_heads, cfg.max_blocks_per_req))
    if selected is not None:
        _need(selected, "selected", torch.int32, 3, T, (cfg.num_kv_heads, _sizes(cfg)[1]))
    if out is not None:
        _need(out, "out", torch.bfloat16, 3, T, (cfg.num_q_heads, cfg.head_dim))
    if lse is not None:
        _need(lse, "lse", torch.float32, 2, T, (cfg.num_q_heads,))


def plan(cfg, seq_lens, block_table, ws, cu_seqlens_q=None, stream=None):
    B = _need_batch(cfg, seq_lens, cu_seqlens_q=cu_seqlens_q)
    _need_block_table(cfg, block_table, B)
    _need_ws(cfg, ws)
    _check("msa_plan", lib().msa_plan(ctypes.byref(cfg), B, _ptr(seq_lens), _ptr(cu_seqlens_q),
                                      _ptr(block_table), block_table.shape[1], _ptr(ws),
                                      _stream(stream)))


def plan_from_req_to_token(cfg, seq_lens, req_to_token, req_pool_indices, ws,
                           cu_seqlens_q=None, stream=None):
    B = _need_batch(cfg, seq_lens, cu_seqlens_q=cu_seqlens_q)
    _need(req_to_token, "req_to_token", torch.int32, 2)
    if req_to_token.shape[1] < cfg.max_blocks_per_req * cfg.block_size:
        raise ValueError("req_to_token rows are shorter than max_blocks_per_req * block_size")
    _need(req_pool_indices, "req_pool_indices", torch.int64, 1, B)
    _need_ws(cfg, ws)
    _check("msa_plan_from_req_to_token", lib().msa_plan_from_req_to_token(
        ctypes.byref(cfg), B, _ptr(seq_lens), _ptr(cu_seqlens_q),
        _ptr(req_to_token), req_to_token.shape[1], _ptr(req_pool_indices), _ptr(ws),
        _stream(stream)))


def cache_write(cfg, ws, k, v, idx_k, k_pages, v_pages, idx_k_pages, out_cache_loc=None,
                stream=None, idx_v=None, idx_v_pages=None):
    """Store the step's new K / V / index-K (and index-V) rows ([T, H_kv, D | d]
    bf16) into the pools, after plan() and before index_score()
    (msa_cache_write).  out_cache_loc: [T] int64 slots (page * 128 + row), or
    None to take each token's slot from the plan's block table and position.
    idx_k may be None; idx_v (with idx_v_pages) only for layers with the
    index-value branch."""
    _need_ws(cfg, ws)
    T = max_tokens(cfg)
    kv_shape = (cfg.num_kv_heads, cfg.head_dim)
    _need(k, "k", torch.bfloat16, 3, T, kv_shape)
    _need(v, "v", torch.bfloat16, 3, T, kv_shape)
    if idx_k is not None:
        _need(idx_k, "idx_k", torch.bfloat16, 3, T, (cfg.num_kv_heads, cfg.index_dim))
    _need_pools(cfg, k_pages, v_pages, idx_k_pages)
    if out_cache_loc is not None:
        _need(out_cache_loc, "out_cache_loc", torch.int64, 1, T)
    if idx_v is not None:
        _need(idx_v, "idx_v", torch.bfloat16, 3, T, (cfg.num_kv_heads, cfg.index_dim))
        _need(idx_v_pages, "idx_v_pages", torch.bfloat16, 4, cfg.num_pages,
              (cfg.num_kv_heads, cfg.block_size, cfg.index_dim))
    _check("msa_cache_write", lib().msa_cache_write(
        ctypes.byref(cfg), _ptr(ws), _ptr(out_cache_loc), _ptr(k), _ptr(v), _ptr(idx_k),
        _ptr(idx_v), _ptr(k_pages), _ptr(v_pages), _ptr(idx_k_pages), _ptr(idx_v_pages),
        _stream(stream)))


def index_attention_scratch_bytes(cfg) -> int:
    return lib().msa_index_attention_scratch_bytes(ctypes.byref(cfg))


def index_attention(cfg, ws, idx_q, idx_k_pages, idx_v_pages, scratch, idx_out, idx_lse=None,
                    stream=None):
    """The index-value branch's idx_o (msa_index_attention): dense causal
    attention of the index head over every visible token (this library's
    reading; the pages name idx_o without its formula).  idx_out [T, H_kv, d]
    bf16, idx_lse [T, H_kv] float or None; scratch of
    index_attention_scratch_bytes(cfg) bytes."""
    _need_ws(cfg, ws)
    T = max_tokens(cfg)
    _need_tokens(cfg, T, idx_q=idx_q)
    _need_pools(cfg, idx_k_pages=idx_k_pages)
    _need(idx_v_pages, "idx_v_pages", torch.bfloat16, 4, cfg.num_pages,
          (cfg.num_kv_heads, cfg.block_size, cfg.index_dim))
    _need(scratch, "scratch", torch.uint8)
    n = index_attention_scratch_bytes(cfg)
    if n == 0 or scratch.numel() < n:
        raise ValueError(f"scratch has {scratch.numel()} bytes, the config needs {n}")
    _need(idx_out, "idx_out", torch.bfloat16, 3, T, (cfg.num_kv_heads, cfg.index_dim))
    if idx_lse is not None:
        _need(idx_lse, "idx_lse", torch.float32, 2, T, (cfg.num_kv_heads,))
    _check("msa_index_attention", lib().msa_index_attention(
        ctypes.byref(cfg), _ptr(ws), _ptr(idx_q), _ptr(idx_k_pages), _ptr(idx_v_pages),
        _ptr(scratch), _ptr(idx_out), _ptr(idx_lse), _stream(stream)))


def index_score(cfg, ws, idx_q, idx_k_pages, block_scores, stream=None):
    _need_ws(cfg, ws)
    T = max_tokens(cfg)
    _need_tokens(cfg, T, idx_q=idx_q, block_scores=block_scores)
    _need_pools(cfg, idx_k_pages=idx_k_pages)
    _check("msa_index_score", lib().msa_index_score(
        ctypes.byref(cfg), _ptr(ws), _ptr(idx_q), _ptr(idx_k_pages), _ptr(block_scores),
        _stream(stream)))


def decode_step(cfg, ws, seq_lens, block_table, idx_q, idx_k_pages, q, k_pages, v_pages,
                block_scores, selected, out, lse, stream=None):
    """One decode / verify step in one call (plan, index score, top-k,
    split-K decode, combine)."""
    B = _need_batch(cfg, seq_lens)
    _need_block_table(cfg, block_table, B)
    _need_ws(cfg, ws)
    T = B * cfg.q_len
    _need_tokens(cfg, T, q=q, idx_q=idx_q, block_scores=block_scores, selected=selected,
                 out=out, lse=lse)
    _need_pools(cfg, k_pages, v_pages, idx_k_pages)
    _check("msa_decode_step", lib().msa_decode_step(
        ctypes.byref(cfg), _ptr(ws), B, _ptr(seq_lens), _ptr(block_table),
        block_table.shape[1], _ptr(idx_q), _ptr(idx_k_pages), _ptr(q), _ptr(k_pages),
        _ptr(v_pages), _ptr(block_scores), _ptr(selected), _ptr(out), _ptr(lse),
        _stream(stream)))


def index_score_topk(cfg, ws, idx_q, idx_k_pages, block_scores, selected, stream=None):
    """index_score then topk_select in one call (msa_index_score_topk)."""
    _need_ws(cfg, ws)
    T = max_tokens(cfg)
    _need_tokens(cfg, T, idx_q=idx_q, block_scores=block_scores, selected=selected)
    _need_pools(cfg, idx_k_pages=idx_k_pages)
    _check("msa_index_score_topk", lib().msa_index_score_topk(
        ctypes.byref(cfg), _ptr(ws), _ptr(idx_q), _ptr(idx_k_pages), _ptr(block_scores),
        _ptr(selected), _stream(stream)))


def topk_select(cfg, ws, block_scores, selected, stream=None):
    _need_ws(cfg, ws)
    _need_tokens(cfg, max_tokens(cfg), block_scores=block_scores, selected=selected)
    _check("msa_topk_select", lib().msa_topk_select(
        ctypes.byref(cfg), _ptr(ws), _ptr(block_scores), _ptr(selected), _stream(stream)))


def sparse_decode(cfg, ws, q, k_pages, v_pages, selected, stream=None):
    _need_ws(cfg, ws)
    _need_tokens(cfg, max_tokens(cfg), q=q, selected=selected)
    _need_pools(cfg, k_pages, v_pages)
    _check("msa_sparse_decode", lib().msa_sparse_decode(
        ctypes.byref(cfg), _ptr(ws), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(selected),
        _stream(stream)))


def compact_selected(cfg, ws, selected, page_table, dense_len, stream=None):
    """Dense-sparse decode, step 1: the selected blocks of every (token, KV
    head) as a compacted page list [T, H_kv, S] and its key count [T, H_kv]
    (msa_compact_selected)."""
    _need_ws(cfg, ws)
    T = max_tokens(cfg)
    _need_tokens(cfg, T, selected=selected)
    _need(page_table, "page_table", torch.int32, 3, T, (cfg.num_kv_heads, _sizes(cfg)[1]))
    _need(dense_len, "dense_len", torch.int32, 2, T, (cfg.num_kv_heads,))
    _check("msa_compact_selected", lib().msa_compact_selected(
        ctypes.byref(cfg), _ptr(ws), _ptr(selected), _ptr(page_table), _ptr(dense_len),
        _stream(stream)))


def paged_decode(cfg, ws, q, k_pages, v_pages, page_table, dense_len, stream=None):
    """Dense-sparse decode, step 2: a dense paged decode over per-(token, KV
    head) page lists and key counts (msa_paged_decode); combine() finishes."""
    _need_ws(cfg, ws)
    T = max_tokens(cfg)
    _need_tokens(cfg, T, q=q)
    _need_pools(cfg, k_pages, v_pages)
    _need(page_table, "page_table", torch.int32, 3, T, (cfg.num_kv_heads, _sizes(cfg)[1]))
    _need(dense_len, "dense_len", torch.int32, 2, T, (cfg.num_kv_heads,))
    _check("msa_paged_decode", lib().msa_paged_decode(
        ctypes.byref(cfg), _ptr(ws), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table),
        _ptr(dense_len), _stream(stream)))


def combine(cfg, ws, out, lse, stream=None):
    _need_ws(cfg, ws)
    _need_tokens(cfg, max_tokens(cfg), out=out, lse=lse)
    _check("msa_combine", lib().msa_combine(ctypes.byref(cfg), _ptr(ws), _ptr(out), _ptr(lse),
                                            _stream(stream)))


def k2q_rows(cfg) -> int:
    return lib().msa_k2q_rows(ctypes.byref(cfg))


def k2q_capacity(cfg) -> int:
    return lib().msa_k2q_capacity(ctypes.byref(cfg))


def build_k2q_csr(cfg, ws, selected, row_ptr, q_indices, stream=None):
    _need_ws(cfg, ws)
    _need_tokens(cfg, max_tokens(cfg), selected=selected)
    _need(row_ptr, "row_ptr", torch.int32, 1, _sizes(cfg)[2] + 1)
    _need(q_indices, "q_indices", torch.int32, 1, _sizes(cfg)[3])
    _check("msa_build_k2q_csr", lib().msa_build_k2q_csr(
        ctypes.byref(cfg), _ptr(ws), _ptr(selected), _ptr(row_ptr), _ptr(q_indices),
        _stream(stream)))


def sparse_prefill(cfg, ws, q, k_pages, v_pages, selected, row_ptr, q_indices, stream=None):
    _need_ws(cfg, ws)
    _need_tokens(cfg, max_tokens(cfg), q=q, selected=selected)
    _need_pools(cfg, k_pages, v_pages)
    _need(row_ptr, "row_ptr", torch.int32, 1, _sizes(cfg)[2] + 1)
    _need(q_indices, "q_indices", torch.int32, 1, _sizes(cfg)[3])
    _check("msa_sparse_prefill", lib().msa_sparse_prefill(
        ctypes.byref(cfg), _ptr(ws), _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(selected),
        _ptr(row_ptr), _ptr(q_indices), _stream(stream)))


def check_device_error(ws, stream=None) -> int:
    """Synchronises the stream; returns the device error bits (0 = none)."""
    flags = ctypes.c_int32(0)
    st = lib().msa_check_device_error(_ptr(ws), ctypes.byref(flags), _stream(stream))
    if st not in (0, 4):
        _check("msa_check_device_error", st)
    return flags.value


def selftest_wait_timeout(cfg: MsaConfig, ws, stream=None):
    """Run the library's bounded wait on a barrier nothing completes (see
    msa_selftest_wait_timeout); the error word then holds MSA_DEVERR_TIMEOUT."""
    _need_ws(cfg, ws)
    _check("msa_selftest_wait_timeout",
           lib().msa_selftest_wait_timeout(ctypes.byref(cfg), _ptr(ws), _stream(stream)))


# ---------------------------------------------------------------- the step
class SparseAttention:
    """Owns the buffers of one configuration and runs the whole path:
    plan -> index score -> top-k select -> sparse decode -> combine."""

    def __init__(self, cfg: MsaConfig, device="cuda", dense_sparse: bool = False):
        """dense_sparse: decode through the compacted page table and the dense
        paged decode (msa_compact_selected + msa_paged_decode) instead of the
        sparse decode over the selected lists."""
        self.cfg = cfg
        self.dense_sparse = dense_sparse
        _check("msa_validate_config", validate_config(cfg))
        T = cfg.max_q_tokens or cfg.max_batch * cfg.q_len
        self.max_tokens = T
        self.width = selected_width(cfg)
        self.ws = torch.empty(workspace_bytes(cfg), dtype=torch.uint8, device=device)
        self.block_scores = torch.empty((T, cfg.num_kv_heads, cfg.max_blocks_per_req),
                                        dtype=torch.float32, device=device)
        self.selected = torch.empty((T, cfg.num_kv_heads, self.width), dtype=torch.int32,
                                    device=device)
        self.out = torch.empty((T, cfg.num_q_heads, cfg.head_dim), dtype=torch.bfloat16,
                               device=device)
        self.lse = torch.empty((T, cfg.num_q_heads), dtype=torch.float32, device=device)
        self.prefill = cfg.mode == MSA_MODE_PREFILL
        if dense_sparse:
            if self.prefill:
                raise ValueError("the dense-sparse form is a decode form")
            self.page_table = torch.empty((T, cfg.num_kv_heads, self.width), dtype=torch.int32,
                                          device=device)
            self.dense_len = torch.empty((T, cfg.num_kv_heads), dtype=torch.int32, device=device)
        if self.prefill:
            self.row_ptr = torch.empty(k2q_rows(cfg) + 1, dtype=torch.int32, device=device)
            self.q_indices = torch.empty(k2q_capacity(cfg), dtype=torch.int32, device=device)

    def run(self, seq_lens, block_table, idx_q, idx_k_pages, q, k_pages, v_pages,
            cu_seqlens_q=None, stream=None, new_kv=None, out_cache_loc=None):
        """Decode / verify: msa_decode_step (plan, index score, top-k,
        split-K decode, combine).  Prefill (cu_seqlens_q required): plan, index
        score, top-k, CSR, sparse prefill tiles, combine.  new_kv = (k, v,
        idx_k) first stores the step's new rows into the pools (cache_write,
        right after the plan; slots from out_cache_loc or from the plan)."""
        c = self.cfg
        if not self.prefill and cu_seqlens_q is None and new_kv is None and not self.dense_sparse:
            decode_step(c, self.ws, seq_lens, block_table, idx_q, idx_k_pages, q, k_pages,
                        v_pages, self.block_scores, self.selected, self.out, self.lse, stream)
            return self.out, self.lse
        plan(c, seq_lens, block_table, self.ws, cu_seqlens_q, stream)
        if new_kv is not None:
            cache_write(c, self.ws, *new_kv[:3], k_pages, v_pages, idx_k_pages, out_cache_loc,
                        stream)
        index_score_topk(c, self.ws, idx_q, idx_k_pages, self.block_scores, self.selected, stream)
        if self.prefill:
            build_k2q_csr(c, self.ws, self.selected, self.row_ptr, self.q_indices, stream)
            sparse_prefill(c, self.ws, q, k_pages, v_pages, self.selected, self.row_ptr,
                           self.q_indices, stream)
        elif self.dense_sparse:
            compact_selected(c, self.ws, self.selected, self.page_table, self.dense_len, stream)
            paged_decode(c, self.ws, q, k_pages, v_pages, self.page_table, self.dense_len, stream)
        else:
            sparse_decode(c, self.ws, q, k_pages, v_pages, self.selected, stream)
        combine(c, self.ws, self.out, self.lse, stream)
        return self.out, self.lse


def sparse_decode_noalloc(cfg, seq_lens, block_table, q, k_pages, v_pages, selected, out, lse,
                          stream=None):
    """Plan + split-K decode + combine without a workspace or any allocation,
    for callers that cannot allocate device memory (their allocator owns all
    of it, or HBM is reserved for the KV cache, or the call sits on a path
    where cudaMalloc is not acceptable).  Scratch is a fixed 16 MiB device
    array inside libmsa; steps that need more raise MsaError (UNSUPPORTED).
    The first call on a device must come before any stream capture; calls
    that overlap on the GPU share that scratch and race.  Device-side data
    errors of the last call: noalloc_check_device_error()."""
    B = _need_batch(cfg, seq_lens)
    _need_block_table(cfg, block_table, B)
    _need_tokens(cfg, B * cfg.q_len, q=q, selected=selected, out=out, lse=lse)
    _need_pools(cfg, k_pages, v_pages)
    _check("msa_sparse_decode_noalloc", lib().msa_sparse_decode_noalloc(
        ctypes.byref(cfg), B, _ptr(seq_lens), _ptr(block_table),
        block_table.shape[1], _ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(selected), _ptr(out),
        _ptr(lse), _stream(stream)),
        "(the step may need more than the 16 MiB scratch: see msa_workspace_bytes)")


def noalloc_check_device_error(stream=None) -> int:
    """Synchronises the stream; returns the device error bits the last
    sparse_decode_noalloc call on the current device recorded (0 = none)."""
    flags = ctypes.c_int32(0)
    st = lib().msa_noalloc_check_device_error(ctypes.byref(flags), _stream(stream))
    if st not in (0, 4):
        _check("msa_noalloc_check_device_error", st)
    return flags.value
