"""fp64 CPU oracle for block-sparse paged MSA attention.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this module.  The CUDA path never does, and this module
imports nothing from it: the two share no code.  It is plain, slow and meant to
be read against the method's description:

* MiniMax-M3 sparse attention as wired by sglang ``minimax_sparse_backend.py``
  (``MiniMaxSparseAttnBackend.__init__``: block size, init / local / top-k block
  counts and the index score type; ``forward_decode`` / ``forward_extend``: the
  cache write precedes attention, then index scoring, top-k block selection and
  attention over the selected blocks) and by vLLM
  ``minimax_m3/nvidia/sparse_attention_msa.py`` (``MiniMaxM3SparseMSAImpl.forward``:
  per-token, per-KV-head selected block lists, GQA with ``qhead_per_kv`` query
  heads per KV head, ``build_k2q_csr`` key-block-to-query lists for prefill).
* The pages leave the index score formula open (only ``score_type`` is named);
  the specification of this build fixes it: a block's score is the maximum over
  its visible tokens of ``idx_q . idx_k``, and ties go to the lower block index.

Every quantity is computed in float64 from exact copies of the inputs (bf16 and
e4m3 values are exactly representable in float64).

Notation: P = block size (= page size, 128), H_kv KV heads, G = H_q / H_kv query
heads per KV head, D head dim, d index dim.  A query token of request r with
n_q new tokens, the i-th of them, sits at position p = seq_len_r - n_q + i and
sees tokens [0, p]; it has nb = floor(p / P) + 1 visible blocks.

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against brute force, hand-computed selections, closed forms or an independent
library routine.  One READING is unpinned: ``index_attention`` (the
index-value branch) computes the textbook attention it states, but the pages
never say that idx_o is that attention -- its parity with the pages is
"parity unpinned".
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence, Tuple

import numpy as np

__all__ = [
    "init_blocks_from_tokens", "local_blocks_from_tokens", "e4m3_to_float",
    "query_positions", "gather_sequence", "block_scores", "select_blocks",
    "attention", "combine", "sparse_attention", "build_k2q_csr", "e4m3_encode",
    "cache_slots", "cache_write", "e2m1_to_float", "nvfp4_dequant", "nvfp4_row_bytes",
    "NVFP4_BLOCK", "e2m1_encode", "nvfp4_quantize", "cache_write_nvfp4", "compact_selection", "paged_attention", "index_attention",
]


# --------------------------------------------------------------------------
# Sparse configuration (sglang MiniMaxSparseAttnBackend.__init__)
# --------------------------------------------------------------------------
def init_blocks_from_tokens(init_tokens: int, block_size: int) -> int:
    """``sparse_init_tokens`` -> init block count: ceil(tokens / block)."""
    return -(-init_tokens // block_size)


def local_blocks_from_tokens(local_tokens: int, block_size: int) -> int:
    """``sparse_local_tokens`` -> local block count: ceil(tokens / block) + 1.

    The extra block is the query's own, partially filled block."""
    return -(-local_tokens // block_size) + 1


# --------------------------------------------------------------------------
# fp8 e4m3 ("fn": no infinities, one NaN per sign) decode, from the format's
# definition: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0
# is subnormal (m/8 * 2^-6); exponent 15 with mantissa 7 is NaN.  The vLLM page
# stores fp8 KV caches as raw e4m3 with per-layer float scales
# (MiniMaxM3SparseMSAImpl.forward, ``_k_scale`` / ``_v_scale``).
# --------------------------------------------------------------------------
def _e4m3_value(code: int) -> float:
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return math.nan
    if exp == 0:
        return sign * (man / 8.0) * 2.0 ** -6
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


_E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)


def e4m3_to_float(codes: np.ndarray) -> np.ndarray:
    """Decode uint8 e4m3 codes to float64."""
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


_E4M3_FINITE = _E4M3_TABLE[:0x7F]   # codes 0x00 .. 0x7E: 0 .. 448, ascending


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Float values -> e4m3fn codes (uint8), from the format's definition: the
    nearest representable value, ties to the code whose last mantissa bit is 0;
    magnitudes beyond the largest finite value (448) saturate to it, as the
    quantise-on-write of an fp8 KV cache clamps instead of making NaN; NaN ->
    0x7F.  The sign bit is kept (a negative value that rounds to zero is 0x80)."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    n = len(_E4M3_FINITE)
    hi = np.clip(np.searchsorted(_E4M3_FINITE, np.nan_to_num(mag, nan=0.0, posinf=1e9)), 0, n - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - _E4M3_FINITE[lo]
    d_hi = _E4M3_FINITE[hi] - mag
    code = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    code = np.where(tie, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(mag >= _E4M3_FINITE[-1], n - 1, code)          # saturate
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


# --------------------------------------------------------------------------
# NVFP4 KV pages (vLLM sparse_attention_msa.py, MiniMaxM3SparseMSANvfp4Backend:
# HND pages in which every KV head has two slots, its keys and its values, each
# token row holding packed FP4 data plus block scales; per-layer k / v scales).
# The format, from its definition: an element is FP4 E2M1 (1 sign bit, 2
# exponent bits with bias 1, 1 mantissa bit; exponent 0 is subnormal m * 0.5),
# two per byte, the even element in the low nibble; every 16 consecutive
# elements share one E4M3 scale.  A D = 128 row is 64 data bytes followed by
# 8 scale bytes (72 bytes).  Value = e2m1(code) * e4m3(scale) * tensor scale.
# --------------------------------------------------------------------------
def _e2m1_value(code: int) -> float:
    sign = -1.0 if code & 0x8 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:
        return sign * man * 0.5
    return sign * (1.0 + man / 2.0) * 2.0 ** (exp - 1)


_E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
NVFP4_BLOCK = 16


def e2m1_to_float(codes: np.ndarray) -> np.ndarray:
    """Decode 4-bit e2m1 codes (0..15) to float64."""
    return _E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def nvfp4_row_bytes(head_dim: int) -> int:
    """Bytes of one token row of an NVFP4 slot: head_dim / 2 data + head_dim / 16 scales."""
    return head_dim // 2 + head_dim // NVFP4_BLOCK


def nvfp4_dequant(rows: np.ndarray, head_dim: int) -> np.ndarray:
    """[..., row_bytes] uint8 NVFP4 rows -> [..., head_dim] float64 (block scales
    applied, the tensor scale not)."""
    rows = np.asarray(rows, dtype=np.uint8)
    data = rows[..., :head_dim // 2]
    scales = rows[..., head_dim // 2:head_dim // 2 + head_dim // NVFP4_BLOCK]
    vals = np.empty(rows.shape[:-1] + (head_dim,), dtype=np.float64)
    vals[..., 0::2] = e2m1_to_float(data & 0xF)
    vals[..., 1::2] = e2m1_to_float(data >> 4)
    return vals * np.repeat(e4m3_to_float(scales), NVFP4_BLOCK, axis=-1)


_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    """Float values -> 4-bit e2m1 codes (uint8 0..15), from the format's
    definition: the nearest representable magnitude, ties to the code whose
    mantissa (last) bit is 0; magnitudes beyond 6 saturate to 6; the sign bit
    is kept (a negative value that rounds to zero is 0x8)."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    hi = np.clip(np.searchsorted(_E2M1_MAG, mag), 0, len(_E2M1_MAG) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - _E2M1_MAG[lo]
    d_hi = _E2M1_MAG[hi] - mag
    code = np.where(d_lo < d_hi, lo, hi)
    code = np.where(d_lo == d_hi, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(mag >= _E2M1_MAG[-1], len(_E2M1_MAG) - 1, code)
    return (code | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


def nvfp4_quantize(x: np.ndarray, scale: float) -> np.ndarray:
    """[..., D] values -> [..., D/2 + D/16] uint8 NVFP4 rows, for a pool with
    tensor scale ``scale``.  (Reading: the pages give the format, not the
    quantiser.)  Every 16-element block's scale is the E4M3 code of
    amax / (6 * scale) -- its largest magnitude onto E2M1's largest, 6 -- and
    each element the E2M1 code of x / (block scale * scale); a block whose
    scale code is 0 stores zero codes.  The operands are fp32, 6 * scale and
    block scale * scale fp32 products, each quotient one IEEE fp32 division:
    the precision in which the kernel takes the same rounding decisions."""
    x = np.asarray(x, dtype=np.float32)
    D = x.shape[-1]
    g = np.float32(scale)
    blocks = x.reshape(x.shape[:-1] + (D // NVFP4_BLOCK, NVFP4_BLOCK))
    amax = np.abs(blocks).max(axis=-1)
    q = (amax / (np.float32(6.0) * g)).astype(np.float32)
    sc = e4m3_encode(q)
    div = (e4m3_to_float(sc).astype(np.float32) * g).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        u = (blocks / div[..., None]).astype(np.float32)
    codes = np.where(div[..., None] == 0, np.uint8(0), e2m1_encode(u)).reshape(x.shape)
    out = np.empty(x.shape[:-1] + (nvfp4_row_bytes(D),), dtype=np.uint8)
    out[..., :D // 2] = codes[..., 0::2] | (codes[..., 1::2] << 4)
    out[..., D // 2:] = sc
    return out


# --------------------------------------------------------------------------
# Geometry of query tokens
# --------------------------------------------------------------------------
def query_positions(seq_lens: Sequence[int], q_lens: Sequence[int]) -> List[Tuple[int, int]]:
    """(request, position) of every query token, token-major.

    ``seq_lens[r]`` counts request r's KV tokens including its ``q_lens[r]`` new
    ones (the fused cache write runs before attention in ``forward_decode`` and
    ``forward_extend``), so the i-th new token is at seq_len - q_len + i.
    A request with seq_len 0 is idle (the idle-batch path of ``forward_decode``
    returns zeros): its tokens get position -1 and see nothing."""
    out = []
    for r, (L, n) in enumerate(zip(seq_lens, q_lens)):
        L, n = int(L), int(n)
        if L == 0:
            out.extend((r, -1) for _ in range(n))
            continue
        assert 0 <= n <= L, (r, L, n)
        for i in range(n):
            out.append((r, L - n + i))
    return out


def gather_sequence(pages: np.ndarray, block_table_row: Sequence[int], n_tokens: int,
                    block_size: int) -> np.ndarray:
    """Dense gather through the block table: logical token t of a request lives
    in page ``block_table_row[t // P]`` at row ``t % P``.

    ``pages``: [num_pages, H, P, X] (any float dtype).  Returns [n_tokens, H, X]
    float64 in logical token order."""
    H, X = pages.shape[1], pages.shape[3]
    seq = np.empty((n_tokens, H, X), dtype=np.float64)
    for t0 in range(0, n_tokens, block_size):
        page = int(block_table_row[t0 // block_size])
        assert 0 <= page < pages.shape[0], f"block {t0 // block_size}: page {page}"
        n = min(block_size, n_tokens - t0)
        # [H, n, X] -> [n, H, X]
        seq[t0:t0 + n] = np.transpose(pages[page, :, :n, :], (1, 0, 2))
    return seq


# --------------------------------------------------------------------------
# Index score: score_j = max over visible tokens t of block j of idx_q . idx_k[t]
# --------------------------------------------------------------------------
def block_scores(idx_q_vec: np.ndarray, idx_k_seq: np.ndarray, position: int,
                 block_size: int) -> np.ndarray:
    """Scores of the visible blocks of one query token and one KV head.

    ``idx_q_vec``: [d]; ``idx_k_seq``: [>= position + 1, d] (logical order).
    Returns [nb] float64 with nb = position // P + 1; only tokens t <= position
    take part (the last visible block may be partial)."""
    nb = position // block_size + 1
    dots = idx_k_seq[:position + 1].astype(np.float64) @ idx_q_vec.astype(np.float64)
    scores = np.empty(nb, dtype=np.float64)
    for j in range(nb):
        scores[j] = dots[j * block_size:min((j + 1) * block_size, position + 1)].max()
    return scores


# --------------------------------------------------------------------------
# Block selection: init blocks  U  local blocks  U  top-k of the rest
# --------------------------------------------------------------------------
def select_blocks(scores: Sequence[float], init_blocks: int, local_blocks: int,
                  topk_blocks: int) -> List[int]:
    """Selected blocks of one (query token, KV head), ascending.

    I  = [0, min(init, nb))              mandatory init (sink) blocks
    Lc = [max(0, nb - local), nb)        mandatory local window, incl. the
                                         query's own block
    C  = [0, nb) minus I minus Lc        candidates
    Top = first min(topk, |C|) of C sorted by (score descending, index ascending)
    Result: sorted(I | Lc | Top), of size min(nb, init + local + topk)."""
    nb = len(scores)
    I = set(range(0, min(init_blocks, nb)))
    Lc = set(range(max(0, nb - local_blocks), nb))
    C = [j for j in range(nb) if j not in I and j not in Lc]
    ranked = sorted(C, key=lambda j: (-float(scores[j]), j))
    top = set(ranked[:min(topk_blocks, len(C))])
    return sorted(I | Lc | top)


# --------------------------------------------------------------------------
# Attention: textbook softmax over a set of key/value rows
# --------------------------------------------------------------------------
def attention(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray,
              scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """out[g] = sum_t softmax_t(scale q_g . k_t) v_t; lse[g] = ln sum_t exp(scale q_g . k_t).

    ``q_rows``: [G, D]; ``k``, ``v``: [n, D].  n = 0 gives out = 0, lse = -inf
    (the idle / empty-request convention of ``forward_decode``)."""
    q_rows = np.asarray(q_rows, dtype=np.float64)
    G = q_rows.shape[0]
    if k.shape[0] == 0:
        return np.zeros((G, v.shape[1])), np.full(G, -np.inf)
    s = scale * (q_rows @ np.asarray(k, dtype=np.float64).T)       # [G, n]
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    out = (e @ np.asarray(v, dtype=np.float64)) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def combine(o_parts: np.ndarray, lse_parts: np.ndarray) -> Tuple[np.ndarray, float]:
    """Merge attention results over disjoint key sets (split-K flash decoding):
    lse = ln sum_s exp(lse_s); out = sum_s exp(lse_s - lse) o_s.
    Parts with lse = -inf (empty) carry no weight; all empty -> (0, -inf)."""
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    o_parts = np.asarray(o_parts, dtype=np.float64)
    if lse_parts.size == 0 or np.all(np.isneginf(lse_parts)):
        return np.zeros(o_parts.shape[1:]), -np.inf
    m = lse_parts.max()
    w = np.exp(lse_parts - m)
    lse = m + math.log(w.sum())
    out = np.tensordot(np.exp(lse_parts - lse), o_parts, axes=(0, 0))
    return out, lse


# --------------------------------------------------------------------------
# The whole path for a batch of query tokens
# --------------------------------------------------------------------------
def sparse_attention(*, seq_lens, q_lens, block_table, idx_q, idx_k_pages, q,
                     k_pages, v_pages, num_kv_heads: int, block_size: int,
                     init_blocks: int, local_blocks: int, topk_blocks: int,
                     softmax_scale: float, k_scale: float = 1.0, v_scale: float = 1.0,
                     kv_is_e4m3: bool = False, kv_is_nvfp4: bool = False, tokens=None,
                     kv_heads=None) -> Dict[str, object]:
    """Index score -> block selection -> attention over the selected blocks.

    Arrays are numpy: ``idx_q [T, H_kv, d]``, ``idx_k_pages [pages, H_kv, P, d]``,
    ``q [T, H_q, D]``, ``k_pages / v_pages [pages, H_kv, P, D]`` (float, or uint8
    e4m3 codes when ``kv_is_e4m3``; dequantised value = decoded code * scale).
    ``kv_is_nvfp4``: ``k_pages`` and ``v_pages`` are NVFP4 pools [pages, 2 H_kv,
    P, row bytes] whose slot 2h holds the keys and slot 2h + 1 the values of KV
    head h; value = nvfp4_dequant(row) * k_scale (keys) or * v_scale (values).
    ``tokens`` / ``kv_heads`` restrict the work to a sample (default: all).

    Returns dict with, per computed (t, h): ``scores[(t, h)]`` [nb],
    ``selected[(t, h)]`` list, and arrays ``out [T, H_q, D]``, ``lse [T, H_q]``
    (NaN where not computed)."""
    T, H_q, D = q.shape
    G = H_q // num_kv_heads
    toks = query_positions(seq_lens, q_lens)
    assert len(toks) == T
    tokens = range(T) if tokens is None else tokens
    kv_heads = range(num_kv_heads) if kv_heads is None else kv_heads
    out = np.full((T, H_q, D), np.nan)
    lse = np.full((T, H_q), np.nan)
    scores, selected = {}, {}
    seq_cache = {}
    for t in tokens:
        r, p = toks[t]
        if r not in seq_cache:
            L = int(seq_lens[r])
            ik = gather_sequence(idx_k_pages, block_table[r], L, block_size)
            if kv_is_nvfp4:
                kk = gather_sequence(k_pages[:, 0::2], block_table[r], L, block_size)
                vv = gather_sequence(v_pages[:, 1::2], block_table[r], L, block_size)
                kk = nvfp4_dequant(kk.astype(np.uint8), q.shape[2]) * k_scale
                vv = nvfp4_dequant(vv.astype(np.uint8), q.shape[2]) * v_scale
            else:
                kk = gather_sequence(k_pages, block_table[r], L, block_size)
                vv = gather_sequence(v_pages, block_table[r], L, block_size)
            if kv_is_e4m3:
                kk = e4m3_to_float(kk.astype(np.uint8)) * k_scale
                vv = e4m3_to_float(vv.astype(np.uint8)) * v_scale
            seq_cache = {r: (ik, kk, vv)}
        ik, kk, vv = seq_cache[r]
        if p < 0:                              # idle request: attends to nothing
            for h in kv_heads:
                scores[(t, h)], selected[(t, h)] = np.zeros(0), []
                out[t, h * G:(h + 1) * G] = 0.0
                lse[t, h * G:(h + 1) * G] = -np.inf
            continue
        for h in kv_heads:
            sc = block_scores(idx_q[t, h], ik[:, h, :], p, block_size)
            sel = select_blocks(sc, init_blocks, local_blocks, topk_blocks)
            scores[(t, h)] = sc
            selected[(t, h)] = sel
            rows = [tt for j in sel
                    for tt in range(j * block_size, min((j + 1) * block_size, p + 1))]
            o, ls = attention(q[t, h * G:(h + 1) * G], kk[rows, h, :], vv[rows, h, :],
                              softmax_scale)
            out[t, h * G:(h + 1) * G] = o
            lse[t, h * G:(h + 1) * G] = ls
    return {"scores": scores, "selected": selected, "out": out, "lse": lse}


# --------------------------------------------------------------------------
# Index-value branch (sglang MiniMaxSparseAttnBackend: layers outside
# disable_value_layer_ids keep an index-value cache beside the index keys,
# get_index_kv_buffer, and the sparse ops return (idx_o, o) with idx_o of shape
# [tokens, num_idx_heads * idx_head_dim]).  The pages do not give idx_o's
# formula.  PARITY UNPINNED: this reading -- the index head as a dense causal
# attention head over every visible token, softmax scale 1 / sqrt(d) -- is
# this build's, not the pages'.  The function itself is the textbook
# `attention` over the gathered index keys and values.
# --------------------------------------------------------------------------
def index_attention(idx_q_vec: np.ndarray, idx_k_seq: np.ndarray, idx_v_seq: np.ndarray,
                    position: int) -> Tuple[np.ndarray, float]:
    """idx_o of one query token and index head: softmax(idx_q . idx_k[u] /
    sqrt(d)) over the tokens u <= position, applied to idx_v[u]."""
    d = idx_q_vec.shape[-1]
    o, lse = attention(np.asarray(idx_q_vec, dtype=np.float64)[None],
                       idx_k_seq[:position + 1], idx_v_seq[:position + 1], 1.0 / math.sqrt(d))
    return o[0], float(lse[0])


# --------------------------------------------------------------------------
# Dense-sparse decode (sglang MiniMaxSparseAttnBackend._dense_sparse_main_decode
# and the SGLANG_OPT_USE_MINIMAX_DENSE_SPARSE_DECODE branch of forward_decode):
# the selected blocks become a compacted page table and a dense paged decode
# runs over it with real_seq_lens, max_seq_len = topk_blocks * block_size.
# --------------------------------------------------------------------------
def compact_selection(selected: Sequence[int], block_table_row: Sequence[int], position: int,
                      block_size: int) -> Tuple[List[int], int]:
    """Pages of the selected blocks in ascending block order, and the number of
    keys of the compacted sequence: each block contributes its tokens at
    positions <= ``position`` (every selected block is full except the query's
    own, which is the last)."""
    pages, n = [], 0
    for j in sorted(selected):
        pages.append(int(block_table_row[j]))
        n += max(0, min(block_size, position + 1 - j * block_size))
    return pages, n


def paged_attention(q_rows: np.ndarray, k_pages: np.ndarray, v_pages: np.ndarray,
                    pages: Sequence[int], seq_len: int, head: int, scale: float,
                    block_size: int) -> Tuple[np.ndarray, np.ndarray]:
    """Dense paged decode: the sequence is the first ``seq_len`` rows of the
    listed pages, in order (rows of page i at positions i*P .. i*P + P - 1);
    every query row of ``q_rows`` attends to all of them (KV head ``head``)."""
    k = gather_sequence(k_pages, pages, seq_len, block_size)[:, head, :]
    v = gather_sequence(v_pages, pages, seq_len, block_size)[:, head, :]
    return attention(q_rows, k, v, scale)


# --------------------------------------------------------------------------
# Cache write before attention (sglang forward_decode / forward_extend call
# ``set_fused_kv_index_buffer(layer, out_cache_loc, k, v, idx_k, idx_v)``
# before the sparse op, which is why seq_lens already counts the new tokens).
# --------------------------------------------------------------------------
def cache_slots(seq_lens: Sequence[int], q_lens: Sequence[int], block_table,
                block_size: int) -> List[int]:
    """Token slot (page * P + row) of every new query token, token-major: token
    i of request r sits at position p = seq_len - q_len + i, in page
    block_table[r][p // P] at row p % P.  Tokens of idle requests: -1."""
    slots = []
    for r, p in query_positions(seq_lens, q_lens):
        if p < 0:
            slots.append(-1)
            continue
        page = int(block_table[r][p // block_size])
        slots.append(page * block_size + p % block_size)
    return slots


def cache_write(pool: np.ndarray, slots: Sequence[int], rows: np.ndarray,
                e4m3_scale=None) -> np.ndarray:
    """A copy of ``pool`` [num_pages, H, P, X] with ``rows[t, h]`` ([T, H, X])
    stored at page slot // P, head h, row slot % P for every token whose slot
    is >= 0.  ``e4m3_scale`` None: stored as given (bf16 values); otherwise the
    pool holds e4m3 codes and each value is stored as the code of
    float32(x) / float32(scale) (one IEEE fp32 division, then round to e4m3)."""
    out = pool.copy()
    P = pool.shape[2]
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        page, row = slot // P, slot % P
        if e4m3_scale is None:
            out[page, :, row, :] = rows[t]
        else:
            q = np.asarray(rows[t], dtype=np.float32) / np.float32(e4m3_scale)
            out[page, :, row, :] = e4m3_encode(q)
    return out


def cache_write_nvfp4(pool: np.ndarray, slots: Sequence[int], rows: np.ndarray, scale: float,
                      kind: int) -> np.ndarray:
    """A copy of the NVFP4 pool [num_pages, 2 H, P, row bytes] with rows[t, h]
    ([T, H, D] values) quantised (nvfp4_quantize, tensor scale ``scale``) into
    slot 2 h + kind (0: keys, 1: values) of page slot // P at row slot % P,
    for every token whose slot is >= 0."""
    out = pool.copy()
    P = pool.shape[2]
    H = pool.shape[1] // 2
    for t, slot in enumerate(slots):
        if slot < 0:
            continue
        page, row = slot // P, slot % P
        for h in range(H):
            out[page, 2 * h + kind, row, :] = nvfp4_quantize(rows[t, h], scale)
    return out


# --------------------------------------------------------------------------
# Key-block -> query CSR for prefill (vLLM MiniMaxM3SparseMSAImpl.forward,
# ``build_k2q_csr``).  Row (h, r, j) lists, ascending, the query tokens of
# request r whose selection for KV head h contains key block j.  Rows are laid
# out on the fixed grid row = (h * num_reqs + r) * max_blocks + j, so the
# structure's shape depends only on sizes, never on data.
# --------------------------------------------------------------------------
def build_k2q_csr(selected: np.ndarray, token_request: Sequence[int], num_reqs: int,
                  max_blocks: int) -> Tuple[np.ndarray, np.ndarray]:
    """``selected``: [T, H_kv, S] int (-1 padded).  Returns (row_ptr
    [H_kv * num_reqs * max_blocks + 1], q_indices [row_ptr[-1]])."""
    T, H, S = selected.shape
    rows: List[List[int]] = [[] for _ in range(H * num_reqs * max_blocks)]
    for t in range(T):
        r = int(token_request[t])
        for h in range(H):
            for j in selected[t, h]:
                if j >= 0:
                    rows[(h * num_reqs + r) * max_blocks + int(j)].append(t)
    row_ptr = np.zeros(len(rows) + 1, dtype=np.int64)
    for i, lst in enumerate(rows):
        row_ptr[i + 1] = row_ptr[i] + len(lst)
    q_indices = np.array([t for lst in rows for t in sorted(lst)], dtype=np.int64)
    return row_ptr, q_indices
