"""Seeded synthetic inputs for block-sparse paged MSA decode, verify and prefill.

This module is the only code shared by the CUDA path's tests and the fp64 oracle.
It draws inputs and nothing else: it holds none of the method's arithmetic (no
scores, no selection, no softmax).  The shapes follow the serving batches that
the MiniMax-M3 sparse-attention backends are built for (sglang
``minimax_sparse_backend.py``, ``MiniMaxSparseAttnBackend.forward_decode`` and
``forward_extend``; vLLM ``minimax_m3/nvidia/sparse_attention_msa.py``,
``MiniMaxM3SparseMSAImpl.forward``):

* a paged KV pool, one page = one 128-token block, stored HND per page:
  ``k_pages, v_pages: [num_pages, H_kv, P, D]`` and the index keys
  ``idx_k_pages: [num_pages, H_kv, P, d]``;
* a block table ``[B, max_blocks]`` int32 that maps request r's logical block j
  to a physical page (entries past a request's last block are -1);
* ``seq_lens[r]``: the KV length of request r *including* its new query tokens
  (the cache write precedes attention in ``forward_decode``); query i of a
  request with ``n_q`` new tokens sits at position ``seq_lens[r] - n_q + i``;
* queries ``q: [T, H_q, D]`` and index queries ``idx_q: [T, H_kv, d]``, token-major;
* an NVFP4 KV pool is one uint8 tensor ``[num_pages, 2 * H_kv, P, D/2 + D/16]``
  (slot 2h: keys of KV head h, slot 2h + 1: its values), passed as both
  ``k_pages`` and ``v_pages``: each 72-byte row is 64 bytes of packed FP4 codes
  followed by 8 E4M3 block scales.

Draw order (fixed, so a seed names one input set): seq_lens, page permutation,
idx_q, idx_k, q, k, v.  Index values are integers in [-4, 4] stored as bf16, so
every index dot product is exact in fp32.  Q/K/V are bf16 N(0, 1).  An fp8 KV
pool stores round-to-nearest-even e4m3 codes of N(0, 1)/scale.  An NVFP4 pool
holds uniformly random FP4 codes (all 16, both signs) with block-scale codes
uniform over the e4m3 codes of [0.25, 1] (0x28 .. 0x38), so dequantised values
reach +-6 with the tensor scale on top.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

BLOCK = 128


@dataclasses.dataclass(frozen=True)
class WorkloadSpec:
    """Shape and value recipe of one synthetic workload."""

    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    index_dim: int
    init_blocks: int
    local_tokens: int
    topk_blocks: int
    num_pages: int
    seed: int
    seq_lens: Optional[tuple] = None          # explicit KV lengths, or
    seq_len_range: Optional[tuple] = None     # inclusive uniform integer range
    q_len: int = 1                            # new query tokens per request
    kv_dtype: str = "bf16"                    # "bf16" | "fp8_e4m3" | "nvfp4"
    kv_scale: float = 1.0                     # per-tensor fp8 / nvfp4 scale (k and v)
    block_size: int = BLOCK
    index_range: int = 4                      # index values uniform in [-r, r]

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def max_seq_len(self) -> int:
        if self.seq_lens is not None:
            return max(self.seq_lens) if self.seq_lens else 0
        return self.seq_len_range[1]

    @property
    def max_blocks(self) -> int:
        return max(1, -(-self.max_seq_len // self.block_size))

    def replace(self, **kw) -> "WorkloadSpec":
        return dataclasses.replace(self, **kw)


# The five configurations of the method's serving workloads.  The names say what
# each one is; ids (1..6) only pick the seed.
WORKLOADS = {
    "tiny_decode": WorkloadSpec(
        name="tiny_decode", batch=2, seq_lens=(1000, 1500), num_q_heads=8,
        num_kv_heads=1, head_dim=128, index_dim=64, init_blocks=1,
        local_tokens=128, topk_blocks=4, num_pages=32, seed=1001),
    "medium_decode": WorkloadSpec(
        name="medium_decode", batch=32, seq_len_range=(8192, 32768),
        num_q_heads=64, num_kv_heads=8, head_dim=128, index_dim=128,
        init_blocks=1, local_tokens=256, topk_blocks=16, num_pages=16384,
        seed=1002),
    "long_decode": WorkloadSpec(
        name="long_decode", batch=128, seq_len_range=(65536, 131072),
        num_q_heads=64, num_kv_heads=8, head_dim=128, index_dim=128,
        init_blocks=1, local_tokens=512, topk_blocks=32, num_pages=114688,
        seed=1003),
    "fp8_decode": WorkloadSpec(
        name="fp8_decode", batch=32, seq_len_range=(8192, 32768),
        num_q_heads=64, num_kv_heads=8, head_dim=128, index_dim=128,
        init_blocks=1, local_tokens=256, topk_blocks=8, num_pages=16384,
        kv_dtype="fp8_e4m3", kv_scale=2.0 ** -5, seed=1004),
    # NVFP4 KV cache with the medium decode shapes
    "nvfp4_decode": WorkloadSpec(
        name="nvfp4_decode", batch=32, seq_len_range=(8192, 32768),
        num_q_heads=64, num_kv_heads=8, head_dim=128, index_dim=128,
        init_blocks=1, local_tokens=256, topk_blocks=16, num_pages=16384,
        kv_dtype="nvfp4", kv_scale=0.75, seed=1007),
    # chunked prefill: 4 requests, 16384 cached tokens + a 2048-token chunk each
    "prefill": WorkloadSpec(
        name="prefill", batch=4, seq_lens=(18432,) * 4, q_len=2048,
        num_q_heads=64, num_kv_heads=8, head_dim=128, index_dim=128,
        init_blocks=1, local_tokens=256, topk_blocks=16, num_pages=1024,
        seed=1005),
    # the same chunked prefill over an NVFP4 KV cache
    "nvfp4_prefill": WorkloadSpec(
        name="nvfp4_prefill", batch=4, seq_lens=(18432,) * 4, q_len=2048,
        num_q_heads=64, num_kv_heads=8, head_dim=128, index_dim=128,
        init_blocks=1, local_tokens=256, topk_blocks=16, num_pages=1024,
        kv_dtype="nvfp4", kv_scale=0.75, seed=1008),
    # speculative verify: 4 draft tokens on a 32768-token context
    "verify": WorkloadSpec(
        name="verify", batch=64, seq_lens=(32768 + 4,) * 64, q_len=4,
        num_q_heads=64, num_kv_heads=8, head_dim=128, index_dim=128,
        init_blocks=1, local_tokens=256, topk_blocks=16, num_pages=24576,
        seed=1006),
}


def small(name: str, **kw) -> WorkloadSpec:
    """A reduced copy of a workload with the same structure (several blocks per
    request, ragged last pages, shuffled pool) that the oracle finishes in
    seconds."""
    base = WORKLOADS[name]
    defaults = {
        "medium_decode": dict(batch=4, seq_len_range=(700, 3000), num_pages=160),
        "fp8_decode": dict(batch=4, seq_len_range=(700, 3000), num_pages=160),
        "nvfp4_decode": dict(batch=4, seq_len_range=(700, 3000), num_pages=160),
        "long_decode": dict(batch=3, seq_len_range=(3000, 6000), num_pages=200),
        "tiny_decode": dict(),
        "verify": dict(batch=4, seq_lens=(1500, 2000, 2600, 3001), num_pages=128),
        "prefill": dict(batch=2, seq_lens=(1400, 900), q_len=300, num_pages=40),
        "nvfp4_prefill": dict(batch=2, seq_lens=(1400, 900), q_len=300, num_pages=40),
    }[name]
    defaults.update(kw)
    return base.replace(name=base.name + "_small", **defaults)


def _draw_seq_lens(spec: WorkloadSpec, gen: torch.Generator, device) -> torch.Tensor:
    if spec.seq_lens is not None:
        return torch.tensor(spec.seq_lens, dtype=torch.int32, device=device)
    lo, hi = spec.seq_len_range
    return torch.randint(lo, hi + 1, (spec.batch,), generator=gen, device=device,
                         dtype=torch.int64).to(torch.int32)


def _randint_bf16(shape, r, gen, device, chunk_rows=4096) -> torch.Tensor:
    """Integers uniform in [-r, r] stored as bf16, drawn page-chunk by page-chunk
    so that no int64 temporary of the full pool is ever held."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        flat[s:e] = torch.randint(-r, r + 1, (e - s, flat.shape[1]), generator=gen,
                                  device=device, dtype=torch.int32).to(torch.bfloat16)
    return out


def _randn_kv(shape, spec: WorkloadSpec, gen, device, chunk_rows=4096) -> torch.Tensor:
    """bf16 N(0,1), or fp8-e4m3 codes of N(0,1)/scale (round to nearest even)."""
    dt = torch.bfloat16 if spec.kv_dtype == "bf16" else torch.float8_e4m3fn
    out = torch.empty(shape, dtype=dt, device=device)
    flat = out.view(shape[0], -1)
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        x = torch.randn((e - s, flat.shape[1]), generator=gen, device=device,
                        dtype=torch.float32)
        if spec.kv_dtype == "bf16":
            flat[s:e] = x.to(torch.bfloat16)
        else:
            flat[s:e] = (x / spec.kv_scale).to(torch.float8_e4m3fn)
    return out


def _nvfp4_pool(spec: WorkloadSpec, gen, device, chunk_rows=256) -> torch.Tensor:
    """[num_pages, 2 H_kv, P, D/2 + D/16] uint8: random FP4 code bytes, then
    block-scale codes uniform over 0x28 .. 0x38 (e4m3 0.25 .. 1.0)."""
    D = spec.head_dim
    shape = (spec.num_pages, 2 * spec.num_kv_heads, spec.block_size, D // 2 + D // 16)
    out = torch.empty(shape, dtype=torch.uint8, device=device)
    flat = out.view(shape[0], -1, shape[-1])
    for s in range(0, shape[0], chunk_rows):
        e = min(shape[0], s + chunk_rows)
        n = flat.shape[1]
        flat[s:e, :, :D // 2] = torch.randint(0, 256, (e - s, n, D // 2), generator=gen,
                                              device=device, dtype=torch.int32).to(torch.uint8)
        flat[s:e, :, D // 2:] = torch.randint(0x28, 0x39, (e - s, n, D // 16), generator=gen,
                                              device=device, dtype=torch.int32).to(torch.uint8)
    return out


@dataclasses.dataclass
class Workload:
    spec: WorkloadSpec
    seq_lens: torch.Tensor        # [B] int32, KV length incl. new tokens
    q_lens: torch.Tensor          # [B] int32, new query tokens per request
    cu_seqlens_q: torch.Tensor    # [B+1] int32
    block_table: torch.Tensor     # [B, max_blocks] int32, -1 past the end
    idx_q: torch.Tensor           # [T, H_kv, d] bf16
    idx_k_pages: torch.Tensor     # [num_pages, H_kv, P, d] bf16
    q: torch.Tensor               # [T, H_q, D] bf16
    k_pages: torch.Tensor         # [num_pages, H_kv, P, D] bf16 | float8_e4m3fn
    v_pages: torch.Tensor

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    def to(self, device) -> "Workload":
        f = {k.name: getattr(self, k.name) for k in dataclasses.fields(self)}
        for k, v in f.items():
            if isinstance(v, torch.Tensor):
                f[k] = v.to(device)
        return Workload(**f)


def make_workload(spec: WorkloadSpec, device="cpu", kv_pool=True) -> Workload:
    """Draw one seeded input set for ``spec`` on ``device``.

    ``kv_pool=False`` skips the q/k/v draws (index-only uses)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(spec.seed)
    B, P = spec.batch, spec.block_size
    seq_lens = _draw_seq_lens(spec, gen, device)
    # seq_len 0 marks an idle request; any other request holds its query tokens
    assert all(L == 0 or L >= spec.q_len for L in seq_lens.tolist())
    nb = [-(-int(s) // P) for s in seq_lens.tolist()]
    need = sum(nb)
    if need > spec.num_pages:
        raise ValueError(f"{spec.name}: {need} blocks do not fit {spec.num_pages} pages")
    perm = torch.randperm(spec.num_pages, generator=gen, device=device).to(torch.int32)
    block_table = torch.full((B, spec.max_blocks), -1, dtype=torch.int32, device=device)
    off = 0
    for r, n in enumerate(nb):
        block_table[r, :n] = perm[off:off + n]
        off += n
    q_lens = torch.full((B,), spec.q_len, dtype=torch.int32, device=device)
    cu = torch.zeros(B + 1, dtype=torch.int32, device=device)
    cu[1:] = torch.cumsum(q_lens, 0).to(torch.int32)
    T = B * spec.q_len
    Hkv, d, D = spec.num_kv_heads, spec.index_dim, spec.head_dim
    idx_q = _randint_bf16((T, Hkv, d), spec.index_range, gen, device)
    idx_k = _randint_bf16((spec.num_pages, Hkv, P, d), spec.index_range, gen, device,
                          chunk_rows=256)
    if kv_pool:
        q = torch.randn((T, spec.num_q_heads, D), generator=gen, device=device,
                        dtype=torch.float32).to(torch.bfloat16)
        if spec.kv_dtype == "nvfp4":
            k = v = _nvfp4_pool(spec, gen, device)     # one pool: K and V slots per head
        else:
            k = _randn_kv((spec.num_pages, Hkv, P, D), spec, gen, device, chunk_rows=256)
            v = _randn_kv((spec.num_pages, Hkv, P, D), spec, gen, device, chunk_rows=256)
    else:
        q = torch.empty((T, spec.num_q_heads, D), dtype=torch.bfloat16, device=device)
        k = v = torch.empty((0, Hkv, P, D), dtype=torch.bfloat16, device=device)
    return Workload(spec, seq_lens, q_lens, cu, block_table, idx_q, idx_k, q, k, v)


def new_token_rows(spec: WorkloadSpec, num_tokens: int, seed: int, device="cpu"):
    """The new tokens' key, value and index-key rows a step writes into the
    cache before attention: k, v [T, H_kv, D] bf16 N(0, 1) and idx_k [T, H_kv,
    d] integers in [-r, r] as bf16, drawn in that order from `seed`."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shape = (num_tokens, spec.num_kv_heads, spec.head_dim)
    k = torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)
    idx_k = _randint_bf16((num_tokens, spec.num_kv_heads, spec.index_dim), spec.index_range,
                          gen, device)
    return k, v, idx_k


def index_values(spec: WorkloadSpec, seed: int, device="cpu") -> torch.Tensor:
    """An index-value pool beside the index keys, [num_pages, H_kv, P, d] bf16
    N(0, 1), drawn from its own seed (the layers that keep an index-value
    cache in the pages' backend)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shape = (spec.num_pages, spec.num_kv_heads, spec.block_size, spec.index_dim)
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    for s in range(0, shape[0], 256):
        e = min(shape[0], s + 256)
        flat[s:e] = torch.randn((e - s, flat.shape[1]), generator=gen, device=device,
                                dtype=torch.float32).to(torch.bfloat16)
    return out
