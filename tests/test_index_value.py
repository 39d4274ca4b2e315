"""The index-value branch (GPU): msa_index_attention and the idx_v cache write.

The pages name the index-value cache (idx_v, get_index_kv_buffer) and idx_o
([tokens, num_idx_heads * idx_head_dim]) without idx_o's formula, so the
reading tested here -- dense causal attention of the index head over every
visible token, scale 1 / sqrt(d) -- is this library's, and its parity with
the pages is unpinned.  What is checked: the kernels compute that reading,
element by element against the oracle's index_attention, for d = 64 and
128, decode and verify, with a flagged page, and the idx_v write lands
byte-exact; replay of a captured call equals eager."""
import numpy as np
import pytest
import torch

import block_sparse_paged_msa_gb300 as msa
import oracle
from block_sparse_paged_msa_gb300 import workloads as wl
from gpu_util import LSE_MAX, OUT_MAX, OUT_MEAN
from oracle_io import to_np

pytestmark = pytest.mark.gpu


def _run(w, idx_v):
    cfg = msa.config_for(w.spec)
    sa = msa.SparseAttention(cfg)
    msa.plan(cfg, w.seq_lens, w.block_table, sa.ws)
    T, H, d = w.num_tokens, w.spec.num_kv_heads, w.spec.index_dim
    scratch = torch.empty(msa.index_attention_scratch_bytes(cfg), dtype=torch.uint8,
                          device="cuda")
    out = torch.full((msa.ops.max_tokens(cfg), H, d), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    lse = torch.full((msa.ops.max_tokens(cfg), H), float("nan"), device="cuda")
    msa.index_attention(cfg, sa.ws, w.idx_q, w.idx_k_pages, idx_v, scratch, out, lse)
    torch.cuda.synchronize()
    return sa, out[:T], lse[:T]


def _compare(w, idx_v, out, lse, tokens=None):
    s = w.spec
    toks = oracle.query_positions(to_np(w.seq_lens), to_np(w.q_lens))
    bt, iq = to_np(w.block_table), to_np(w.idx_q)
    ik, iv = to_np(w.idx_k_pages), to_np(idx_v)
    o, ls = to_np(out), lse.cpu().numpy().astype(np.float64)
    errs, lerrs = [], []
    for t, (r, p) in enumerate(toks):
        if tokens is not None and t not in tokens:
            continue
        if p < 0:
            assert np.all(o[t] == 0) and np.all(np.isneginf(ls[t]))
            continue
        kseq = oracle.gather_sequence(ik, bt[r], p + 1, s.block_size)
        vseq = oracle.gather_sequence(iv, bt[r], p + 1, s.block_size)
        for h in range(s.num_kv_heads):
            want, wl_ = oracle.index_attention(iq[t, h], kseq[:, h], vseq[:, h], p)
            errs.append(np.abs(o[t, h] - want))
            lerrs.append(abs(ls[t, h] - wl_))
    e = np.concatenate(errs)
    assert e.max() <= OUT_MAX and e.mean() <= OUT_MEAN and max(lerrs) <= LSE_MAX, \
        (e.max(), e.mean(), max(lerrs))


@pytest.mark.parametrize("name,kw", [("medium_decode", dict(batch=3)), ("tiny_decode", {}),
                                     ("verify", {}),
                                     ("medium_decode", dict(seq_lens=(1, 128, 129, 900, 0),
                                                            seq_len_range=None, batch=5))])
def test_index_attention_every_element(name, kw):
    spec = wl.small(name, **kw) if name != "tiny_decode" else wl.WORKLOADS[name]
    w = wl.make_workload(spec, device="cuda")
    idx_v = wl.index_values(spec, seed=spec.seed + 77, device="cuda")
    sa, out, lse = _run(w, idx_v)
    assert msa.check_device_error(sa.ws) == 0
    _compare(w, idx_v, out, lse)


def test_index_attention_skips_flagged_pages():
    spec = wl.small("medium_decode", batch=3)
    w = wl.make_workload(spec, device="cuda")
    w.block_table[1, 2] = spec.num_pages + 4
    idx_v = wl.index_values(spec, seed=9, device="cuda")
    sa, out, lse = _run(w, idx_v)
    assert msa.check_device_error(sa.ws) & 1
    _compare(w, idx_v, out, lse, tokens=[0, 2])
    assert torch.isfinite(out[1].float()).all()


def test_idx_v_cache_write_bytes_match_oracle():
    spec = wl.small("medium_decode", batch=3)
    w = wl.make_workload(spec, device="cuda")
    cfg = msa.config_for(spec)
    sa = msa.SparseAttention(cfg)
    idx_v = wl.index_values(spec, seed=10, device="cuda")
    T = w.num_tokens
    k, v, idx_k = wl.new_token_rows(spec, T, seed=11, device="cuda")
    new_v = wl.new_token_rows(spec, T, seed=12, device="cuda")[0][..., :spec.index_dim].contiguous()
    slots = oracle.cache_slots(to_np(w.seq_lens), to_np(w.q_lens), to_np(w.block_table), 128)
    want = oracle.cache_write(to_np(idx_v), slots, to_np(new_v))
    msa.plan(cfg, w.seq_lens, w.block_table, sa.ws)
    msa.cache_write(cfg, sa.ws, k, v, idx_k, w.k_pages, w.v_pages, w.idx_k_pages,
                    idx_v=new_v, idx_v_pages=idx_v)
    assert msa.check_device_error(sa.ws) == 0
    assert np.array_equal(to_np(idx_v), want)


def test_index_attention_graph_replay_equals_eager():
    base = wl.small("medium_decode", batch=3)
    w = wl.make_workload(base, device="cuda")
    cfg = msa.config_for(base)
    idx_v = wl.index_values(base, seed=13, device="cuda")
    sa = msa.SparseAttention(cfg)
    scratch = torch.empty(msa.index_attention_scratch_bytes(cfg), dtype=torch.uint8,
                          device="cuda")
    T, H, d = w.num_tokens, base.num_kv_heads, base.index_dim
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((T, H), device="cuda")
    bufs = {k: getattr(w, k).clone() for k in ("seq_lens", "block_table", "idx_q", "idx_k_pages")}

    def call():
        msa.plan(cfg, bufs["seq_lens"], bufs["block_table"], sa.ws)
        msa.index_attention(cfg, sa.ws, bufs["idx_q"], bufs["idx_k_pages"], idx_v, scratch, out,
                            lse)

    call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(graph, stream=st):
            call()
    torch.cuda.current_stream().wait_stream(st)
    w2 = wl.make_workload(base.replace(seed=501), device="cuda")
    for k, v in bufs.items():
        v.copy_(getattr(w2, k))
    graph.replay()
    torch.cuda.synchronize()
    g_out, g_lse = out.clone(), lse.clone()
    call()
    torch.cuda.synchronize()
    assert torch.equal(g_out, out) and torch.equal(g_lse, lse)
