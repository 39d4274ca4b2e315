"""msa_decode_step (one call for the whole decode / verify step) gives the same
results, bit for bit, as the separate stage calls (GPU)."""
import pytest
import torch

import block_sparse_paged_msa_gb300 as msa
from block_sparse_paged_msa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _separate(cfg, w):
    sa = msa.SparseAttention(cfg)
    msa.plan(cfg, w.seq_lens, w.block_table, sa.ws)
    msa.index_score(cfg, sa.ws, w.idx_q, w.idx_k_pages, sa.block_scores)
    msa.topk_select(cfg, sa.ws, sa.block_scores, sa.selected)
    msa.sparse_decode(cfg, sa.ws, w.q, w.k_pages, w.v_pages, sa.selected)
    msa.combine(cfg, sa.ws, sa.out, sa.lse)
    return sa


@pytest.mark.parametrize("name,kw", [("medium_decode", {}), ("verify", {}),
                                     ("fp8_decode", {}), ("nvfp4_decode", {}),
                                     ("long_decode", {}),
                                     ("medium_decode", dict(index_dim=64, topk_blocks=0)),
                                     ("medium_decode", dict(seq_lens=(1, 128, 129, 3000, 0),
                                                            seq_len_range=None, batch=5))])
def test_decode_step_equals_separate(name, kw):
    spec = wl.small(name, **kw)
    w = wl.make_workload(spec, device="cuda")
    cfg = msa.config_for(spec)
    a = _separate(cfg, w)
    b = msa.SparseAttention(cfg)
    b.block_scores.fill_(float("nan"))
    b.selected.fill_(-7)
    msa.ops.decode_step(cfg, b.ws, w.seq_lens, w.block_table, w.idx_q, w.idx_k_pages, w.q,
                        w.k_pages, w.v_pages, b.block_scores, b.selected, b.out, b.lse)
    torch.cuda.synchronize()
    assert msa.check_device_error(a.ws) == 0 and msa.check_device_error(b.ws) == 0
    T = w.num_tokens
    assert torch.equal(a.selected[:T], b.selected[:T])
    assert torch.equal(a.out[:T], b.out[:T]) and torch.equal(a.lse[:T], b.lse[:T])


def test_decode_step_with_bad_pages():
    """A request with a bad page is flagged and still gets a full selection."""
    spec = wl.small("medium_decode", batch=3)
    w = wl.make_workload(spec, device="cuda")
    w.block_table[1, 3] = spec.num_pages + 1
    cfg = msa.config_for(spec)
    sa = msa.SparseAttention(cfg)
    sa.selected.fill_(-7)
    sa.run(w.seq_lens, w.block_table, w.idx_q, w.idx_k_pages, w.q, w.k_pages, w.v_pages)
    assert msa.check_device_error(sa.ws) & 1
    assert bool((sa.selected[:3] != -7).all())


@pytest.mark.parametrize("name,kw", [("medium_decode", {}), ("fp8_decode", {}),
                                     ("medium_decode", dict(index_dim=64, topk_blocks=0)),
                                     ("medium_decode", dict(seq_lens=(1, 128, 129, 3000, 0),
                                                            seq_len_range=None, batch=5)),
                                     ("verify", {})])
def test_index_score_topk_equals_two_calls(name, kw):
    """msa_index_score_topk writes the same block scores and selections, bit
    for bit, as msa_index_score then msa_topk_select, including idle requests
    and a flagged page; twice on the same workspace."""
    spec = wl.small(name, **kw)
    w = wl.make_workload(spec, device="cuda")
    if w.block_table.shape[0] > 2 and int(w.seq_lens[2]) > 300:
        w.block_table[2, 1] = spec.num_pages + 3
    cfg = msa.config_for(spec)
    a = msa.SparseAttention(cfg)
    msa.plan(cfg, w.seq_lens, w.block_table, a.ws)
    msa.index_score(cfg, a.ws, w.idx_q, w.idx_k_pages, a.block_scores)
    msa.topk_select(cfg, a.ws, a.block_scores, a.selected)
    b = msa.SparseAttention(cfg)
    T = w.num_tokens
    for _ in range(2):
        b.block_scores.fill_(float("nan"))
        b.selected.fill_(-7)
        msa.plan(cfg, w.seq_lens, w.block_table, b.ws)
        msa.index_score_topk(cfg, b.ws, w.idx_q, w.idx_k_pages, b.block_scores, b.selected)
        torch.cuda.synchronize()
        assert torch.equal(a.selected[:T], b.selected[:T])
        for t in range(T):
            pos = int(w.seq_lens[t // spec.q_len]) - spec.q_len + t % spec.q_len
            if pos < 0 or int(w.seq_lens[t // spec.q_len]) == 0:
                continue
            nb = pos // 128 + 1
            assert torch.equal(a.block_scores[t, :, :nb], b.block_scores[t, :, :nb]), t
    assert msa.check_device_error(a.ws) == msa.check_device_error(b.ws)
