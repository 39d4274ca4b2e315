"""Chunked prefill: CUDA path vs the fp64 oracle (GPU).

Per-token block scores and selections bit-exact; the key-block -> query CSR
identical to the oracle's (built from the same selections); out / lse within
the parity bounds.  Small chunks are compared on every element; the full-size
prefill (4 requests x (16384 cached + 2048 new) tokens) on sampled pairs plus
structural CSR properties over every row."""
import numpy as np
import pytest
import torch

import block_sparse_paged_msa_gb300 as msa
import oracle
from block_sparse_paged_msa_gb300 import workloads as wl
from gpu_util import BF16_OUT_REL, compare, compare_sampled, run_gpu
from oracle_io import run_oracle, to_np

pytestmark = pytest.mark.gpu


def _csr_matches_oracle(w, sa):
    spec = w.spec
    T = w.num_tokens
    sel = sa.selected[:T].cpu().numpy().astype(np.int64)
    tok_req = np.repeat(np.arange(spec.batch), w.q_lens.cpu().numpy())
    rp, qi = oracle.build_k2q_csr(sel, tok_req, spec.batch, spec.max_blocks)
    got_rp = sa.row_ptr.cpu().numpy().astype(np.int64)
    assert np.array_equal(got_rp, rp)
    assert np.array_equal(sa.q_indices[:len(qi)].cpu().numpy().astype(np.int64), qi)


@pytest.mark.parametrize("kw", [dict(), dict(num_q_heads=32, num_kv_heads=2),
                                dict(num_q_heads=16, num_kv_heads=4, index_dim=64),
                                dict(seq_lens=(700, 129), q_len=129, topk_blocks=2),
                                dict(num_q_heads=4, num_kv_heads=4),
                                dict(num_q_heads=8, num_kv_heads=4, seq_lens=(300, 1100))],
                         ids=["g8", "g16", "g4_d64", "chunk129_topk2", "g1", "g2"])
def test_small_prefill_every_element(kw):
    spec = wl.small("prefill", **kw)
    w = wl.make_workload(spec, device="cuda")
    sa = run_gpu(w)
    assert sa.prefill
    assert msa.check_device_error(sa.ws) == 0
    print(compare(w, sa, run_oracle(w.to("cpu"))))
    _csr_matches_oracle(w, sa)


@pytest.mark.parametrize("kw", [dict(), dict(num_q_heads=16, num_kv_heads=4, index_dim=64),
                                dict(seq_lens=(700, 129), q_len=129, topk_blocks=2)],
                         ids=["g8", "g4_d64", "chunk129_topk2"])
def test_small_nvfp4_prefill_every_element(kw):
    """NVFP4 KV (E2M1 codes with E4M3 block scales, a key and a value slot per
    KV head) in the prefill tiles: each CSR row's slots are dequantised in
    shared memory (keys to bf16, values to fp16, both exact) with k_scale in
    the softmax scale and v_scale on the output; compared on every element
    with the oracle fed the same dequantised pool."""
    spec = wl.small("nvfp4_prefill", **kw)
    w = wl.make_workload(spec, device="cuda")
    sa = run_gpu(w)
    assert sa.prefill
    assert msa.check_device_error(sa.ws) == 0
    print(compare(w, sa, run_oracle(w.to("cpu"))))
    _csr_matches_oracle(w, sa)


@pytest.mark.parametrize("half,mult", [(1, 2.5), (1, 12.0), (0, 12.0)],
                         ids=["late_x2.5", "late_x12", "early_x12"])
def test_prefill_score_spread_across_a_block(half, mult):
    """Keys 64..127 (or 0..63) of every page scaled up: a tile row's later
    64-key chunk then tops the first chunk's max by far (x12: the softmax
    reference moves up and the first chunk's P is rescaled), by about the
    rescale threshold (x2.5: both paths, P values up to 4 against a stale
    reference), or the first chunk dominates (early).  Compared on every
    element; the peaked softmax returns near single value rows (|o| up to
    ~4.5), so the max bound carries the bf16 output rounding allowance."""
    spec = wl.small("prefill")
    w = wl.make_workload(spec, device="cuda")
    sl = slice(64, 128) if half else slice(0, 64)
    w.k_pages[:, :, sl, :] = (w.k_pages[:, :, sl, :].float() * mult).to(torch.bfloat16)
    sa = run_gpu(w)
    assert msa.check_device_error(sa.ws) == 0
    print(compare(w, sa, run_oracle(w.to("cpu")), out_rel=BF16_OUT_REL))


def test_prefill_whole_sequence_is_dense_causal():
    """A chunk that is the whole sequence with top-k covering every block is
    plain causal attention."""
    spec = wl.small("prefill", seq_lens=(600,), q_len=600, batch=1, topk_blocks=16,
                    num_pages=8)
    w = wl.make_workload(spec, device="cuda")
    sa = run_gpu(w)
    ref = run_oracle(w.to("cpu"))
    compare(w, sa, ref)
    for (t, h), s in ref["selected"].items():
        assert s == list(range(t // 128 + 1))


@pytest.mark.parametrize("name", ["prefill", "nvfp4_prefill"])
def test_prefill_full_size_sampled(name):
    spec = wl.WORKLOADS[name]
    w = wl.make_workload(spec, device="cuda")
    sa = run_gpu(w)
    assert msa.check_device_error(sa.ws) == 0
    samples = [(0, 0), (2047, 7), (2048, 3), (4100, 1), (6000, 5), (8191, 2)]
    print(compare_sampled(w, sa, samples))
    # CSR structure over every row: sizes add up to the selections, each row
    # ascending and inside its request, every entry's selection holds the block
    T = w.num_tokens
    sel = sa.selected[:T]
    rp = sa.row_ptr.long()
    total = int(rp[-1])
    assert total == int((sel >= 0).sum())
    assert bool((rp[1:] >= rp[:-1]).all())
    qi = sa.q_indices[:total].long()
    rows = torch.repeat_interleave(torch.arange(rp.numel() - 1, device="cuda"), rp[1:] - rp[:-1])
    NB, B = spec.max_blocks, spec.batch
    j = rows % NB
    r = (rows // NB) % B
    h = rows // (NB * B)
    assert bool((qi // spec.q_len == r).all())
    same_row = rows[1:] == rows[:-1]
    assert bool((qi[1:][same_row] > qi[:-1][same_row]).all())
    assert bool((sel[qi, h] == j[:, None]).any(-1).all())
    assert torch.isfinite(sa.out[:T].float()).all()


@pytest.mark.parametrize("name", ["prefill", "nvfp4_prefill"])
def test_prefill_graph_replay_equals_eager(name):
    base = wl.small(name)
    w = wl.make_workload(base, device="cuda")
    cfg = msa.config_for(base)
    sa = msa.SparseAttention(cfg)
    bufs = {k: v.clone() for k, v in w.__dict__.items() if isinstance(v, torch.Tensor)}
    args = lambda: (bufs["seq_lens"], bufs["block_table"], bufs["idx_q"], bufs["idx_k_pages"],
                    bufs["q"], bufs["k_pages"], bufs["v_pages"])
    sa.run(*args(), cu_seqlens_q=bufs["cu_seqlens_q"])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            sa.run(*args(), cu_seqlens_q=bufs["cu_seqlens_q"])
    torch.cuda.current_stream().wait_stream(s)
    for seed in (201, 202):
        w2 = wl.make_workload(base.replace(seed=seed), device="cuda")
        for k, v in bufs.items():
            v.copy_(getattr(w2, k))
        graph.replay()
        torch.cuda.synchronize()
        g_out, g_lse, g_rp = sa.out.clone(), sa.lse.clone(), sa.row_ptr.clone()
        eager = msa.SparseAttention(cfg)
        eager.run(w2.seq_lens, w2.block_table, w2.idx_q, w2.idx_k_pages, w2.q, w2.k_pages,
                  w2.v_pages, cu_seqlens_q=w2.cu_seqlens_q)
        torch.cuda.synchronize()
        T = w2.num_tokens
        assert torch.equal(g_rp, eager.row_ptr)
        assert torch.equal(g_out[:T], eager.out[:T]) and torch.equal(g_lse[:T], eager.lse[:T])


def _pcombo(seed):
    """A seeded draw of one small chunked-prefill configuration."""
    rng = np.random.default_rng(seed)
    kv = ["prefill", "nvfp4_prefill"][int(rng.integers(2))]
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 8, 16]))
    q_len = int(rng.choice([5, 64, 129, 300]))
    batch = int(rng.integers(1, 4))
    lens = tuple(int(x) for x in rng.integers(q_len, 1800, size=batch))
    return dict(name=kv, num_q_heads=g * hkv, num_kv_heads=hkv, q_len=q_len,
                index_dim=int(rng.choice([64, 128])), topk_blocks=int(rng.choice([0, 2, 16])),
                seq_lens=lens, batch=batch, num_pages=64, seed=seed)


@pytest.mark.parametrize("seed", range(1600, 1608))
def test_random_prefill_sweep_every_element(seed):
    """Seeded draws over KV type (bf16, NVFP4), query heads per KV head, KV
    heads, chunk length (5 .. 300 new tokens per request), index dim, top-k and
    ragged prefixes: every element agrees with the oracle, and the CSR with the
    oracle's."""
    kw = _pcombo(seed)
    spec = wl.small(kw.pop("name"), **kw)
    w = wl.make_workload(spec, device="cuda")
    sa = run_gpu(w)
    assert sa.prefill
    assert msa.check_device_error(sa.ws) == 0
    print(compare(w, sa, run_oracle(w.to("cpu"))))
    _csr_matches_oracle(w, sa)
