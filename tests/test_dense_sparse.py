"""The dense-sparse decode (GPU): msa_compact_selected + msa_paged_decode.

sglang's MiniMaxSparseAttnBackend.forward_decode can turn the selected blocks
into a page table with real sequence lengths and run a dense paged decode over
it (_dense_sparse_main_decode, max_seq_len = topk_blocks * block_size).  Checked
here: the compacted lists bit-exact against the oracle's compaction of the
oracle's own selection; the step's out / lse bit-exact against the sparse
decode (same keys, same order, same splits) and within the bounds against the
oracle; the paged decode on page lists and lengths built by the caller against
the oracle's dense paged attention; bad pages flagged; graph replay == eager."""
import numpy as np
import pytest
import torch

import block_sparse_paged_msa_gb300 as msa
import oracle
from block_sparse_paged_msa_gb300 import workloads as wl
from gpu_util import LSE_MAX, OUT_MAX, OUT_MEAN, compare
from oracle_io import run_oracle, to_np

pytestmark = pytest.mark.gpu


def _spec(name):
    return wl.small(name) if name == "verify" else wl.small(name, batch=3)


def _run(w, dense):
    cfg = msa.config_for(w.spec)
    sa = msa.SparseAttention(cfg, dense_sparse=dense)
    sa.run(w.seq_lens, w.block_table, w.idx_q, w.idx_k_pages, w.q, w.k_pages, w.v_pages)
    torch.cuda.synchronize()
    assert msa.check_device_error(sa.ws) == 0
    return sa


@pytest.mark.parametrize("name", ["medium_decode", "fp8_decode", "nvfp4_decode", "verify",
                                  "long_decode"])
def test_dense_sparse_equals_sparse_and_oracle(name):
    w = wl.make_workload(_spec(name), device="cuda")
    dense, sparse = _run(w, True), _run(w, False)
    T = w.num_tokens
    ref = run_oracle(w.to("cpu"))
    # compaction of the oracle's own selection
    toks = oracle.query_positions(to_np(w.seq_lens), to_np(w.q_lens))
    bt = to_np(w.block_table)
    pt, dl = dense.page_table[:T].cpu().numpy(), dense.dense_len[:T].cpu().numpy()
    S = pt.shape[-1]
    for t, (r, p) in enumerate(toks):
        for h in range(w.spec.num_kv_heads):
            pages, n = oracle.compact_selection(ref["selected"][(t, h)], bt[r], p, 128)
            assert pt[t, h].tolist() == pages + [-1] * (S - len(pages)), (t, h)
            assert dl[t, h] == n, (t, h)
    assert torch.equal(dense.out[:T], sparse.out[:T]) and torch.equal(dense.lse[:T], sparse.lse[:T])
    compare(w, dense, ref)


def test_paged_decode_on_caller_page_lists():
    """A dense paged decode over page lists and lengths that no selection made:
    distinct random pages, random lengths up to S * 128 (0 included)."""
    spec = wl.small("medium_decode", batch=4, num_q_heads=16, num_kv_heads=2)
    w = wl.make_workload(spec, device="cuda")
    cfg = msa.config_for(spec)
    sa = msa.SparseAttention(cfg, dense_sparse=True)
    T, H, S = w.num_tokens, spec.num_kv_heads, sa.width
    g = torch.Generator(device="cuda").manual_seed(17)
    pt = torch.stack([torch.randperm(spec.num_pages, generator=g, device="cuda")[:S]
                      for _ in range(T * H)]).view(T, H, S).to(torch.int32)
    lens = torch.randint(0, S * 128 + 1, (T, H), generator=g, device="cuda", dtype=torch.int32)
    lens[0, 0], lens[1, 1] = 0, S * 128
    msa.plan(cfg, w.seq_lens, w.block_table, sa.ws)
    msa.paged_decode(cfg, sa.ws, w.q, w.k_pages, w.v_pages, pt, lens)
    msa.combine(cfg, sa.ws, sa.out, sa.lse)
    torch.cuda.synchronize()
    assert msa.check_device_error(sa.ws) == 0
    q, kp, vp = to_np(w.q), to_np(w.k_pages), to_np(w.v_pages)
    out, lse = to_np(sa.out[:T]), sa.lse[:T].cpu().numpy().astype(np.float64)
    G, errs, lerrs = spec.group, [], []
    for t in range(T):
        for h in range(H):
            n = int(lens[t, h])
            pages = pt[t, h, :(n + 127) // 128].tolist()
            o, l = oracle.paged_attention(q[t, h * G:(h + 1) * G], kp, vp, pages, n, h,
                                          spec.softmax_scale, 128)
            errs.append(np.abs(out[t, h * G:(h + 1) * G] - o).ravel())
            if n == 0:
                assert np.all(np.isneginf(lse[t, h * G:(h + 1) * G]))
            else:
                lerrs.append(np.abs(lse[t, h * G:(h + 1) * G] - l))
    e, le = np.concatenate(errs), np.concatenate(lerrs)
    assert e.max() <= OUT_MAX and e.mean() <= OUT_MEAN and le.max() <= LSE_MAX, (e.max(), e.mean())


def test_paged_decode_flags_pages_outside_the_pool():
    spec = wl.small("medium_decode", batch=2)
    w = wl.make_workload(spec, device="cuda")
    sa = _run(w, True)
    sa.page_table[0, 0, 1] = spec.num_pages + 2
    cfg = sa.cfg
    msa.paged_decode(cfg, sa.ws, w.q, w.k_pages, w.v_pages, sa.page_table, sa.dense_len)
    assert msa.check_device_error(sa.ws) & 1


def test_dense_sparse_graph_replay_equals_eager():
    base = wl.small("medium_decode", batch=3)
    w = wl.make_workload(base, device="cuda")
    cfg = msa.config_for(base)
    sa = msa.SparseAttention(cfg, dense_sparse=True)
    bufs = {k: v.clone() for k, v in w.__dict__.items() if isinstance(v, torch.Tensor)}
    args = lambda b: (b["seq_lens"], b["block_table"], b["idx_q"], b["idx_k_pages"], b["q"],  # noqa
                      b["k_pages"], b["v_pages"])
    sa.run(*args(bufs))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(graph, stream=st):
            sa.run(*args(bufs))
    torch.cuda.current_stream().wait_stream(st)
    for seed in (401, 402):
        w2 = wl.make_workload(base.replace(seed=seed), device="cuda")
        for k, v in bufs.items():
            v.copy_(getattr(w2, k))
        graph.replay()
        torch.cuda.synchronize()
        eager = _run(w2, True)
        T = w2.num_tokens
        assert torch.equal(sa.page_table[:T], eager.page_table[:T])
        assert torch.equal(sa.out[:T], eager.out[:T]) and torch.equal(sa.lse[:T], eager.lse[:T])
