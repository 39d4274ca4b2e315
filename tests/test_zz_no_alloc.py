"""msa_sparse_decode_noalloc: the decode step for callers that cannot allocate
device memory (their framework's allocator owns all of it, HBM is reserved for
the KV cache, or cudaMalloc is not acceptable on the call's path).

Called through the C ABI with no workspace, twice in a row (the second call
runs on scratch left by the first), it must give the same out / lse, bit for
bit, as the workspace-based entry points: the same kernels run with the same
fixed split order.  Steps too large for its fixed scratch are refused before
any launch; bad data found on the device is reported through
msa_noalloc_check_device_error; a captured call replays to the eager result.
Collected last so that a failure here never hides another test's result."""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_paged_msa_gb300 as msa
from block_sparse_paged_msa_gb300 import ops
from block_sparse_paged_msa_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _noalloc(cfg, w, selected, out, lse):
    st = ops.lib().msa_sparse_decode_noalloc(
        ctypes.byref(cfg), w.seq_lens.shape[0], w.seq_lens.data_ptr(), w.block_table.data_ptr(),
        w.block_table.shape[1], w.q.data_ptr(), w.k_pages.data_ptr(), w.v_pages.data_ptr(),
        selected.data_ptr(), out.data_ptr(), lse.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0, ops.status_string(st)


def _close(a_out, a_lse, b_out, b_lse):
    assert torch.equal(a_out, b_out)
    assert torch.equal(a_lse, b_lse)


@pytest.mark.parametrize("first,second", [("medium_decode", "fp8_decode"),
                                          ("nvfp4_decode", "medium_decode")])
def test_noalloc_matches_workspace_path_two_calls(first, second):
    for name in (first, second):
        spec = wl.small(name, batch=4)
        w = wl.make_workload(spec, device="cuda")
        cfg = msa.config_for(spec)
        assert msa.workspace_bytes(cfg) <= ops.NOALLOC_SCRATCH_BYTES
        ref = msa.SparseAttention(cfg)
        ref.run(w.seq_lens, w.block_table, w.idx_q, w.idx_k_pages, w.q, w.k_pages, w.v_pages)
        T = w.num_tokens
        for call in range(2):
            out = torch.full_like(ref.out[:T], float("nan"))
            lse = torch.full_like(ref.lse[:T], float("nan"))
            _noalloc(cfg, w, ref.selected, out, lse)
            torch.cuda.synchronize()
            _close(out, lse, ref.out[:T], ref.lse[:T])


def test_noalloc_full_size_medium_decode():
    spec = wl.WORKLOADS["medium_decode"]
    w = wl.make_workload(spec, device="cuda")
    cfg = msa.config_for(spec)
    ref = msa.SparseAttention(cfg)
    ref.run(w.seq_lens, w.block_table, w.idx_q, w.idx_k_pages, w.q, w.k_pages, w.v_pages)
    T = w.num_tokens
    for _ in range(2):
        out = torch.empty_like(ref.out[:T])
        lse = torch.empty_like(ref.lse[:T])
        msa.ops.sparse_decode_noalloc(cfg, w.seq_lens, w.block_table, w.q, w.k_pages, w.v_pages,
                                      ref.selected, out, lse)
        torch.cuda.synchronize()
        _close(out, lse, ref.out[:T], ref.lse[:T])


def test_noalloc_refuses_steps_beyond_its_scratch():
    spec = wl.small("medium_decode", batch=4)
    w = wl.make_workload(spec, device="cuda")
    big = msa.config_for(spec, max_batch=4096, blocks_per_split=1)
    assert msa.workspace_bytes(big) > ops.NOALLOC_SCRATCH_BYTES
    out = torch.zeros((4, 64, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((4, 64), dtype=torch.float32, device="cuda")
    sel = torch.zeros((4, 8, 20), dtype=torch.int32, device="cuda")
    with pytest.raises(msa.MsaError, match="UNSUPPORTED"):
        msa.ops.sparse_decode_noalloc(big, w.seq_lens, w.block_table, w.q, w.k_pages, w.v_pages,
                                      sel, out, lse)
    assert bool((out == 0).all())


def test_noalloc_reports_device_errors():
    """A page id outside the pool is flagged in the scratch's error words (no
    fault) and read back without a workspace; the next clean call clears it."""
    spec = wl.small("medium_decode", batch=3)
    w = wl.make_workload(spec, device="cuda")
    cfg = msa.config_for(spec)
    ref = msa.SparseAttention(cfg)
    ref.run(w.seq_lens, w.block_table, w.idx_q, w.idx_k_pages, w.q, w.k_pages, w.v_pages)
    T = w.num_tokens
    out = torch.empty_like(ref.out[:T])
    lse = torch.empty_like(ref.lse[:T])
    bad = w.block_table.clone()
    bad[1, 0] = spec.num_pages + 3
    msa.ops.sparse_decode_noalloc(cfg, w.seq_lens, bad, w.q, w.k_pages, w.v_pages,
                                  ref.selected, out, lse)
    assert msa.ops.noalloc_check_device_error() & 1
    msa.ops.sparse_decode_noalloc(cfg, w.seq_lens, w.block_table, w.q, w.k_pages, w.v_pages,
                                  ref.selected, out, lse)
    assert msa.ops.noalloc_check_device_error() == 0
    _close(out, lse, ref.out[:T], ref.lse[:T])


def test_noalloc_graph_replay_equals_eager():
    """One eager call first (it looks up the scratch address), then a call
    captured in a CUDA graph; replays on new inputs written in place equal
    eager calls bit for bit."""
    base = wl.small("medium_decode", batch=4)
    w = wl.make_workload(base, device="cuda")
    cfg = msa.config_for(base)
    sel_src = msa.SparseAttention(cfg)
    sel_src.run(w.seq_lens, w.block_table, w.idx_q, w.idx_k_pages, w.q, w.k_pages, w.v_pages)
    T = w.num_tokens
    bufs = {k: getattr(w, k).clone() for k in ("seq_lens", "block_table", "q", "k_pages",
                                               "v_pages")}
    sel = sel_src.selected.clone()
    out = torch.empty_like(sel_src.out[:T])
    lse = torch.empty_like(sel_src.lse[:T])

    def call():
        msa.ops.sparse_decode_noalloc(cfg, bufs["seq_lens"], bufs["block_table"], bufs["q"],
                                      bufs["k_pages"], bufs["v_pages"], sel, out, lse)

    call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            call()
    torch.cuda.current_stream().wait_stream(s)
    for seed in (201, 202):
        w2 = wl.make_workload(base.replace(seed=seed), device="cuda")
        e = msa.SparseAttention(cfg)
        e.run(w2.seq_lens, w2.block_table, w2.idx_q, w2.idx_k_pages, w2.q, w2.k_pages,
              w2.v_pages)
        for k, v in bufs.items():
            v.copy_(getattr(w2, k))
        sel.copy_(e.selected)
        graph.replay()
        torch.cuda.synchronize()
        assert msa.ops.noalloc_check_device_error() == 0
        _close(out, lse, e.out[:T], e.lse[:T])
