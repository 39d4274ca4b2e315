"""The seeded input generator: determinism and the stated structure."""
import torch

from block_sparse_paged_msa_gb300 import workloads as wl


def test_seed_names_one_input_set():
    a = wl.make_workload(wl.small("medium_decode"))
    b = wl.make_workload(wl.small("medium_decode"))
    for f in ("seq_lens", "block_table", "idx_q", "idx_k_pages", "q", "k_pages", "v_pages"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f


def test_structure():
    spec = wl.small("medium_decode")
    w = wl.make_workload(spec)
    lo, hi = spec.seq_len_range
    assert w.seq_lens.dtype == torch.int32
    assert int(w.seq_lens.min()) >= lo and int(w.seq_lens.max()) <= hi
    used = []
    for r in range(spec.batch):
        nb = -(-int(w.seq_lens[r]) // 128)
        row = w.block_table[r]
        assert bool((row[:nb] >= 0).all()) and bool((row[nb:] == -1).all())
        used += row[:nb].tolist()
    assert len(set(used)) == len(used) and max(used) < spec.num_pages
    iq = w.idx_q.float()
    assert torch.equal(iq, iq.round()) and iq.abs().max() <= 4
    ik = w.idx_k_pages.float()
    assert torch.equal(ik, ik.round()) and ik.abs().max() <= 4 and ik.min() == -4
    assert w.q.shape == (spec.batch, spec.num_q_heads, 128)
    assert w.k_pages.shape == (spec.num_pages, spec.num_kv_heads, 128, 128)
    assert abs(float(w.k_pages.float().std()) - 1.0) < 0.01


def test_tiny_decode_matches_its_recipe():
    w = wl.make_workload(wl.WORKLOADS["tiny_decode"])
    assert w.seq_lens.tolist() == [1000, 1500]
    assert w.idx_q.shape == (2, 1, 64) and w.q.shape == (2, 8, 128)
    # 8 + 12 pages drawn from a permutation of the 32-page pool
    assert sorted(w.block_table[w.block_table >= 0].tolist()) != list(range(20))


def test_fp8_pool_codes():
    spec = wl.small("fp8_decode", batch=1, num_pages=40)
    w = wl.make_workload(spec)
    assert w.k_pages.dtype == torch.float8_e4m3fn
    x = w.k_pages.float() * spec.kv_scale
    assert abs(float(x.std()) - 1.0) < 0.02
    assert float(w.k_pages.float().abs().max()) < 448


def test_prefill_and_verify_geometry():
    w = wl.make_workload(wl.small("prefill"), kv_pool=False)
    assert w.cu_seqlens_q.tolist() == [0, 300, 600]
    w = wl.make_workload(wl.small("verify"), kv_pool=False)
    assert w.q_lens.tolist() == [4] * 4 and w.idx_q.shape[0] == 16
