"""CUDA path vs the fp64 oracle for decode and speculative verify (GPU).

Selections and block scores are compared bit-exactly (integer-valued index
vectors make every dot product exact in fp32 and fp64); out and LSE within the
bounds in gpu_util.  Small cases span several blocks and ragged last pages and
are compared on every element; the full-size medium decode (batch 32, seq_lens
8k..32k, 64/8 heads), long decode (batch 128, seq_lens 64k..128k, a 114 688-page
pool: 90 GB of K, V and index keys), fp8 decode and verify run in the launch
configuration the bench times and are compared on sampled (token, KV head)
pairs."""
import numpy as np
import pytest
import torch

import block_sparse_paged_msa_gb300 as msa
from block_sparse_paged_msa_gb300 import workloads as wl
from gpu_util import compare, compare_sampled, run_gpu
from oracle_io import run_oracle

pytestmark = pytest.mark.gpu


def _full_case(spec):
    w = wl.make_workload(spec, device="cuda")
    sa = run_gpu(w)
    assert msa.check_device_error(sa.ws) == 0
    return compare(w, sa, run_oracle(w.to("cpu")))


@pytest.mark.parametrize("name", ["tiny_decode", "medium_decode", "fp8_decode", "nvfp4_decode",
                                  "long_decode", "verify"])
def test_small_workloads_every_element(name):
    spec = wl.WORKLOADS[name] if name == "tiny_decode" else wl.small(name)
    print(name, _full_case(spec))


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_random_seeds_ragged(seed):
    spec = wl.small("medium_decode", seed=seed, batch=5, seq_len_range=(1, 2200),
                    num_pages=120)
    _full_case(spec)


def test_group_16_and_index_dim_64():
    spec = wl.small("medium_decode", num_q_heads=32, num_kv_heads=2, index_dim=64, batch=3)
    _full_case(spec)


def test_group_1_and_topk_0():
    spec = wl.small("medium_decode", num_q_heads=4, num_kv_heads=4, topk_blocks=0, batch=3)
    _full_case(spec)


@pytest.mark.parametrize("bps", [1, 2, 7, 32])
def test_split_sizes_agree(bps):
    spec = wl.small("medium_decode", batch=3)
    w = wl.make_workload(spec, device="cuda")
    ref = run_oracle(w.to("cpu"))
    sa = run_gpu(w, blocks_per_split=bps)
    compare(w, sa, ref)


@pytest.mark.parametrize("name", ["medium_decode", "verify"])
def test_step_batch_below_config_max(name):
    """A step of 3 requests on a config sized for 8: the work items of the
    missing tokens are skipped (no selected row of theirs is read); q and idx_q
    are padded to the config's token count, as the binding requires."""
    spec = (wl.small(name, batch=3) if name != "verify"
            else wl.small(name, batch=3, seq_lens=(1500, 2000, 3001)))
    w = wl.make_workload(spec, device="cuda")
    ref = run_oracle(w.to("cpu"))
    cfg = msa.config_for(spec, max_batch=8)
    sa = msa.SparseAttention(cfg)
    T, Tmax = w.num_tokens, msa.ops.max_tokens(cfg)
    q = torch.full((Tmax,) + tuple(w.q.shape[1:]), float("nan"), dtype=w.q.dtype, device="cuda")
    idx_q = torch.zeros((Tmax,) + tuple(w.idx_q.shape[1:]), dtype=w.idx_q.dtype, device="cuda")
    q[:T] = w.q
    idx_q[:T] = w.idx_q
    sa.run(w.seq_lens, w.block_table, idx_q, w.idx_k_pages, q, w.k_pages, w.v_pages)
    torch.cuda.synchronize()
    assert msa.check_device_error(sa.ws) == 0
    print(compare(w, sa, ref))


def test_block_boundaries_and_short_requests():
    # exact multiples of the block, one token, within init+local, one past a block
    spec = wl.small("medium_decode", seq_lens=(128, 1, 384, 129, 1024, 255), seq_len_range=None,
                    batch=6, num_pages=64)
    _full_case(spec)


def test_medium_decode_full_size_sampled():
    spec = wl.WORKLOADS["medium_decode"]
    w = wl.make_workload(spec, device="cuda")
    sa = run_gpu(w)
    assert msa.check_device_error(sa.ws) == 0
    rng = np.random.default_rng(0)
    samples = [(int(t), int(h)) for t, h in zip(rng.integers(0, spec.batch, 6),
                                                 rng.integers(0, spec.num_kv_heads, 6))]
    samples += [(0, 0), (spec.batch - 1, spec.num_kv_heads - 1)]
    print(compare_sampled(w, sa, samples))
    # properties that hold everywhere: selection sizes and bounds
    P = 128
    nb = (w.seq_lens.long() + P - 1) // P
    sel = sa.selected[:spec.batch].long()
    width = sel.shape[-1]
    assert bool((sel[..., :width] >= -1).all())
    assert bool(((sel >= 0).sum(-1) == torch.clamp(nb, max=width)[:, None]).all())
    assert torch.isfinite(sa.out[:spec.batch].float()).all()


def test_verify_full_size_sampled():
    spec = wl.WORKLOADS["verify"]
    w = wl.make_workload(spec, device="cuda")
    sa = run_gpu(w)
    assert msa.check_device_error(sa.ws) == 0
    samples = [(0, 0), (1, 3), (2, 7), (3, 5), (255, 7), (128, 2)]
    print(compare_sampled(w, sa, samples))


@pytest.mark.parametrize("name,samples", [
    ("long_decode", [(0, 0), (127, 7), (37, 3), (64, 5), (100, 1), (5, 6)]),
    ("fp8_decode", [(0, 0), (31, 7), (9, 3), (17, 5), (25, 1), (4, 6)]),
    ("nvfp4_decode", [(0, 0), (31, 7), (9, 3), (17, 5), (25, 1), (4, 6)]),
])
def test_full_size_sampled(name, samples):
    spec = wl.WORKLOADS[name]
    w = wl.make_workload(spec, device="cuda")
    sa = run_gpu(w)
    assert msa.check_device_error(sa.ws) == 0
    print(name, compare_sampled(w, sa, samples))
    del w, sa
    torch.cuda.empty_cache()


@pytest.mark.parametrize("q_len,seq_lens", [(1, (140000, 131300)), (4, (139001, 133004))])
def test_requests_beyond_1024_blocks_every_element(q_len, seq_lens):
    """Requests longer than 1 024 blocks (131 072 tokens) take the CTA-wide
    radix select of msa_topk_select instead of the warp one; with 1 KV head
    and 8 query heads the oracle checks every selection, every block score and
    every output element.  Integer-valued index vectors make tied block scores
    common among the ~1 000 candidates, so the tie rule is exercised."""
    spec = wl.WORKLOADS["medium_decode"].replace(
        name="beyond_1024_blocks", batch=2, seq_lens=seq_lens, seq_len_range=None,
        q_len=q_len, num_q_heads=8, num_kv_heads=1, num_pages=2200, seed=1101 + q_len)
    assert spec.max_blocks > 1024
    w = wl.make_workload(spec, device="cuda")
    sa = run_gpu(w)
    assert msa.check_device_error(sa.ws) == 0
    print(compare(w, sa, run_oracle(w.to("cpu"))))


@pytest.mark.parametrize("q_len", [2, 3, 4])
@pytest.mark.parametrize("index_dim", [64, 128])
def test_verify_q_len_and_index_dim_every_element(q_len, index_dim):
    """Speculative verify with 2, 3 or 4 new tokens per request: the index
    scores run on the tensor-core kernel (keys as M = 128, the request's query
    rows as N); block scores and selections bit-exact, every output element
    within the bounds.  Draft positions straddle block boundaries (ragged
    lengths), so the per-token causal limits inside the last block differ."""
    spec = wl.small("verify", q_len=q_len, index_dim=index_dim,
                    seq_lens=(1500, 127 + q_len, 2600, 3001, 256 + 1), batch=5, num_pages=128,
                    seed=1200 + 10 * q_len + index_dim // 64)
    _full_case(spec)


def test_verify_bad_page_flagged_and_scored_minus_inf():
    spec = wl.small("verify", batch=4)
    w = wl.make_workload(spec, device="cuda")
    w.block_table[2, 3] = spec.num_pages + 9
    sa = run_gpu(w)
    assert msa.check_device_error(sa.ws) & 1
    # the other requests are exact
    ref = run_oracle(w.to("cpu"), tokens=list(range(0, 8)) + list(range(12, 16)))
    compare(w, sa, ref, tokens=list(range(0, 8)) + list(range(12, 16)))


@pytest.mark.parametrize("q_len", [1, 4])
def test_nvfp4_group_16_index_64_and_verify_every_element(q_len):
    """NVFP4 slots with 16 query heads per KV head, index dim 64, and four
    speculative tokens per request (ragged, straddling a block boundary)."""
    spec = wl.small("nvfp4_decode", num_q_heads=32, num_kv_heads=2, index_dim=64, q_len=q_len,
                    seq_lens=(700, 127 + q_len, 2900), seq_len_range=None, batch=3,
                    num_pages=64, seed=1300 + q_len)
    _full_case(spec)


@pytest.mark.parametrize("groups", [(32, 2), (4, 4)], ids=["g16", "g1"])
@pytest.mark.parametrize("q_len", [1, 4])
def test_fp8_groups_and_verify_every_element(groups, q_len):
    """e4m3 K/V with 16 query heads per KV head (index dim 64) or one, alone and
    with four speculative tokens per request (ragged, straddling a block
    boundary): K feeds the fp16 MMAs from the tile, V is converted per warp,
    k_scale / v_scale fold into the softmax scale and the output."""
    hq, hkv = groups
    spec = wl.small("fp8_decode", num_q_heads=hq, num_kv_heads=hkv,
                    index_dim=64 if hq // hkv == 16 else 128, q_len=q_len,
                    seq_lens=(700, 127 + q_len, 2900), seq_len_range=None, batch=3,
                    num_pages=64, seed=1400 + 10 * q_len + hq)
    _full_case(spec)


def _combo(seed):
    """A seeded draw of one small decode / verify configuration."""
    rng = np.random.default_rng(seed)
    kv = ["medium_decode", "fp8_decode", "nvfp4_decode"][int(rng.integers(3))]
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 8, 16]))
    q_len = int(rng.integers(1, 5))
    batch = int(rng.integers(1, 5))
    lens = tuple(int(x) for x in rng.integers(q_len, 2600, size=batch))
    return dict(name=kv, num_q_heads=g * hkv, num_kv_heads=hkv, q_len=q_len,
                index_dim=int(rng.choice([64, 128])), topk_blocks=int(rng.choice([0, 3, 16])),
                seq_lens=lens, seq_len_range=None, batch=batch, num_pages=96, seed=seed)


@pytest.mark.parametrize("seed", range(1500, 1512))
def test_random_configuration_sweep_every_element(seed):
    """Seeded draws over KV type (bf16, e4m3, NVFP4), query heads per KV head
    (1..16), KV heads, new tokens per request (1..4, verify from 2), index dim,
    top-k (0, 3, 16) and ragged lengths: every combination the kernels accept
    agrees with the oracle on every element."""
    kw = _combo(seed)
    spec = wl.small(kw.pop("name"), **kw)
    _full_case(spec)
