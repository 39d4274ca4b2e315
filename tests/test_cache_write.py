"""msa_cache_write against the oracle's cache write (GPU).

The fused K / V / index-key write that precedes attention (sglang
MiniMaxSparseAttnBackend.forward_decode / forward_extend,
set_fused_kv_index_buffer) is byte work: the pools after the write must equal,
byte for byte, the oracle's pools -- rows placed by the plan's block table and
positions, or by explicit out_cache_loc slots; e4m3 pools hold the codes of
x / scale, rounded to nearest even and saturated (planted values beyond +-448
and in the subnormal range); NVFP4 pools hold E2M1 codes under E4M3 block
scales of amax / (6 * scale), keys in slot 2h and values in slot 2h + 1 (a
planted block of exact rounding ties and signed zeros).  Bad slots are flagged
and skipped.  Written and then attended over in one captured CUDA graph, the
step equals eager execution bit for bit and the oracle within the parity
bounds."""
import numpy as np
import pytest
import torch

import block_sparse_paged_msa_gb300 as msa
import oracle
from block_sparse_paged_msa_gb300 import workloads as wl
from gpu_util import compare
from oracle_io import run_oracle, to_np

pytestmark = pytest.mark.gpu


def _rows(spec, T, seed, plant=False):
    k, v, idx_k = wl.new_token_rows(spec, T, seed, device="cuda")
    if plant:   # beyond the e4m3 range after the scale, and e4m3 subnormals
        vals = torch.tensor([20.0, -31.0, 1e-4, -7e-5, 14.0, 0.0, -0.0, 3e-3],
                            device="cuda").to(torch.bfloat16)
        k[0, 0, :8] = vals
        v[-1, -1, -8:] = vals
        # one 16-element block whose quotients are exact E2M1 ties at tensor
        # scale 0.75: amax 3 -> block scale 0.6875, divisor 33/64; plus -0 and 0
        d = 33.0 / 64.0
        tie = torch.tensor([3.0, 0.25 * d, -0.75 * d, 1.25 * d, -1.75 * d, 2.5 * d, 3.5 * d,
                            -5.0 * d, -0.0, 0.0, 0.5 * d, -3.0 * d, 6.0 * d, 4.0 * d, 0.0,
                            -0.0], device="cuda")
        assert torch.equal(tie.to(torch.bfloat16).float(), tie)
        k[min(1, T - 1), 0, 16:32] = tie.to(torch.bfloat16)
    return k, v, idx_k


def _expected(w, k, v, idx_k, slots):
    s = w.spec
    if s.kv_dtype == "nvfp4":    # K and V slots of every head in each pool
        kp = oracle.cache_write_nvfp4(to_np(w.k_pages), slots, to_np(k), s.kv_scale, 0)
        vp = oracle.cache_write_nvfp4(to_np(w.v_pages), slots, to_np(v), s.kv_scale, 1)
        if w.k_pages.data_ptr() == w.v_pages.data_ptr():
            kp = vp = oracle.cache_write_nvfp4(kp, slots, to_np(v), s.kv_scale, 1)
        return kp, vp, oracle.cache_write(to_np(w.idx_k_pages), slots, to_np(idx_k))
    scale = s.kv_scale if s.kv_dtype == "fp8_e4m3" else None
    return (oracle.cache_write(to_np(w.k_pages), slots, to_np(k), e4m3_scale=scale),
            oracle.cache_write(to_np(w.v_pages), slots, to_np(v), e4m3_scale=scale),
            oracle.cache_write(to_np(w.idx_k_pages), slots, to_np(idx_k)))


def _check_pools(w, want):
    for name, exp in zip(("k_pages", "v_pages", "idx_k_pages"), want):
        got = to_np(getattr(w, name))
        assert np.array_equal(got, exp), name


@pytest.mark.parametrize("name", ["medium_decode", "fp8_decode", "nvfp4_decode", "verify",
                                  "prefill", "nvfp4_prefill"])
@pytest.mark.parametrize("explicit_slots", [False, True])
def test_cache_write_bytes_match_oracle(name, explicit_slots):
    spec = wl.small(name, batch=3) if name.endswith("_decode") else wl.small(name)
    w = wl.make_workload(spec, device="cuda")
    cfg = msa.config_for(spec)
    sa = msa.SparseAttention(cfg)
    T = w.num_tokens
    k, v, idx_k = _rows(spec, T, seed=77, plant=True)
    if explicit_slots:   # any distinct slots of the pool (sglang's out_cache_loc)
        g = torch.Generator(device="cuda").manual_seed(5)
        loc = torch.randperm(spec.num_pages * 128, generator=g, device="cuda")[:T]
        slots = loc.tolist()
    else:
        loc = None
        slots = oracle.cache_slots(to_np(w.seq_lens), to_np(w.q_lens), to_np(w.block_table), 128)
    want = _expected(w, k, v, idx_k, slots)
    msa.plan(cfg, w.seq_lens, w.block_table, sa.ws, w.cu_seqlens_q if sa.prefill else None)
    msa.cache_write(cfg, sa.ws, k, v, idx_k, w.k_pages, w.v_pages, w.idx_k_pages,
                    out_cache_loc=loc)
    torch.cuda.synchronize()
    assert msa.check_device_error(sa.ws) == 0
    _check_pools(w, want)


def test_bad_slots_are_flagged_and_skipped():
    spec = wl.small("fp8_decode", batch=3)
    w = wl.make_workload(spec, device="cuda")
    cfg = msa.config_for(spec)
    sa = msa.SparseAttention(cfg)
    k, v, idx_k = _rows(spec, w.num_tokens, seed=78)
    loc = torch.tensor([5 * 128 + 7, spec.num_pages * 128, -3], dtype=torch.int64,
                       device="cuda")
    want = _expected(w, k, v, idx_k, [5 * 128 + 7, -1, -1])
    msa.plan(cfg, w.seq_lens, w.block_table, sa.ws)
    msa.cache_write(cfg, sa.ws, k, v, idx_k, w.k_pages, w.v_pages, w.idx_k_pages,
                    out_cache_loc=loc)
    assert msa.check_device_error(sa.ws) & 1
    _check_pools(w, want)


def test_idle_request_writes_nothing_and_index_key_is_optional():
    spec = wl.small("medium_decode", seq_lens=(900, 0, 300), seq_len_range=None, batch=3,
                    num_pages=40)
    w = wl.make_workload(spec, device="cuda")
    cfg = msa.config_for(spec)
    sa = msa.SparseAttention(cfg)
    k, v, idx_k = _rows(spec, w.num_tokens, seed=79)
    slots = oracle.cache_slots(to_np(w.seq_lens), to_np(w.q_lens), to_np(w.block_table), 128)
    assert slots[1] == -1
    want = _expected(w, k, v, idx_k, slots)
    want = (want[0], want[1], to_np(w.idx_k_pages))      # no index-key write
    msa.plan(cfg, w.seq_lens, w.block_table, sa.ws)
    msa.cache_write(cfg, sa.ws, k, v, None, w.k_pages, w.v_pages, w.idx_k_pages)
    assert msa.check_device_error(sa.ws) == 0
    _check_pools(w, want)


@pytest.mark.parametrize("name", ["medium_decode", "fp8_decode", "nvfp4_decode", "verify"])
def test_write_then_decode_graph_replay_equals_eager_and_oracle(name):
    """The cache write and the whole decode step captured as one CUDA graph;
    replayed on new inputs written in place, it equals eager execution bit for
    bit, and the oracle (fed the pools after the write) within the bounds."""
    base = wl.small(name, batch=3) if name != "verify" else wl.small(name)
    w = wl.make_workload(base, device="cuda")
    cfg = msa.config_for(base)
    T = w.num_tokens
    bufs = {kk: vv.clone() for kk, vv in w.__dict__.items() if isinstance(vv, torch.Tensor)}
    if w.k_pages.data_ptr() == w.v_pages.data_ptr():   # NVFP4: one pool for K and V
        bufs["v_pages"] = bufs["k_pages"]
    rows = [t.clone() for t in _rows(base, T, seed=80)]
    sa = msa.SparseAttention(cfg)

    def step(b, r, s):
        s.run(b["seq_lens"], b["block_table"], b["idx_q"], b["idx_k_pages"], b["q"],
              b["k_pages"], b["v_pages"], new_kv=tuple(r))

    step(bufs, rows, sa)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(graph, stream=st):
            step(bufs, rows, sa)
    torch.cuda.current_stream().wait_stream(st)
    for seed in (301, 302):
        w2 = wl.make_workload(base.replace(seed=seed), device="cuda")
        new = _rows(base, T, seed=seed + 1000)
        for kk, vv in bufs.items():
            vv.copy_(getattr(w2, kk))
        for dst, src in zip(rows, new):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        assert msa.check_device_error(sa.ws) == 0
        eager = msa.SparseAttention(cfg)
        step(w2.__dict__, new, eager)
        torch.cuda.synchronize()
        for kk in ("k_pages", "v_pages", "idx_k_pages"):
            assert torch.equal(bufs[kk].view(torch.uint8), getattr(w2, kk).view(torch.uint8))
        assert torch.equal(sa.selected[:T], eager.selected[:T])
        assert torch.equal(sa.out[:T], eager.out[:T]) and torch.equal(sa.lse[:T], eager.lse[:T])
        compare(w2, eager, run_oracle(w2.to("cpu")))
