"""Benchmark: block-sparse paged MSA decode on GB300.

Headline: one step = the whole decode path for one batch (plan -> index score
-> top-k select -> sparse decode -> combine) on the medium decode workload:
batch 32, seq_lens uniform in [8192, 32768], 64 query / 8 KV heads, head dim
128, block 128, init 1 + local 3 + top-16 blocks, index dim 128, 16384-page
pool.  Inputs are resident in HBM (1.6 GB touched per step, well above the
129 MB L2, so no flush is needed).  The same run then measures every other
configuration (chunked prefill, fp8 KV decode, speculative verify, long-context
decode) under the "workloads" key, and times the fp64 oracle on the host cores
(all of them, and one alone) as the CPU baseline.  Prints one JSON line
(rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload medium_decode|long_decode|fp8_decode|verify|prefill|tiny_decode]
                  [--others LIST|none] [--no-cpu-baseline]

N > 1 runs N independent replicas (one per GPU, launched by torchrun); the
path needs no exchange between GPUs.  ``--impl reference`` times the fp64 CPU
oracle on every host core instead (one (token, KV head) pair per core per step).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

# The oracle legs run single-threaded BLAS; set before numpy loads.
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_sparse_paged_msa_gb300 import workloads as wl  # noqa: E402

METRIC = "sparse-decode query-tokens/s"


def max_over_ranks(values, world, device):
    """Each timing's maximum over the ranks (the slowest replica sets the job
    time); a collective on timings only, none on the data path."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def replica_throughput(units_per_step, world, steps, ms):
    """Whole-job throughput of `world` independent replicas, each processing
    units_per_step per step, over `steps` steps taking `ms` (the slowest rank's)."""
    return units_per_step * world * steps / (ms / 1e3)

UNIT = "q-tokens/s"
FALLBACK_HBM_GBS = 6800.0

# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant
# kernel, from the ncu captures summarised in profiles/ (None until captured for
# the current kernel).
NCU_TRAFFIC_BYTES = {
    # batch-8 / 2048-page capture of the current kernel (half-tile units):
    # 371.6 MB (368.3 read + 3.4 written) for 367.7 MB algorithmic, scaled by
    # bytes to a full medium-decode launch (1.2608 GB)
    ("medium_decode", "index_score"): 1.2743e9,
    # full-size one-pass capture of the prefill tile kernel (work items of 20
    # M-tiles taken request by request): 649.1 MB read (Q gathers mostly L2
    # hits, K/V tiles) + 2 666.3 MB written (the fp16 partials)
    ("prefill", "sparse_prefill"): 3.3154e9,
}


# ----------------------------------------------------------------- helpers
def algorithmic_bytes(w: wl.Workload):
    """Bytes a step must move at minimum, by kernel.

    index score: every visible index key once per request and KV head
                 (L_r * H_kv * d * 2 bytes), the index queries, and one fp32
                 score per (token, head, visible block);
    decode:      the visible tokens of every selected block, K and V
                 (n_valid * D * elem * 2 per (token, KV head, block)), q, and
                 the split partials (written, then read by combine);
    combine:     partials read + out (bf16) + lse (fp32) written."""
    s = w.spec
    P, Hkv, d, D = s.block_size, s.num_kv_heads, s.index_dim, s.head_dim
    L = w.seq_lens.long().cpu()
    nb = (L + P - 1) // P
    T = w.num_tokens
    idx = int(L.sum()) * Hkv * d * 2 + T * Hkv * d * 2 + int(nb.sum()) * s.q_len * Hkv * 4
    return {"index_score": idx, "nb": nb, "L": L}


def decode_bytes(w: wl.Workload, selected: torch.Tensor, nsplit: int) -> dict:
    s = w.spec
    P, D = s.block_size, s.head_dim
    row = {"bf16": 2 * D, "fp8_e4m3": D, "nvfp4": D // 2 + D // 16}[s.kv_dtype]
    T = w.num_tokens
    sel = selected[:T].long()                                   # [T, Hkv, S]
    q_lens = w.q_lens.long()
    pos = (w.seq_lens.long().repeat_interleave(q_lens)
           - q_lens.repeat_interleave(q_lens)
           + torch.cat([torch.arange(int(n), device=q_lens.device) for n in q_lens.tolist()]))
    vis = (pos[:, None, None] + 1 - sel * P).clamp(0, P)
    vis = torch.where(sel >= 0, vis, torch.zeros_like(vis))
    kv = int(vis.sum()) * row * 2
    partial = T * s.num_q_heads * nsplit * (D + 1) * 4
    q = T * s.num_q_heads * D * 2
    out = T * s.num_q_heads * (D * 2 + 4)
    return {"decode": kv + q + partial, "combine": partial + out, "kv": kv}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    """(value, "measured" | "fallback") for hbm_gbs, bf16_tflops and
    bf16_tflops_sustained."""
    fallback = {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": 1900.0,
                "bf16_tflops_sustained": 1700.0}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
    except (OSError, ValueError):
        m = {}
    return {k: ((float(m[k]), "measured") if k in m else (v, "fallback"))
            for k, v in fallback.items()}


def prefill_flops(w: wl.Workload, selected: torch.Tensor) -> dict:
    """Algorithmic FLOPs of a prefill step.

    index score: 2 * d per (query token, KV head, visible key);
    sparse prefill (selected tiles): 4 * D per (query token, query head,
    visible key of a selected block) -- QK^T and PV."""
    s = w.spec
    P = s.block_size
    T = w.num_tokens
    q_lens = w.q_lens.long()
    pos = (w.seq_lens.long().repeat_interleave(q_lens) - q_lens.repeat_interleave(q_lens)
           + torch.cat([torch.arange(int(n), device=q_lens.device) for n in q_lens.tolist()]))
    idx = int((pos + 1).sum()) * s.num_kv_heads * 2 * s.index_dim
    sel = selected[:T].long()
    vis = (pos[:, None, None] + 1 - sel * P).clamp(0, P)
    vis = torch.where(sel >= 0, vis, torch.zeros_like(vis))
    att = int(vis.sum()) * s.group * 4 * s.head_dim
    return {"index_score": idx, "sparse_prefill": att}


# ----------------------------------------------------------------- oracle leg
def _oracle_problems(w: wl.Workload, seed: int = 0):
    """An endless seeded stream of (token, KV head) pairs of the workload, each
    as a one-request, one-head host problem (that request's pages only, float32
    copies of the bf16 values, raw codes for e4m3)."""
    s = w.spec
    rng = np.random.default_rng(seed)
    G = s.group
    cu = w.cu_seqlens_q.cpu()
    while True:
        t = int(rng.integers(0, w.num_tokens))
        h = int(rng.integers(0, s.num_kv_heads))
        r = int(torch.searchsorted(cu, torch.tensor([t], dtype=torch.int32), right=True)[0]) - 1
        L = int(w.seq_lens[r])
        nb = -(-L // s.block_size)
        pages = w.block_table[r, :nb].long()
        q0, nq = int(cu[r]), int(w.q_lens[r])

        hs = slice(2 * h, 2 * h + 2) if s.kv_dtype == "nvfp4" else slice(h, h + 1)

        def host(x, hs=hs):
            x = x[pages][:, hs].cpu()
            return x.view(torch.uint8).numpy() if x.dtype == torch.float8_e4m3fn \
                else x.float().numpy()
        yield dict(
            seq_lens=np.array([L]), q_lens=np.array([nq]), block_table=np.arange(nb)[None],
            idx_q=w.idx_q[q0:q0 + nq, h:h + 1].float().cpu().numpy(),
            idx_k_pages=host(w.idx_k_pages, slice(h, h + 1)),
            q=w.q[q0:q0 + nq, h * G:(h + 1) * G].float().cpu().numpy(),
            k_pages=host(w.k_pages), v_pages=host(w.v_pages), token=np.array([t - q0]))


def _run_oracle_problem(oracle, s: wl.WorkloadSpec, pr):
    return oracle.sparse_attention(
        seq_lens=pr["seq_lens"], q_lens=pr["q_lens"], block_table=pr["block_table"],
        idx_q=pr["idx_q"], idx_k_pages=pr["idx_k_pages"], q=pr["q"], k_pages=pr["k_pages"],
        v_pages=pr["v_pages"], num_kv_heads=1, block_size=s.block_size,
        init_blocks=s.init_blocks,
        local_blocks=oracle.local_blocks_from_tokens(s.local_tokens, s.block_size),
        topk_blocks=s.topk_blocks, softmax_scale=s.softmax_scale, k_scale=s.kv_scale,
        v_scale=s.kv_scale, kv_is_e4m3=s.kv_dtype == "fp8_e4m3",
        kv_is_nvfp4=s.kv_dtype == "nvfp4", tokens=[int(pr["token"][0])])


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_worker(shm_name, layout, spec, first, warmup, steps, budget_s, barrier, results):
    """One host core: attach the shared problems, wait for every worker, run
    `warmup` problems untimed, then `steps` problems (or, with steps = 0, as
    many as fit in budget_s) and report (count, seconds)."""
    from multiprocessing import shared_memory
    import oracle
    shm = shared_memory.SharedMemory(name=shm_name)
    try:
        probs = [{k: np.ndarray(shape, np.dtype(dt), buffer=shm.buf, offset=off)
                  for k, (off, shape, dt) in lay.items()} for lay in layout]
        i = first
        for _ in range(warmup):
            _run_oracle_problem(oracle, spec, probs[i % len(probs)])
            i += 1
        barrier.wait()
        n, t0 = 0, time.perf_counter()
        while (steps and n < steps) or (not steps and time.perf_counter() - t0 < budget_s):
            _run_oracle_problem(oracle, spec, probs[i % len(probs)])
            i += 1
            n += 1
        results.put((n, time.perf_counter() - t0))
        del probs
    finally:
        shm.close()


def run_oracle_pool(w: wl.Workload, workers: int, n_problems: int, *, warmup=1, steps=0,
                    budget_s=10.0, seed=0):
    """The oracle, as it stands, on `workers` host processes at once (spawned,
    so no CUDA state is inherited), single-threaded BLAS in each.  They share
    n_problems (token, KV head) problems of the workload through shared
    memory, worker i starting at problem i.  Returns (pairs done, seconds of
    the slowest worker)."""
    import multiprocessing as mp
    from multiprocessing import shared_memory
    gen = _oracle_problems(w, seed=seed)
    probs = [next(gen) for _ in range(n_problems)]
    layout, off = [], 0
    for pr in probs:
        lay = {}
        for k, v in pr.items():
            v = np.ascontiguousarray(v)
            lay[k] = (off, v.shape, v.dtype.str)
            off += (v.nbytes + 63) // 64 * 64
        layout.append(lay)
    shm = shared_memory.SharedMemory(create=True, size=max(off, 64))
    try:
        for pr, lay in zip(probs, layout):
            for k, (o, shape, dt) in lay.items():
                np.ndarray(shape, np.dtype(dt), buffer=shm.buf, offset=o)[...] = pr[k]
        del probs
        ctx = mp.get_context("spawn")
        barrier, results = ctx.Barrier(workers), ctx.Queue()
        procs = [ctx.Process(target=_oracle_worker,
                             args=(shm.name, layout, w.spec, i, warmup, steps, budget_s,
                                   barrier, results)) for i in range(workers)]
        for p in procs:
            p.start()
        got = [results.get(timeout=600) for _ in procs]
        for p in procs:
            p.join(timeout=60)
    finally:
        shm.close()
        shm.unlink()
    return sum(n for n, _ in got), max(t for _, t in got)


def cpu_baseline(w: wl.Workload, budget_s: float = 10.0):
    """The oracle as it stands on the host: all host cores at once (one process
    per core) and one core alone, each over a bounded sample of (token, KV
    head) pairs for about budget_s seconds; q-tokens/s = pairs / H_kv / s."""
    s = w.spec
    cores = host_cores()
    n_all, t_all = run_oracle_pool(w, cores, min(16, cores), budget_s=budget_s)
    n_one, t_one = run_oracle_pool(w, 1, 4, budget_s=budget_s, seed=1)
    return {"value": n_all / s.num_kv_heads / t_all, "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "one_core": {"value": n_one / s.num_kv_heads / t_one, "cores": 1},
            "sample": f"random (token, KV head) pairs of {s.name} (one request's pages each), "
                      f"fp64 numpy, single-threaded BLAS per process: {n_all} pairs on "
                      f"{cores} processes in {t_all:.1f} s, {n_one} pairs on one in "
                      f"{t_one:.1f} s"}


# ----------------------------------------------------------------- our arm
LAUNCHES_PER_CALL = {"plan": 1, "index_score": 1, "topk_select": 1, "build_k2q_csr": 7,
                     "sparse_prefill": 1, "sparse_decode": 1, "combine": 1,
                     "compact_selected": 1}


def launches_per_call(name, spec):
    """Kernels one call launches: the decode index scan (one new token per
    request) sets the scores to -inf first and then scans half tiles."""
    if name == "index_score" and spec.q_len == 1:
        return 2
    return LAUNCHES_PER_CALL[name]


def _step_calls(msa, sa, w):
    """The step's calls, as msa_decode_step chains them (decode / verify),
    SparseAttention.run does (prefill), or the dense-sparse form runs them
    (compaction + dense paged decode in place of the sparse decode)."""
    c = sa.cfg
    cu = w.cu_seqlens_q if sa.prefill else None
    calls = [
        ("plan", lambda: msa.plan(c, w.seq_lens, w.block_table, sa.ws, cu)),
        ("index_score", lambda: msa.index_score(c, sa.ws, w.idx_q, w.idx_k_pages,
                                                sa.block_scores)),
        ("topk_select", lambda: msa.topk_select(c, sa.ws, sa.block_scores, sa.selected)),
    ]
    if sa.prefill:
        calls += [
            ("build_k2q_csr", lambda: msa.ops.build_k2q_csr(c, sa.ws, sa.selected, sa.row_ptr,
                                                            sa.q_indices)),
            ("sparse_prefill", lambda: msa.ops.sparse_prefill(
                c, sa.ws, w.q, w.k_pages, w.v_pages, sa.selected, sa.row_ptr, sa.q_indices)),
        ]
    elif sa.dense_sparse:
        calls += [
            ("compact_selected", lambda: msa.compact_selected(c, sa.ws, sa.selected, sa.page_table,
                                                              sa.dense_len)),
            ("sparse_decode", lambda: msa.paged_decode(c, sa.ws, w.q, w.k_pages, w.v_pages,
                                                       sa.page_table, sa.dense_len)),
        ]
    else:
        calls += [("sparse_decode", lambda: msa.sparse_decode(c, sa.ws, w.q, w.k_pages,
                                                              w.v_pages, sa.selected))]
    calls += [("combine", lambda: msa.combine(c, sa.ws, sa.out, sa.lse))]
    return calls


def _e2e(msa, sa, w, cfg, dev, stream, K, warmup, world):
    """Throughput through the public API with host buffers: SparseAttention.run
    per step, each step's inputs copied from pinned host memory and its result
    read back inside the timed region.  Pipelined as a serving loop would run
    it: step i+1's inputs go host -> device on a copy stream while step i
    computes, and step i's result comes back on a second copy stream while step
    i+1 computes (two SparseAttention instances and two input buffers
    alternate)."""
    step_inputs = ("seq_lens", "block_table", "idx_q", "q") + (("cu_seqlens_q",) if sa.prefill
                                                               else ())
    pin = {k: getattr(w, k).cpu().pin_memory() for k in step_inputs}
    sas = [sa, msa.SparseAttention(cfg, device=dev)]
    dbufs = [{k: torch.empty_like(getattr(w, k)) for k in pin} for _ in range(2)]
    outs_h = [(torch.empty(sa.out.shape, dtype=sa.out.dtype).pin_memory(),
               torch.empty(sa.lse.shape, dtype=sa.lse.dtype).pin_memory()) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in outs_h[0])
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)]
          for k in ("in_ready", "in_free", "out_ready", "out_free")}
    for b in range(2):          # every buffer starts free
        ev["in_free"][b].record(stream)
        ev["out_free"][b].record(stream)

    def upload(b):
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev["in_free"][b])
            for k, t in pin.items():
                dbufs[b][k].copy_(t, non_blocking=True)
            ev["in_ready"][b].record(s_in)

    def e2e_steps(n, start_ev=None):
        if start_ev is not None:
            s_in.wait_event(start_ev)
        upload(0)
        for i in range(n):
            b = i & 1
            stream.wait_event(ev["in_ready"][b])
            stream.wait_event(ev["out_free"][b])
            d = dbufs[b]
            sas[b].run(d["seq_lens"], d["block_table"], d["idx_q"], w.idx_k_pages, d["q"],
                       w.k_pages, w.v_pages, cu_seqlens_q=d.get("cu_seqlens_q"))
            ev["in_free"][b].record(stream)
            ev["out_ready"][b].record(stream)
            if i + 1 < n:
                upload(1 - b)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev["out_ready"][b])
                outs_h[b][0].copy_(sas[b].out, non_blocking=True)
                outs_h[b][1].copy_(sas[b].lse, non_blocking=True)
                ev["out_free"][b].record(s_out)
        for b in range(2):
            stream.wait_event(ev["out_free"][b])

    e2e_steps(max(3, warmup // 4))
    torch.cuda.synchronize()
    Ke = max(10, K // 2)
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    e2e_steps(Ke, start_ev=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    assert all(msa.check_device_error(x.ws) == 0 for x in sas)
    del sas[1]
    return Ke, e2e_ms, h2d, d2h


def _traffic(spec, kernel):
    """The kernel's DRAM bytes per launch from the committed ncu capture, for
    the workload at its stated sizes only (None once they are overridden)."""
    base = wl.WORKLOADS.get(spec.name)
    if base is None or base.replace(seed=spec.seed) != spec:
        return None
    return NCU_TRAFFIC_BYTES.get((spec.name, kernel))


def _device_times(calls, stream, n=20, reps=5):
    """Device time per launch of each call of the step: the call repeated n
    times in a CUDA graph (every call of the step is idempotent on its inputs),
    the median of `reps` replays divided by n.  Without the host launch that
    a per-call event pair also brackets."""
    out = {}
    for name, fn in calls:
        graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for _ in range(n):
                    fn()
        stream.wait_stream(side)
        graph.replay()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / n)
        out[name] = sorted(ts)[reps // 2]
        del graph
    return out


def _cache_write_cost(msa, sa, w, spec, stream, n):
    """The K / V / index-key cache write that precedes a step (msa_cache_write,
    slots from the plan), timed alone over n calls after the step's plan: it is
    not part of the timed step.  Algorithmic bytes: the new rows read (bf16)
    and written (bf16, e4m3 or NVFP4 K / V rows, bf16 index keys)."""
    c = sa.cfg
    T = w.num_tokens
    k, v, idx_k = wl.new_token_rows(spec, msa.ops.max_tokens(c), seed=spec.seed + 500,
                                    device=w.q.device)
    D = spec.head_dim
    row = {"fp8_e4m3": D, "nvfp4": D // 2 + D // 16}.get(spec.kv_dtype, 2 * D)   # stored K / V row
    per = spec.num_kv_heads * (2 * D * 2 + 2 * row + 2 * spec.index_dim * 2)
    msa.plan(c, w.seq_lens, w.block_table, sa.ws, w.cu_seqlens_q if sa.prefill else None)
    call = lambda: msa.cache_write(c, sa.ws, k, v, idx_k, w.k_pages, w.v_pages,  # noqa: E731
                                   w.idx_k_pages)
    call()
    torch.cuda.synchronize()
    # a launch this small is paced by the host: time n launches captured in a
    # CUDA graph, replayed back to back
    graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for _ in range(n):
                call()
    stream.wait_stream(side)
    graph.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(3):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    assert msa.check_device_error(sa.ws) == 0
    ms = e0.elapsed_time(e1) / (3 * n)
    return {"ms": ms, "bytes": T * per, "gbs": T * per / (ms / 1e3) / 1e9,
            "note": "msa_cache_write before the step (not in the timed step), timed alone "
                    f"from a CUDA graph of {n} launches"}


def _index_attention_cost(msa, sa, w, spec, stream, n):
    """The index-value branch (msa_index_attention) on the step's plan, timed
    alone over n calls: a layer that keeps index values runs it beside the
    step.  Algorithmic bytes: every visible index key and index value once per
    token and KV head (the verify drafts each read their own), idx_q, idx_o."""
    c = sa.cfg
    if sa.prefill:
        return None
    idx_v = wl.index_values(spec, seed=spec.seed + 600, device=w.q.device)
    scratch = torch.empty(msa.index_attention_scratch_bytes(c), dtype=torch.uint8,
                          device=w.q.device)
    T, H, d = msa.ops.max_tokens(c), spec.num_kv_heads, spec.index_dim
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=w.q.device)
    lse = torch.empty((T, H), dtype=torch.float32, device=w.q.device)
    msa.plan(c, w.seq_lens, w.block_table, sa.ws)
    call = lambda: msa.index_attention(c, sa.ws, w.idx_q, w.idx_k_pages, idx_v,  # noqa: E731
                                       scratch, out, lse)
    for _ in range(3):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    assert msa.check_device_error(sa.ws) == 0
    ms = e0.elapsed_time(e1) / n
    q_lens = w.q_lens.long()
    pos = (w.seq_lens.long().repeat_interleave(q_lens) - q_lens.repeat_interleave(q_lens)
           + torch.cat([torch.arange(int(k), device=q_lens.device) for k in q_lens.tolist()]))
    nbytes = int((pos + 1).sum()) * H * d * 2 * 2 + w.num_tokens * H * d * 4
    return {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms / 1e3) / 1e9,
            "note": "msa_index_attention (index-value branch; parity of its reading unpinned), "
                    "timed alone, not in the timed step"}


def measure(spec, steps, warmup, dev, world, clock_gpu, e2e=False, dense_sparse=False):
    """Times `steps` steps of one workload after `warmup` untimed ones, the
    dominant kernel bracketed by CUDA events in the timed region, then a
    per-kernel breakdown from further steps.  Returns the bench fields.
    dense_sparse: the decode runs as compaction + dense paged decode."""
    import block_sparse_paged_msa_gb300 as msa
    w = wl.make_workload(spec, device=dev)
    cfg = msa.config_for(spec)
    sa = msa.SparseAttention(cfg, device=dev, dense_sparse=dense_sparse)
    stream = torch.cuda.current_stream()
    calls = _step_calls(msa, sa, w)
    names = [n for n, _ in calls]
    dominant = "sparse_prefill" if sa.prefill else "index_score"
    dom_i = names.index(dominant)

    def step(evs=None, only=None):
        """One step; events around every call (evs) or only around call `only`.
        An event between two kernels keeps the second from launching early
        (programmatic dependent launch), so the timed steps bracket only the
        dominant kernel."""
        for i, (_, fn) in enumerate(calls):
            timed = evs is not None and (only is None or i == only)
            if timed:
                evs[i][0].record(stream)
            fn()
            if timed:
                evs[i][1].record(stream)

    K = steps
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in names] for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(clock_gpu) as clk:
        # the warm-up steps run once the sampler is up, right before the timed
        # region, so that the GPU does not sit idle between them
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        assert msa.check_device_error(sa.ws) == 0
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for k in range(K):
            step(evs[k], only=dom_i)
        stop.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
    ms = start.elapsed_time(stop)
    dom_ms = sum(evs[k][dom_i][0].elapsed_time(evs[k][dom_i][1]) for k in range(K)) / K
    # per-kernel breakdown, after the timed region (every call bracketed)
    Kb = min(K, 200)
    for k in range(Kb):
        step(evs[k])
    torch.cuda.synchronize()
    assert msa.check_device_error(sa.ws) == 0
    per_kernel = {n: sum(evs[k][i][0].elapsed_time(evs[k][i][1]) for k in range(Kb)) / Kb
                  for i, n in enumerate(names)}
    per_kernel_dev = _device_times(calls, stream)
    e2e_res = _e2e(msa, sa, w, cfg, dev, stream, K, warmup, world) if e2e else None
    cw = _cache_write_cost(msa, sa, w, spec, stream, Kb)
    ia = _index_attention_cost(msa, sa, w, spec, stream, min(Kb, 50)) if e2e else None

    T = w.num_tokens
    times = [ms, dom_ms] + ([e2e_res[1]] if e2e_res else [])
    times = max_over_ranks(times, world, dev)
    ms, dom_ms = times[0], times[1]
    peaks = measured_peaks()
    r = {
        "metric": METRIC if not sa.prefill else "sparse-prefill query-tokens/s",
        "value": replica_throughput(T, world, K, ms), "unit": UNIT, "steps": K,
        "warmup": warmup, "ms_per_step": ms / K,
        "dtype": spec.kv_dtype,
        "config": {"workload": spec.name, "batch": spec.batch,
                   "seq_lens": list(spec.seq_len_range or spec.seq_lens[:1]),
                   "q_per_request": spec.q_len,
                   "q_heads": spec.num_q_heads, "kv_heads": spec.num_kv_heads,
                   "head_dim": spec.head_dim, "index_dim": spec.index_dim,
                   "block": spec.block_size, "init_local_topk": [spec.init_blocks,
                   cfg.local_blocks, spec.topk_blocks],
                   "pool_pages": spec.num_pages, "parallelism": f"replicas{world}",
                   "decode_form": ("dense_sparse (compacted pages + dense paged decode)"
                                   if dense_sparse else "sparse (selected lists)")},
        "kernels_ms": per_kernel,
        "kernels_ms_note": ("dominant kernel timed in the timed region; the others in "
                            f"{Kb} further steps with every call bracketed by events "
                            "(the host launch of a short call shows in its time)"),
        "kernels_device_ms": per_kernel_dev,
        "kernels_device_ms_note": ("each call of the step alone, 20 launches back to back "
                                   "replayed from a CUDA graph: device time per launch"),
        "gpu_launches": sum(launches_per_call(n, spec) for n in names) * K,
        "clocks": clk.summary(),
        "cache_write": cw,
    }
    if ia is not None:
        r["index_attention"] = ia
    if e2e_res is not None:
        Ke, e2e_ms, h2d, d2h = e2e_res
        r["e2e"] = {"value": replica_throughput(T, world, Ke, times[2]), "unit": UNIT,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "how": "SparseAttention.run per step; inputs of step i+1 uploaded and the "
                           "result of step i read back on copy streams while step i+1 "
                           "computes"}
    if sa.prefill:
        fl = prefill_flops(w, sa.selected)
        achieved = {n: fl[n] / (per_kernel[n] / 1e3) / 1e12
                    for n in ("index_score", "sparse_prefill")}
        achieved["sparse_prefill"] = fl["sparse_prefill"] / (dom_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops_sustained"]
        r["roofline"] = {
            "bound": "tensor", "kernel": "sparse_prefill", "achieved": achieved["sparse_prefill"],
            "peak": peak[0], "unit": "TFLOP/s", "frac": achieved["sparse_prefill"] / peak[0],
            "peak_source": f"{peak[1]} bf16_tflops_sustained", "launch_ms": dom_ms,
            "traffic": _traffic(spec, "sparse_prefill")}
        r["kernel_tflops"] = achieved
        r["flops_per_step"] = {k: fl[k] for k in ("index_score", "sparse_prefill")}
        r["config"]["l2"] = "no flush: K/V + index pools 0.9 GB and 2.7 GB of partials > L2"
    else:
        ab = algorithmic_bytes(w)
        db = decode_bytes(w, sa.selected, msa.num_splits(cfg))
        peak = peaks["hbm_gbs"]
        idx_gbs = ab["index_score"] / (dom_ms / 1e3) / 1e9
        step_bytes = ab["index_score"] + db["decode"] + db["combine"]
        r["roofline"] = {"bound": "hbm", "kernel": "index_score", "achieved": idx_gbs,
                         "peak": peak[0], "unit": "GB/s", "frac": idx_gbs / peak[0],
                         "peak_source": f"{peak[1]} hbm_gbs", "launch_ms": dom_ms,
                         "traffic": _traffic(spec, "index_score")}
        r["step_hbm"] = {"algorithmic_bytes": step_bytes,
                         "achieved_gbs": step_bytes / (ms / K / 1e3) / 1e9,
                         "frac": step_bytes / (ms / K / 1e3) / 1e9 / peak[0]}
        r["kernel_gbs"] = {
            "index_score": idx_gbs,
            "sparse_decode": db["decode"] / (per_kernel["sparse_decode"] / 1e3) / 1e9,
            "combine": db["combine"] / (per_kernel["combine"] / 1e3) / 1e9}
        r["kv_bytes_per_step"] = db["kv"]
        r["config"]["l2"] = (f"no flush: {step_bytes / 1e9:.2f} GB touched per step "
                             f"> 129 MB L2")
    del sa
    return r, w


# The other configurations the default run measures beside the headline, with
# their timed / warm-up steps (each a few dozen milliseconds of GPU time; most
# of their cost is drawing the inputs, 90 GB for the long decode).  A name
# "<workload>:dense_sparse" runs that workload's decode in the dense-sparse
# form (the A/B of the two decode formulations).
OTHER_WORKLOADS = {"prefill": (40, 5), "nvfp4_prefill": (40, 5), "fp8_decode": (200, 10),
                   "nvfp4_decode": (200, 10),
                   "verify": (100, 5), "long_decode": (40, 5),
                   "medium_decode:dense_sparse": (200, 10)}


def run_ours(args, rank, world, local_rank):
    import block_sparse_paged_msa_gb300 as msa
    from block_sparse_paged_msa_gb300 import build as msa_build
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if rank == 0 or not os.path.exists(msa.ops.lib_path()):
        msa_build.build()
    if world > 1:
        torch.distributed.barrier()
    clock_gpu = local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else 0
    base = workload_spec(args)
    spec = base.replace(seed=base.seed + rank)
    result, w = measure(spec, args.steps, args.warmup, dev, world, clock_gpu, e2e=True)
    result.update({"n_gpus": world, "higher_is_better": True, "scaling": "weak",
                   "vs_baseline": None,
                   "data": "synthetic (seeded; integer-valued bf16 index vectors, N(0,1) bf16 "
                           "q/k/v)"})
    others = [n for n in args.others.split(",") if n and n != "none" and n != spec.name]
    bad = [n for n in others if n.partition(":")[0] not in wl.WORKLOADS]
    if bad:
        raise SystemExit(f"unknown workloads {bad}")
    if others:
        # the headline's inputs are kept (the CPU baseline samples them)
        torch.cuda.empty_cache()
        result["workloads"] = {}
        for name in others:
            K, W = OTHER_WORKLOADS.get(name, (40, 5))
            base_name, _, form = name.partition(":")
            o = wl.WORKLOADS[base_name]
            r, wo = measure(o.replace(seed=o.seed + rank), K, W, dev, world, clock_gpu,
                            dense_sparse=form == "dense_sparse")
            keep = ("metric", "value", "unit", "ms_per_step", "steps", "warmup", "dtype",
                    "roofline", "kernels_ms", "kernels_device_ms", "kernel_gbs",
                    "kernel_tflops", "step_hbm",
                    "clocks", "gpu_launches", "config", "cache_write")
            result["workloads"][name] = {k: r[k] for k in keep if k in r}
            del wo
            torch.cuda.empty_cache()
    return result, w


def workload_spec(args) -> wl.WorkloadSpec:
    spec = wl.WORKLOADS[args.workload]
    kw = {}
    if args.batch is not None:
        kw["batch"] = args.batch
        if spec.seq_lens is not None:
            kw["seq_lens"] = (spec.seq_lens * args.batch)[:args.batch]
    if args.pool_pages is not None:
        kw["num_pages"] = args.pool_pages
    return spec.replace(**kw) if kw else spec


def run_reference(args):
    """The fp64 oracle on every host core: each step is one (token, KV head)
    pair per core, all cores at once; the timed steps end when the slowest
    core finishes its share."""
    spec = workload_spec(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = wl.make_workload(spec, device=dev)
    cores = host_cores()
    n, dt = run_oracle_pool(w, cores, min(16, cores), warmup=args.warmup, steps=args.steps,
                            seed=1)
    value = n / spec.num_kv_heads / dt
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": {"workload": spec.name},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step one (token, KV head) pair of {spec.name} per "
                                   f"core (one request's pages), {cores} processes, fp64 "
                                   f"numpy, single-threaded BLAS per process"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="medium_decode", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--others", default=None,
                    help="comma-separated workloads measured beside the headline (default: "
                         "every other configuration when the headline is medium_decode at "
                         "its full size; 'none' to skip)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (smaller profiling captures)")
    ap.add_argument("--pool-pages", type=int, default=None,
                    help="override the workload's KV pool size in pages")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.others is None:
        default = args.workload == "medium_decode" and args.batch is None \
            and args.pool_pages is None
        args.others = ",".join(OTHER_WORKLOADS) if default else "none"
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    result, w = run_ours(args, rank, world, local_rank)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
