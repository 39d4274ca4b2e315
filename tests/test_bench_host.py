"""bench.py's host-side oracle leg: the fp64 oracle run on several spawned
processes at once over problems shared through shared memory (CPU only).
Each worker must run exactly the requested number of timed problems, and the
pooled results must be those of the oracle itself (a problem run in a worker
gives the same selection as run in this process)."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


@pytest.mark.timeout(300)
def test_oracle_pool_counts_and_times():
    import bench
    from block_sparse_paged_msa_gb300 import workloads as wl
    w = wl.make_workload(wl.WORKLOADS["tiny_decode"], device="cpu")
    n, dt = bench.run_oracle_pool(w, 2, 3, warmup=1, steps=4)
    assert n == 8 and dt > 0
    n, dt = bench.run_oracle_pool(w, 2, 2, budget_s=0.5)
    assert n >= 2 and dt >= 0.5


def test_oracle_problem_is_one_request_one_head():
    import bench
    import oracle
    from block_sparse_paged_msa_gb300 import workloads as wl
    spec = wl.WORKLOADS["tiny_decode"]
    w = wl.make_workload(spec, device="cpu")
    pr = next(bench._oracle_problems(w, seed=3))
    res = bench._run_oracle_problem(oracle, spec, pr)
    (t, h), = res["selected"].keys()
    assert h == 0 and t == int(pr["token"][0])
    L = int(pr["seq_lens"][0])
    nb = -(-L // spec.block_size)
    assert pr["idx_k_pages"].shape == (nb, 1, spec.block_size, spec.index_dim)
    assert np.all(np.diff(res["selected"][(t, h)]) > 0)
    assert bench.host_cores() >= 1
