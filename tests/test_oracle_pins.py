"""Pins of the fp64 oracle to facts other than itself (no GPU needed).

Each test checks one oracle function against brute force, a hand-computed
fixture, a closed form, an invariant of the mathematics, or an independent
library routine, so that a dropped term, a wrong sign, an off-by-one or a
transposed operand anywhere in the oracle fails at least one of them.  The
mutation tests at the bottom plant such mistakes in the oracle (on the CPU) and
check that the pins catch them."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from block_sparse_paged_msa_gb300 import workloads as wl
from oracle_io import oracle_local_blocks, run_oracle, to_np

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- config
def test_block_counts_from_tokens():
    g = _golden("config_resolution.json")
    P = g["block_size"]
    for tokens, blocks in g["local"]:
        assert oracle.local_blocks_from_tokens(tokens, P) == blocks, tokens
    for tokens, blocks in g["init"]:
        assert oracle.init_blocks_from_tokens(tokens, P) == blocks, tokens


# ---------------------------------------------------------------- fp8
def test_e4m3_decode_matches_torch_and_known_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_float(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    known = {0x00: 0.0, 0x38: 1.0, 0xB8: -1.0, 0x7E: 448.0, 0xFE: -448.0,
             0x01: 2.0 ** -9, 0x08: 2.0 ** -6, 0x07: 7 * 2.0 ** -9, 0x40: 2.0,
             0x3C: 1.5, 0x30: 0.5}
    for c, v in known.items():
        assert ours[c] == v, hex(c)
    assert math.isnan(ours[0x7F]) and math.isnan(ours[0xFF])


# ---------------------------------------------------------------- geometry
def test_query_positions_decode_verify_prefill():
    assert oracle.query_positions([1000, 1500], [1, 1]) == [(0, 999), (1, 1499)]
    assert oracle.query_positions([10], [4]) == [(0, 6), (0, 7), (0, 8), (0, 9)]
    assert oracle.query_positions([5, 3], [2, 3]) == [(0, 3), (0, 4), (1, 0), (1, 1), (1, 2)]
    assert oracle.query_positions([7], [0]) == []
    # an idle request (seq_len 0) keeps its token rows, at position -1
    assert oracle.query_positions([0, 3], [1, 1]) == [(0, -1), (1, 2)]


def test_gather_sequence_follows_block_table():
    rng = np.random.default_rng(0)
    P, H, X, pages = 4, 2, 3, 6
    logical = rng.integers(-50, 50, size=(21, H, X)).astype(np.float64)
    table = [4, 0, 5, 2, 1, 3]
    pool = np.full((pages, H, P, X), np.nan)
    for t in range(21):
        pool[table[t // P], :, t % P, :] = logical[t]
    got = oracle.gather_sequence(pool, table, 21, P)
    assert np.array_equal(got, logical)


# ---------------------------------------------------------------- scores
def _paged(logical, P, rng, extra_pages=3):
    """Scatter a logical [L, H, X] sequence into a shuffled pool."""
    L, H, X = logical.shape
    nb = -(-L // P)
    pages = nb + extra_pages
    perm = rng.permutation(pages)[:nb]
    pool = rng.standard_normal((pages, H, P, X)) * 1e6  # garbage outside
    for t in range(L):
        pool[perm[t // P], :, t % P, :] = logical[t]
    return pool, perm


def test_block_scores_exact_against_integer_brute_force():
    rng = np.random.default_rng(1)
    P, d, L = 8, 5, 61
    for trial in range(5):
        ik = rng.integers(-4, 5, size=(L, 1, d))
        iq = rng.integers(-4, 5, size=d)
        pool, table = _paged(ik.astype(np.float64), P, rng)
        seq = oracle.gather_sequence(pool, table, L, P)
        for pos in (L - 1, 40, 8, 7, 0):
            got = oracle.block_scores(iq.astype(np.float64), seq[:, 0, :], pos, P)
            # pure-Python integer arithmetic straight on the logical sequence
            nb = pos // P + 1
            want = []
            for j in range(nb):
                best = None
                for t in range(j * P, min(j * P + P, pos + 1)):
                    dot = sum(int(iq[k]) * int(ik[t, 0, k]) for k in range(d))
                    best = dot if best is None else max(best, dot)
                want.append(best)
            assert got.tolist() == want, (trial, pos)


# ---------------------------------------------------------------- selection
@pytest.mark.parametrize("case", _golden("selection_cases.json")["cases"],
                         ids=lambda c: c["name"])
def test_selection_hand_computed(case):
    P, L, d = case["block_size"], case["n_tokens"], 4
    ik = np.zeros((L, 1, d))
    for t, val in case["planted"].items():
        ik[int(t), 0, 0] = val
    iq = np.zeros(d)
    iq[0] = case["q0"]
    rng = np.random.default_rng(7)
    pool, table = _paged(ik, P, rng)
    seq = oracle.gather_sequence(pool, table, L, P)
    scores = oracle.block_scores(iq, seq[:, 0, :], case["position"], P)
    assert scores.tolist() == case["scores"]
    sel = oracle.select_blocks(scores, case["init"], case["local"], case["topk"])
    assert sel == case["selected"]


def _random_scores(rng, nb, distinct):
    return rng.integers(-distinct, distinct + 1, size=nb).astype(np.float64)


def test_selection_invariants_random():
    rng = np.random.default_rng(2)
    for _ in range(400):
        nb = int(rng.integers(1, 70))
        init, local, topk = (int(rng.integers(0, 4)), int(rng.integers(1, 5)),
                             int(rng.integers(0, 20)))
        scores = _random_scores(rng, nb, int(rng.integers(0, 6)))  # many ties
        sel = oracle.select_blocks(scores, init, local, topk)
        I = set(range(min(init, nb)))
        Lc = set(range(max(0, nb - local), nb))
        assert sel == sorted(set(sel)), "ascending, unique"
        assert I | Lc <= set(sel), "superset of init and local"
        assert len(sel) == min(nb, init + local + topk), "size"
        cand_sel = [j for j in sel if j not in I | Lc]
        cand_rest = [j for j in range(nb) if j not in I | Lc and j not in sel]
        for a in cand_sel:
            for b in cand_rest:
                # every chosen candidate beats every rejected one, lower index on ties
                assert (scores[a], -a) > (scores[b], -b)


def test_selection_against_exhaustive_subset_search():
    """Brute force: among all candidate subsets of the right size, the selected one
    maximises the sorted score vector, then prefers the lexicographically smallest
    index set."""
    rng = np.random.default_rng(3)
    for _ in range(60):
        nb = int(rng.integers(4, 11))
        init, local, topk = 1, 2, int(rng.integers(1, 4))
        scores = _random_scores(rng, nb, 2)
        cands = list(range(init, nb - local))
        k = min(topk, len(cands))
        best = None
        for sub in itertools.combinations(cands, k):
            key = (sorted((scores[j] for j in sub), reverse=True),
                   [-j for j in sub])
            if best is None or key > best[0]:
                best = (key, sub)
        want = sorted(set(range(init)) | set(range(nb - local, nb)) | set(best[1]))
        assert oracle.select_blocks(scores, init, local, topk) == want


# ---------------------------------------------------------------- attention
def _dense_reference(q_rows, k, v, scale):
    s = scale * (q_rows @ k.T)
    return scipy.special.softmax(s, axis=1) @ v, scipy.special.logsumexp(s, axis=1)


def test_attention_special_cases():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((3, 16))
    k = rng.standard_normal((9, 16))
    # single key: out = v, lse = its logit
    o, l = oracle.attention(q, k[:1], k[1:2], 0.3)
    assert np.allclose(o, np.repeat(k[1:2], 3, 0), atol=0, rtol=0)
    assert np.allclose(l, 0.3 * q @ k[0], atol=1e-15)
    # softmax weights sum to one: v = ones -> out = 1
    o, l = oracle.attention(q, k, np.ones((9, 5)), 0.25)
    assert np.allclose(o, 1.0, atol=1e-15)
    # lse bounds: max s <= lse <= max s + ln n
    s = 0.25 * q @ k.T
    assert np.all(l >= s.max(1) - 1e-15) and np.all(l <= s.max(1) + math.log(9) + 1e-15)
    # shift invariance: an extra coordinate adds c/scale * 1 to every logit
    v = rng.standard_normal((9, 4))
    o1, l1 = oracle.attention(q, k, v, 0.5)
    c = 1.7
    q2 = np.concatenate([q, np.full((3, 1), c / 0.5)], 1)
    k2 = np.concatenate([k, np.ones((9, 1))], 1)
    o2, l2 = oracle.attention(q2, k2, v, 0.5)
    assert np.allclose(o1, o2, atol=1e-13) and np.allclose(l2, l1 + c, atol=1e-13)
    # empty key set: zeros and -inf
    o, l = oracle.attention(q, k[:0], v[:0], 0.5)
    assert np.all(o == 0) and np.all(np.isneginf(l))
    # matches scipy's softmax / logsumexp
    o, l = oracle.attention(q, k, v, 0.5)
    ro, rl = _dense_reference(q, k, v, 0.5)
    assert np.allclose(o, ro, atol=1e-13) and np.allclose(l, rl, atol=1e-13)
    # a transposed / permuted operand is caught: q rows are not interchangeable
    assert not np.allclose(oracle.attention(q[::-1], k, v, 0.5)[0], o)


def test_combine_equals_unsplit():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((4, 8))
    k = rng.standard_normal((50, 8)) * 3
    v = rng.standard_normal((50, 8))
    o_all, l_all = oracle.attention(q, k, v, 0.7)
    for cuts in ([25], [1, 2, 49], [10, 20, 30, 40], [0, 50]):
        bounds = [0] + cuts + [50]
        parts = [(a, b) for a, b in zip(bounds[:-1], bounds[1:])]
        for g in range(4):
            os_, ls_ = [], []
            for a, b in parts:
                o, l = oracle.attention(q[g:g + 1], k[a:b], v[a:b], 0.7)
                os_.append(o[0])
                ls_.append(l[0])
            o, l = oracle.combine(np.array(os_), np.array(ls_))
            assert np.allclose(o, o_all[g], atol=1e-12) and abs(l - l_all[g]) < 1e-12
    o, l = oracle.combine(np.zeros((3, 8)), np.full(3, -np.inf))
    assert np.all(o == 0) and np.isneginf(l)


# ---------------------------------------------------------------- whole path
def _logical_sequences(w):
    """Per request: logical idx_k, k, v in token order, read from the pool with
    torch indexing (independent of the oracle's gather)."""
    out = []
    P = w.spec.block_size
    for r in range(w.spec.batch):
        L = int(w.seq_lens[r])
        nb = -(-L // P)
        pages = w.block_table[r, :nb].long()
        def seq(pool):
            x = pool[pages]                               # [nb, H, P, X]
            return x.permute(0, 2, 1, 3).reshape(nb * P, *x.shape[1:2], x.shape[3])[:L]
        out.append((to_np(seq(w.idx_k_pages)), to_np(seq(w.k_pages)), to_np(seq(w.v_pages))))
    return out


def test_dense_when_topk_covers_every_block():
    """topk >= nb - init - local: every visible token is attended, so the result
    is plain causal attention (scipy softmax) over the logical sequence."""
    spec = wl.small("verify", topk_blocks=64, num_kv_heads=2, num_q_heads=6)
    w = wl.make_workload(spec)
    res = run_oracle(w)
    seqs = _logical_sequences(w)
    q = to_np(w.q)
    G = spec.group
    for t, (r, p) in enumerate(oracle.query_positions(to_np(w.seq_lens), to_np(w.q_lens))):
        _, k, v = seqs[r]
        for h in range(spec.num_kv_heads):
            ro, rl = _dense_reference(q[t, h * G:(h + 1) * G], k[:p + 1, h], v[:p + 1, h],
                                      spec.softmax_scale)
            assert np.allclose(res["out"][t, h * G:(h + 1) * G], ro, atol=1e-12)
            assert np.allclose(res["lse"][t, h * G:(h + 1) * G], rl, atol=1e-12)
            assert res["selected"][(t, h)] == list(range(p // 128 + 1))


def test_sparse_equals_dense_over_selected_tokens():
    """With a real top-k the output equals dense attention restricted to the
    tokens of the selected blocks (re-derived here by masking logits)."""
    spec = wl.small("medium_decode", num_kv_heads=2, num_q_heads=4, batch=2)
    w = wl.make_workload(spec)
    res = run_oracle(w)
    seqs = _logical_sequences(w)
    q = to_np(w.q)
    for t, (r, p) in enumerate(oracle.query_positions(to_np(w.seq_lens), to_np(w.q_lens))):
        _, k, v = seqs[r]
        for h in range(2):
            sel = res["selected"][(t, h)]
            assert len(sel) == min(p // 128 + 1, spec.init_blocks
                                   + oracle_local_blocks(w) + spec.topk_blocks)
            s = spec.softmax_scale * q[t, 2 * h:2 * h + 2] @ k[:p + 1, h].T
            mask = np.full(p + 1, -np.inf)
            for j in sel:
                mask[j * 128:(j + 1) * 128] = 0.0
            s = s + mask
            ro = scipy.special.softmax(s, axis=1) @ v[:p + 1, h]
            assert np.allclose(res["out"][t, 2 * h:2 * h + 2], ro, atol=1e-12)
            assert np.allclose(res["lse"][t, 2 * h:2 * h + 2],
                               scipy.special.logsumexp(s, axis=1), atol=1e-12)


def test_page_permutation_invariance():
    spec = wl.small("medium_decode", batch=3, num_kv_heads=2, num_q_heads=4)
    w = wl.make_workload(spec)
    res = run_oracle(w)
    rng = np.random.default_rng(8)
    perm = torch.from_numpy(rng.permutation(spec.num_pages))     # new = perm[old]
    inv = torch.argsort(perm)
    w2 = wl.Workload(**{**w.__dict__})
    w2.idx_k_pages = w.idx_k_pages[inv]
    w2.k_pages = w.k_pages[inv]
    w2.v_pages = w.v_pages[inv]
    bt = w.block_table.clone()
    valid = bt >= 0
    bt[valid] = perm[bt[valid].long()].to(torch.int32)
    w2.block_table = bt
    res2 = run_oracle(w2)
    assert res["selected"] == res2["selected"]
    assert np.array_equal(res["out"], res2["out"]) and np.array_equal(res["lse"], res2["lse"])


def test_fp8_path_uses_dequantised_values():
    spec = wl.small("fp8_decode", batch=2, num_kv_heads=1, num_q_heads=4)
    w = wl.make_workload(spec)
    res = run_oracle(w)
    w2 = wl.Workload(**{**w.__dict__})
    w2.k_pages = (w.k_pages.to(torch.float64) * spec.kv_scale)
    w2.v_pages = (w.v_pages.to(torch.float64) * spec.kv_scale)
    w2.spec = spec.replace(kv_dtype="bf16")
    res2 = run_oracle(w2)
    assert res["selected"] == res2["selected"]
    assert np.allclose(res["out"], res2["out"], atol=1e-13)
    assert np.allclose(res["lse"], res2["lse"], atol=1e-13)


def test_k2q_csr_round_trip():
    rng = np.random.default_rng(9)
    T, H, S, R, NB = 40, 3, 5, 3, 12
    tok_req = np.sort(rng.integers(0, R, size=T))
    sel = np.full((T, H, S), -1)
    for t in range(T):
        for h in range(H):
            n = int(rng.integers(0, S + 1))
            sel[t, h, :n] = np.sort(rng.choice(NB, size=n, replace=False))
    row_ptr, qi = oracle.build_k2q_csr(sel, tok_req, R, NB)
    assert row_ptr[0] == 0 and np.all(np.diff(row_ptr) >= 0)
    assert row_ptr[-1] == (sel >= 0).sum() == len(qi)
    back = {}
    for h in range(H):
        for r in range(R):
            for j in range(NB):
                row = (h * R + r) * NB + j
                lst = qi[row_ptr[row]:row_ptr[row + 1]].tolist()
                assert lst == sorted(lst)
                for t in lst:
                    assert tok_req[t] == r
                    back.setdefault((t, h), []).append(j)
    for t in range(T):
        for h in range(H):
            assert sorted(back.get((t, h), [])) == [j for j in sel[t, h] if j >= 0]


# ---------------------------------------------------------------- cache write
def test_e4m3_encode_round_trips_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_to_float(codes)), codes)


def test_e4m3_encode_matches_torch_on_every_bf16_value_in_range():
    """Every finite bf16 value (all 2^16 bit patterns) whose magnitude is at most
    464 (beyond it torch returns NaN where the cache write saturates) encodes
    to torch's own float8_e4m3fn code: round to nearest, ties to even."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    x = bits.float()
    keep = torch.isfinite(x) & (x.abs() <= 464)
    x = x[keep]
    want = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x.numpy())
    assert np.array_equal(got, want)
    # and scaled by 2^-5, the fp8 workloads' scale, as the cache write divides
    y = (x / 2.0 ** -5)
    ok = y.abs() <= 464
    assert np.array_equal(oracle.e4m3_encode(y[ok].numpy()),
                          y[ok].to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_e4m3_encode_saturates_and_keeps_nan():
    x = np.array([448.0, 464.0, 465.0, 1e6, np.inf, -500.0, -np.inf, np.nan, 2.0 ** -10,
                  3 * 2.0 ** -11, -1e-9])
    want = [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x00, 0x01, 0x80]
    assert oracle.e4m3_encode(x).tolist() == want


def test_cache_slots_hand_computed():
    # request 0: 300 tokens, 1 new -> position 299 = block 2 row 43;
    # request 1: idle; request 2: 130 tokens, 3 new -> positions 127, 128, 129
    bt = [[7, 3, 9], [0, 0, 0], [5, 2, 0]]
    slots = oracle.cache_slots([300, 0, 130], [1, 2, 3], bt, 128)
    assert slots == [9 * 128 + 43, -1, -1, 5 * 128 + 127, 2 * 128 + 0, 2 * 128 + 1]


def test_cache_write_places_rows_and_leaves_the_rest():
    P, H, X = 4, 2, 3
    pool = np.zeros((5, H, P, X))
    rows = np.arange(3 * H * X, dtype=np.float64).reshape(3, H, X) + 1
    out = oracle.cache_write(pool, [2 * P + 3, -1, 0 * P + 1], rows)
    want = np.zeros_like(pool)
    want[2, :, 3, :] = rows[0]
    want[0, :, 1, :] = rows[2]
    assert np.array_equal(out, want) and not pool.any()
    # e4m3: the stored codes are those of float32(x) / float32(scale)
    codes = np.zeros((5, H, P, X), dtype=np.uint8)
    x = np.array([[[0.3, -1.7, 9.0], [100.0, -0.01, 1e4]]])
    out8 = oracle.cache_write(codes, [4 * P], x, e4m3_scale=0.5)
    want8 = torch.tensor(x[0] / 0.5, dtype=torch.float32).clamp(-448, 448).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(out8[4, :, 0, :], want8)
    assert out8.sum() == want8.astype(np.int64).sum()


# ---------------------------------------------------------------- NVFP4
def test_e2m1_codes_are_the_published_value_set():
    """FP4 E2M1 from the format's definition: the eight magnitudes are
    0, 0.5, 1, 1.5, 2, 3, 4, 6 in code order, the sign bit negates."""
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert oracle.e2m1_to_float(np.arange(8)).tolist() == mags
    neg = oracle.e2m1_to_float(np.arange(8, 16))
    assert neg.tolist() == [-m for m in mags] and np.signbit(neg).all()


def test_nvfp4_row_hand_decoded():
    """One 72-byte row built by hand: nibble order (even element low), block
    scale indexing (elements 16b .. 16b + 15 use scale byte b) and the scale
    values (e4m3 codes)."""
    D = 128
    assert oracle.nvfp4_row_bytes(D) == 72
    row = np.zeros(72, dtype=np.uint8)
    row[0] = 0x3 | (0xA << 4)           # element 0: code 3 = 1.5, element 1: code 10 = -1.0
    row[8] = 0x7                         # element 16: 6.0 (block 1), element 17: 0
    row[63] = 0xF << 4                   # element 127: -6.0 (block 7)
    row[64] = 0x38                       # block 0 scale: 1.0
    row[65] = 0x30                       # block 1 scale: 0.5
    row[71] = 0x01                       # block 7 scale: the smallest subnormal, 2^-9
    got = oracle.nvfp4_dequant(row, D)
    want = np.zeros(D)
    want[0], want[1], want[16], want[127] = 1.5, -1.0, 3.0, -6.0 * 2.0 ** -9
    assert np.array_equal(got, want)


def test_e2m1_encode_hand_values():
    """E2M1 rounding from the format's definition: nearest of 0, 0.5, 1, 1.5, 2,
    3, 4, 6; a midpoint goes to the code with mantissa bit 0 (the even code);
    beyond 6 saturates; the sign bit is kept, also on a value that rounds to 0."""
    x = [0.0, 0.25, 0.26, 0.5, 0.75, 1.25, 1.74, 1.75, 2.5, 3.5, 5.0, 5.01, 6.0, 7.0, 1e9,
         -0.1, -0.25, -0.3, -2.5, -100.0, -0.0]
    want = [0, 0, 1, 1, 2, 2, 3, 4, 4, 6, 6, 7, 7, 7, 7,
            8, 8, 9, 12, 15, 8]
    assert oracle.e2m1_encode(np.array(x)).tolist() == want


def test_e2m1_encode_is_nearest_code_by_exhaustive_search():
    """Every multiple of 1/64 in [-8, 8] (every midpoint among them): the code
    is the one of the 16 whose value is nearest, ties to the even code;
    magnitudes beyond 6 take +-6."""
    x = np.arange(-512, 513) / 64.0
    got = oracle.e2m1_encode(x)
    vals = oracle.e2m1_to_float(np.arange(16))
    for xi, c in zip(x, got):
        target = min(max(xi, -6.0), 6.0)
        d = np.abs(vals - target)
        best = [k for k in range(16) if d[k] == d.min() and np.signbit(vals[k]) == np.signbit(xi)]
        if len(best) > 1:
            best = [k for k in best if k % 2 == 0]
        assert c == best[0], (xi, c, best)


def test_nvfp4_quantize_round_trips_representable_blocks():
    """A block whose values are e2m1(code) * e4m3(s) * scale and whose largest
    magnitude is 6 * e4m3(s) * scale quantises back to exactly those codes and
    that scale byte (powers of two as tensor scales keep every product exact)."""
    rng = np.random.default_rng(5)
    D = 128
    for scale in (1.0, 0.5, 2.0 ** -6):
        codes = rng.integers(0, 16, size=(6, D)).astype(np.uint8)
        codes[:, ::16] = rng.choice([7, 15], size=(6, D // 16))   # a +-6 in every block
        sc = rng.integers(0x08, 0x60, size=(6, D // 16)).astype(np.uint8)
        rows = np.zeros((6, oracle.nvfp4_row_bytes(D)), dtype=np.uint8)
        rows[:, :D // 2] = codes[:, 0::2] | (codes[:, 1::2] << 4)
        rows[:, D // 2:] = sc
        x = oracle.nvfp4_dequant(rows, D) * scale
        assert np.array_equal(oracle.nvfp4_quantize(x.astype(np.float32), scale), rows)


def test_nvfp4_quantize_hand_block():
    """One row worked by hand, tensor scale 0.75 (6 * 0.75 = 4.5).
    Block 0: amax 3 -> 3 / 4.5 = 0.667 -> nearest e4m3 0.6875 (0x33; 0.625 is
    farther), divisor 0.6875 * 0.75 = 0.515625; its elements sit at quotients
    5.818 -> 6, 1.25 -> 1 (tie, even), 2.5 -> 2 (tie), 5 -> 4 (tie), 0.75 -> 1
    (tie, even code 2), 0.25 -> 0 (tie), -0.25 -> -0 (sign kept), -1.745 -> -1.5.
    Block 1: all zero -> scale 0, codes 0.  Block 2: amax 3.9 at tensor scale
    0.75 -> 3.9 / 4.5 = 0.8667 -> e4m3 0.875 (0x36), divisor 0.65625,
    3.9 / 0.65625 = 5.94 -> 6.  Block 3: amax 1e4 -> the scale saturates at 448
    (0x7E), divisor 336, 1e4 / 336 = 29.8 -> 6 (saturated).  Block 4: amax 1e-4
    -> 1e-4 / 4.5 rounds to the e4m3 zero -> scale 0 and zero codes."""
    D = 128
    x = np.zeros(D, dtype=np.float32)
    d = 0.515625
    x[0:8] = [3.0, 1.25 * d, 2.5 * d, 5.0 * d, 0.75 * d, 0.25 * d, -0.25 * d, -0.9]
    x[32], x[33] = 3.9, -1.0
    x[48], x[49] = 1e4, -100.0
    x[64], x[65] = 1e-4, -5e-5
    got = oracle.nvfp4_quantize(x, 0.75)
    want = np.zeros(72, dtype=np.uint8)
    want[0:4] = [0x7 | (0x2 << 4), 0x4 | (0x6 << 4), 0x2 | (0x0 << 4), 0x8 | (0xB << 4)]
    want[16] = 0x7 | (0xB << 4)                 # 3.9 -> 6; -1.0 / 0.65625 = -1.52 -> -1.5
    want[24] = 0x7 | (0x9 << 4)                 # 1e4 -> 6; -100 / 336 = -0.298 -> -0.5
    want[64:72] = [0x33, 0x00, 0x36, 0x7E, 0x00, 0x00, 0x00, 0x00]
    assert got.tolist() == want.tolist()


def test_nvfp4_quantize_error_bound_random():
    """Random rows: every element dequantises to within half an E2M1 step (at
    its quotient) of its value, scaled by the block divisor, unless the block
    scale rounded down and the element saturated at 6; then within 6.25% of
    the block's amax (half the relative spacing of normal e4m3 scales, which
    these magnitudes keep)."""
    rng = np.random.default_rng(11)
    D = 128
    x = (rng.standard_normal((64, D)) * rng.choice([0.2, 1.0, 50.0], size=(64, 1))).astype(
        np.float32)
    scale = 0.75
    q = oracle.nvfp4_quantize(x, scale)
    xh = oracle.nvfp4_dequant(q, D) * scale
    div = oracle.e4m3_to_float(q[:, D // 2:]).repeat(16, axis=1) * scale
    u = np.abs(x) / div
    step = np.where(u < 2, 0.5, np.where(u < 4, 1.0, 2.0))
    amax = np.abs(x.reshape(64, 8, 16)).max(-1).repeat(16, axis=1)
    err = np.abs(xh - x)
    ok = (err <= 0.5 * step * div * (1 + 1e-5)) | ((u > 6) & (err <= 0.0625 * amax * (1 + 1e-5)))
    assert (q[:, D // 2:] >= 0x08).all()   # normal scales only
    assert ok.all()


def test_cache_write_nvfp4_places_slots():
    """Keys go to slot 2h, values to slot 2h + 1 of the token's page row; the
    other slots and rows keep their bytes."""
    P, H, D = 4, 2, 32
    RB = oracle.nvfp4_row_bytes(D)
    pool = np.full((3, 2 * H, P, RB), 0xAB, dtype=np.uint8)
    rows = np.arange(2 * H * D, dtype=np.float32).reshape(2, H, D) / 7.0 - 5.0
    k_out = oracle.cache_write_nvfp4(pool, [1 * P + 2, -1], rows, 0.5, 0)
    v_out = oracle.cache_write_nvfp4(pool, [1 * P + 2, -1], rows, 0.5, 1)
    want_k, want_v = pool.copy(), pool.copy()
    for h in range(H):
        want_k[1, 2 * h, 2] = oracle.nvfp4_quantize(rows[0, h], 0.5)
        want_v[1, 2 * h + 1, 2] = oracle.nvfp4_quantize(rows[0, h], 0.5)
    assert np.array_equal(k_out, want_k) and np.array_equal(v_out, want_v)
    assert (pool == 0xAB).all()


def test_nvfp4_path_uses_dequantised_values():
    """Attention over an NVFP4 pool equals attention over the float pools that
    hold its dequantised values times the tensor scales (K from slot 2h, V from
    slot 2h + 1)."""
    spec = wl.small("nvfp4_decode", batch=2, seq_len_range=(300, 700), num_pages=16,
                    num_q_heads=8, num_kv_heads=2)
    w = wl.make_workload(spec)
    res = run_oracle(w)
    pool = to_np(w.k_pages)
    P, D = spec.block_size, spec.head_dim
    kf = oracle.nvfp4_dequant(pool[:, 0::2].astype(np.uint8), D) * 0.75
    vf = oracle.nvfp4_dequant(pool[:, 1::2].astype(np.uint8), D) * 0.75
    plain = oracle.sparse_attention(
        seq_lens=to_np(w.seq_lens), q_lens=to_np(w.q_lens), block_table=to_np(w.block_table),
        idx_q=to_np(w.idx_q), idx_k_pages=to_np(w.idx_k_pages), q=to_np(w.q), k_pages=kf,
        v_pages=vf, num_kv_heads=spec.num_kv_heads, block_size=P, init_blocks=1,
        local_blocks=oracle_local_blocks(w), topk_blocks=spec.topk_blocks,
        softmax_scale=spec.softmax_scale)
    assert spec.kv_scale == 0.75
    assert np.array_equal(res["out"], plain["out"]) and np.array_equal(res["lse"], plain["lse"])
    assert kf.max() <= 6 * 1.0 * 0.75 and np.abs(vf).max() > 0


# ---------------------------------------------------------------- dense-sparse decode
def test_compact_selection_hand_computed():
    bt = [40, 41, 42, 43, 44, 45, 46, 47]
    pages, n = oracle.compact_selection([7, 0, 3], bt, 7 * 128 + 5, 128)
    assert pages == [40, 43, 47] and n == 2 * 128 + 6
    pages, n = oracle.compact_selection([0, 1], bt, 1 * 128 + 127, 128)
    assert pages == [40, 41] and n == 256
    assert oracle.compact_selection([], bt, 5, 128) == ([], 0)


def test_dense_sparse_equals_sparse_attention():
    """The compacted sequence holds exactly the selected blocks' visible keys,
    in order, so the dense paged decode over it reproduces the sparse result
    bit for bit (same rows, same order, same arithmetic)."""
    spec = wl.small("verify", batch=2, seq_lens=(900, 1100), num_pages=24, num_q_heads=16,
                    num_kv_heads=2)
    w = wl.make_workload(spec)
    res = run_oracle(w)
    bt, q = to_np(w.block_table), to_np(w.q)
    kp, vp = to_np(w.k_pages), to_np(w.v_pages)
    toks = oracle.query_positions(to_np(w.seq_lens), to_np(w.q_lens))
    G = spec.group
    for t, (r, p) in enumerate(toks):
        for h in range(spec.num_kv_heads):
            pages, n = oracle.compact_selection(res["selected"][(t, h)], bt[r], p, 128)
            o, l = oracle.paged_attention(q[t, h * G:(h + 1) * G], kp, vp, pages, n, h,
                                          spec.softmax_scale, 128)
            assert np.array_equal(o, res["out"][t, h * G:(h + 1) * G])
            assert np.array_equal(l, res["lse"][t, h * G:(h + 1) * G])


# ---------------------------------------------------------------- index-value branch
def test_index_attention_is_softmax_over_visible_tokens():
    """The reading itself is unpinned (the pages give no formula for idx_o);
    what is pinned is that the function computes what it states: scipy's
    softmax of idx_q . idx_k / sqrt(d) over tokens <= position, applied to
    idx_v, and a single visible token returns its own value row."""
    rng = np.random.default_rng(4)
    d, n = 64, 300
    q = rng.integers(-4, 5, d).astype(np.float64)
    k = rng.integers(-4, 5, (n, d)).astype(np.float64)
    v = rng.standard_normal((n, d))
    for pos in (0, 17, 299):
        o, lse = oracle.index_attention(q, k, v, pos)
        logits = k[:pos + 1] @ q / math.sqrt(d)
        w = scipy.special.softmax(logits)
        assert np.allclose(o, w @ v[:pos + 1], rtol=0, atol=1e-12)
        assert abs(lse - scipy.special.logsumexp(logits)) < 1e-12
    o, _ = oracle.index_attention(q, k, v, 0)
    assert np.allclose(o, v[0], atol=1e-15)


# ---------------------------------------------------------------- mutations
def _mutants():
    """Plausible mistakes, each planted in a copy of one oracle function."""
    real_scores, real_select = oracle.block_scores, oracle.select_blocks
    real_attn, real_combine = oracle.attention, oracle.combine

    def scores_sum(q, seq, pos, P):      # sum instead of max
        nb = pos // P + 1
        dots = seq[:pos + 1] @ q
        return np.array([dots[j * P:(j + 1) * P].sum() for j in range(nb)])

    def scores_no_causal(q, seq, pos, P):  # last block not masked at the position
        nb = pos // P + 1
        dots = seq @ q
        return np.array([dots[j * P:(j + 1) * P].max() for j in range(nb)])

    def select_high_tie(scores, i, l, k):  # ties toward the higher index
        nb = len(scores)
        I = set(range(min(i, nb))); L = set(range(max(0, nb - l), nb))
        C = [j for j in range(nb) if j not in I | L]
        top = sorted(C, key=lambda j: (-scores[j], -j))[:k]
        return sorted(I | L | set(top))

    def select_local_off_by_one(scores, i, l, k):
        return real_select(scores, i, l - 1, k + 1)

    def attn_no_scale(q, k, v, scale):
        return real_attn(q, k, v, 1.0)

    def attn_transposed_v(q, k, v, scale):
        o, l = real_attn(q, k, v, scale)
        return o[:, ::-1], l

    def combine_lse_is_max(o, l):        # drops the log-sum term of the lse
        out, _ = real_combine(o, l)
        return out, float(np.max(l))

    real_encode, real_slots = oracle.e4m3_encode, oracle.cache_slots

    def encode_ties_away(x):             # round half away from zero
        x = np.asarray(x, dtype=np.float64)
        nudged = np.nextafter(np.abs(x), np.inf) * np.sign(x)
        return real_encode(np.where(np.isnan(x), x, nudged))

    def slots_one_late(seq_lens, q_lens, bt, P):   # position seq_len - q_len + i + 1
        return real_slots([L + (L > 0) for L in seq_lens], q_lens, bt, P)

    real_e2m1 = oracle.e2m1_to_float
    real_nvfp4 = oracle.nvfp4_dequant

    def e2m1_no_subnormal(codes):        # exponent 0 read as a normal number
        c = np.asarray(codes, dtype=np.uint8) & 0xF
        v = real_e2m1(c)
        sub = ((c >> 1) & 3) == 0
        return np.where(sub & ((c & 1) == 1), np.where(c & 8, -1.5, 1.5), v)

    def nvfp4_nibbles_swapped(rows, D):  # odd element in the low nibble
        rows = np.asarray(rows, dtype=np.uint8).copy()
        rows[..., :D // 2] = (rows[..., :D // 2] >> 4) | ((rows[..., :D // 2] & 0xF) << 4)
        return real_nvfp4(rows, D)

    real_compact = oracle.compact_selection

    def compact_all_full(selected, bt_row, position, P):   # the partial last block counted full
        pages, n = real_compact(selected, bt_row, position, P)
        return pages, P * len(pages)

    real_e2m1_enc, real_quant = oracle.e2m1_encode, oracle.nvfp4_quantize

    def e2m1_ties_away(x):                # round half away from zero
        x = np.asarray(x, dtype=np.float64)
        return real_e2m1_enc(np.nextafter(np.abs(x), np.inf) * np.where(np.signbit(x), -1, 1))

    def quant_no_tensor_scale(x, scale):  # the block scale from amax / 6 alone
        x = np.asarray(x, dtype=np.float32)
        D = x.shape[-1]
        out = real_quant(x, 1.0)
        div = (oracle.e4m3_to_float(out[..., D // 2:]) * scale).repeat(16, axis=-1)
        with np.errstate(divide="ignore", invalid="ignore"):
            c = np.where(div == 0, 0, real_e2m1_enc(x / div)).astype(np.uint8)
        out[..., :D // 2] = c[..., 0::2] | (c[..., 1::2] << 4)
        return out

    def quant_scale_from_mean(x, scale):  # the block scale from the mean magnitude
        x = np.asarray(x, dtype=np.float32)
        b = np.abs(x.reshape(x.shape[:-1] + (-1, 16)))
        ratio = (b.max(-1) / np.maximum(b.mean(-1), 1e-30)).repeat(16, axis=-1)
        return real_quant(np.where(b.reshape(x.shape) > 0, x / ratio.reshape(x.shape), x), scale)

    real_cw4 = oracle.cache_write_nvfp4

    def cw4_slot_swapped(pool, slots, rows, scale, kind):   # values in the key slot
        return real_cw4(pool, slots, rows, scale, 1 - kind)

    return [("compact_selection", compact_all_full),
            ("e2m1_encode", e2m1_ties_away), ("nvfp4_quantize", quant_no_tensor_scale),
            ("nvfp4_quantize", quant_scale_from_mean), ("cache_write_nvfp4", cw4_slot_swapped),
            ("e2m1_to_float", e2m1_no_subnormal), ("nvfp4_dequant", nvfp4_nibbles_swapped),
            ("e4m3_encode", encode_ties_away), ("cache_slots", slots_one_late),
            ("block_scores", scores_sum), ("block_scores", scores_no_causal),
            ("select_blocks", select_high_tie), ("select_blocks", select_local_off_by_one),
            ("attention", attn_no_scale), ("attention", attn_transposed_v),
            ("combine", combine_lse_is_max)]


_PINS = [
    test_block_scores_exact_against_integer_brute_force,
    lambda: [test_selection_hand_computed(c) for c in _golden("selection_cases.json")["cases"]],
    test_selection_invariants_random,
    test_selection_against_exhaustive_subset_search,
    test_attention_special_cases,
    test_combine_equals_unsplit,
    test_dense_when_topk_covers_every_block,
    test_sparse_equals_dense_over_selected_tokens,
    test_e4m3_encode_round_trips_every_finite_code,
    test_e4m3_encode_matches_torch_on_every_bf16_value_in_range,
    test_e4m3_encode_saturates_and_keeps_nan,
    test_cache_slots_hand_computed,
    test_cache_write_places_rows_and_leaves_the_rest,
    test_e2m1_codes_are_the_published_value_set,
    test_nvfp4_row_hand_decoded,
    test_e2m1_encode_hand_values,
    test_e2m1_encode_is_nearest_code_by_exhaustive_search,
    test_nvfp4_quantize_round_trips_representable_blocks,
    test_nvfp4_quantize_hand_block,
    test_nvfp4_quantize_error_bound_random,
    test_cache_write_nvfp4_places_slots,
    test_compact_selection_hand_computed,
]


@pytest.mark.parametrize("mutant", _mutants(), ids=lambda m: f"{m[0]}:{m[1].__name__}")
def test_pins_catch_planted_mistake(mutant, monkeypatch):
    name, fn = mutant
    monkeypatch.setattr(oracle, name, fn)
    monkeypatch.setattr(oracle.msa_oracle, name, fn)
    caught = 0
    for pin in _PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught += 1
    assert caught > 0, f"no pin caught the mutant {fn.__name__}"
