"""The byte-range narrowing of the warp top-k's radix select
(topk_warp_kernel in block_sparse_paged_msa_gb300/csrc/topk.cu), replayed on
the CPU and checked against a brute-force sort by (key desc, index asc).

The kernel finds the key of the K-th best candidate 8 bits at a time from the
top, but only over the bytes where the candidates' keys differ: diff = OR over
candidates of (key ^ largest key); above diff's highest byte every key equals
the largest key's bits, below its lowest byte every key carries the same bits.
A plausible mistake, taking diff = smallest ^ largest key, misses low bits in
which a middle key differs from both; the clustered cases below catch it.
(The device code itself is covered by the GPU parity tests.)"""
import random


def select(keys, K, diff_fn):
    """(threshold key, how many keys equal to it win)."""
    if K == len(keys):
        return 0, 0
    kmax = max(keys)
    diff = diff_fn(keys, kmax)
    if diff:
        top = ((diff.bit_length() - 1) >> 3) << 3
        bot = (((diff & -diff).bit_length() - 1) >> 3) << 3
    else:
        top, bot = -8, 0
    mask = 0 if top >= 24 else (0xFFFFFFFF << (top + 8)) & 0xFFFFFFFF
    prefix = kmax & mask
    krem = K
    for shift in range(top, bot - 1, -8):
        hist = [0] * 256
        for k in keys:
            if (k & mask) == prefix:
                hist[(k >> shift) & 255] += 1
        c = 0
        for b in range(255, -1, -1):
            if c + hist[b] >= krem:
                krem -= c
                break
            c += hist[b]
        prefix |= b << shift
        mask |= 0xFF << shift
    return prefix | (kmax & ~mask & 0xFFFFFFFF), krem


def winners(keys, K, diff_fn):
    thr, ktie = select(keys, K, diff_fn)
    if K == len(keys):
        return list(range(len(keys)))
    out, tie = [], 0
    for i, k in enumerate(keys):
        if k > thr:
            out.append(i)
        elif k == thr:
            if tie < ktie:
                out.append(i)
            tie += 1
    return out


def brute(keys, K):
    return sorted(sorted(range(len(keys)), key=lambda i: (-keys[i], i))[:K])


def or_diff(keys, kmax):
    d = 0
    for k in keys:
        d |= k ^ kmax
    return d


def draw(rng, n, mode):
    if mode == 0:
        return [rng.getrandbits(32) | 1 for _ in range(n)]
    if mode == 1:   # integer-valued scores in [128, 256): one exponent
        return [0xC3000000 | (rng.randint(0, 127) << 16) for _ in range(n)]
    if mode == 2:   # middle keys differing in low bits where min and max agree
        return [0xC3000000 | (rng.randint(0, 3) << 16) | (rng.randint(0, 3) << 1) for _ in range(n)]
    return [rng.choice([5, 9, 9, 0x80000000, 0x80000001]) for _ in range(n)]   # heavy ties


def test_narrowed_select_equals_brute_force():
    rng = random.Random(0)
    for trial in range(4000):
        n = rng.randint(1, 300)
        K = rng.randint(0, n)
        keys = draw(rng, n, trial % 4)
        assert winners(keys, K, or_diff) == brute(keys, K), (trial, K)


def test_min_max_difference_is_not_enough():
    rng = random.Random(1)
    minmax = lambda keys, kmax: min(keys) ^ kmax
    wrong = 0
    for _ in range(2000):
        n = rng.randint(2, 300)
        K = rng.randint(1, n - 1)
        keys = draw(rng, n, 2)
        wrong += winners(keys, K, minmax) != brute(keys, K)
    assert wrong > 0
