"""The FMA-pipe exp2 of the prefill softmax (exp2_poly2 in
block_sparse_paged_msa_gb300/csrc/msa_device.cuh), replayed step by step in
fp32 on the CPU with the coefficients read from that header: relative error
within 1e-4 of 2^x over the range that matters to an fp16 probability, no
sign or exponent wrap for very negative x, and exact powers of two at the
integers up to the cubic's constant term.  (The device path is also covered
end to end by the prefill parity tests.)"""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "block_sparse_paged_msa_gb300", "csrc", "msa_device.cuh")


def coefficients():
    text = open(HDR).read()
    c = {int(k): np.float32(v) for k, v in re.findall(r"kExp2C(\d) = ([0-9.eE+-]+)f;", text)}
    assert sorted(c) == [0, 1, 2, 3]
    return [c[i] for i in range(4)]


def exp2_poly(x):
    """The device steps in fp32: clamp, round by the 1.5 * 2^23 shift, cubic in
    f = x - n (Horner, one rounding per step), n added to the exponent bits."""
    c0, c1, c2, c3 = coefficients()
    x = np.maximum(x.astype(np.float32), np.float32(-126.0))
    shift = np.float32(12582912.0)
    t = (x + shift).astype(np.float32)
    n = (t - shift).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = (c3 * f + c2).astype(np.float32)
    p = (p * f + c1).astype(np.float32)
    p = (p * f + c0).astype(np.float32)
    bits = p.view(np.uint32).astype(np.uint64) + ((t.view(np.uint32).astype(np.uint64) << 23) & 0xFFFFFFFF)
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_relative_error_bound():
    x = np.linspace(-60.0, 0.0, 2_000_001).astype(np.float32)
    got = exp2_poly(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got / want - 1.0)
    assert rel.max() < 1e-4, rel.max()


def test_fraction_grid_near_zero():
    # every fp32 value in [-1, 0] on a fine grid, where P ~ 1 matters most
    x = -np.arange(0, 1 << 20, dtype=np.float32) / np.float32(1 << 20)
    rel = np.abs(exp2_poly(x).astype(np.float64) / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < 1e-4


def test_very_negative_inputs_underflow_cleanly():
    x = np.array([-126.0, -127.0, -200.0, -1e30, -np.inf], dtype=np.float32)
    got = exp2_poly(x)
    assert np.all(got >= 0.0) and np.all(np.isfinite(got))
    assert np.all(got < 2.0 ** -120)
    # fp16 (the P operand) rounds them to zero
    assert np.all(got.astype(np.float16) == 0)


def test_integers_scale_by_powers_of_two():
    c0 = coefficients()[0]
    for k in range(0, 120):
        y = exp2_poly(np.array([-float(k)], dtype=np.float32))[0]
        assert y == np.float32(c0) * np.float32(2.0 ** -k), k
