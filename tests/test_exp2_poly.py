"""The FMA-pipe 2^x of the attention softmax (exp2_poly in msa_device.cuh).

The device helper splits x <= 0 into round(x) and a fraction in [-0.5, 0.5]. It evaluates a
degree-3 polynomial for 2^fraction and adds round(x) to the exponent bits. This test reads its
constants from the header and re-runs the same float32 steps on the host against 2^x in float64.
"""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "block_sparse_attention_04_gb300", "csrc", "msa_device.cuh")


def coefficients():
    src = open(HDR).read()
    c = {int(k): float(v.rstrip("f")) for k, v in re.findall(r"kExp2C(\d) = ([0-9.e+-]+f)", src)}
    assert sorted(c) == [0, 1, 2, 3]
    return [np.float32(c[k]) for k in range(4)]


def fma32(a, b, c):
    # one rounding, as the device FFMA does
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(np.float32)


def exp2_poly_host(x):
    c0, c1, c2, c3 = coefficients()
    x = np.maximum(x.astype(np.float32), np.float32(-126.0))
    t = (x + np.float32(12582912.0)).astype(np.float32)
    f = (x - (t - np.float32(12582912.0))).astype(np.float32)
    p = fma32(fma32(fma32(np.full_like(f, c3), f, np.full_like(f, c2)), f,
                    np.full_like(f, c1)), f, np.full_like(f, c0))
    bits = p.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)
    return ((bits & 0xFFFFFFFF).astype(np.uint32)).view(np.float32)


def test_relative_error_over_the_softmax_range():
    x = np.concatenate([np.linspace(-125.0, 0.0, 2_000_001), -np.logspace(-8, 0, 10001)])
    x = x.astype(np.float32)
    got = exp2_poly_host(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got / want - 1)
    assert rel.max() < 1e-4, rel.max()          # bf16 rounding of P is 2^-9 ~ 2e-3


def test_integers_and_halves_land_on_powers_of_two():
    for j in range(-120, 1):
        v = float(exp2_poly_host(np.array([j], np.float32))[0])
        assert abs(v / 2.0 ** j - 1) < 1e-4, (j, v)
    # round-half cases split either way and stay continuous
    x = np.array([-0.5, -1.5, -2.5, -10.5], np.float32)
    assert np.all(np.abs(exp2_poly_host(x) / np.exp2(x.astype(np.float64)) - 1) < 1e-4)


def test_far_below_range_is_tiny_not_garbage():
    x = np.array([-126.0, -200.0, -1e6, -3.0e38], np.float32)
    v = exp2_poly_host(x)
    assert np.all(np.isfinite(v)) and np.all(v >= 0) and np.all(v < 1e-37)

