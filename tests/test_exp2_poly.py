"""The FMA-pipe exp2 used for part of the attention probabilities: its coefficients (read from
the CUDA header) and its range reduction, evaluated in float32 here, stay within the stated
relative error bound of 2^x, and x <= -127 gives exactly 0."""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def coefficients():
    src = open(os.path.join(ROOT, "free_block_sparse_gb300", "csrc", "common.cuh")).read()
    return [np.float32(float(re.search(r"EXP2_C%d = ([0-9.e+-]+)f;" % k, src).group(1))) for k in (1, 2, 3)]


def exp2_poly(x):
    c1, c2, c3 = coefficients()
    x = np.maximum(np.asarray(x, np.float32), np.float32(-127.0))
    rnd = np.float32(12582912.0)
    t = (x + rnd).astype(np.float32)
    n = (t - rnd).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = ((f * c3 + c2) * f + c1) * f + np.float32(1.0)
    bits = p.astype(np.float32).view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.view(np.float32)


def test_relative_error_bound():
    x = np.linspace(-120.0, 8.0, 2_000_001, dtype=np.float32)
    got = exp2_poly(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(got - ref) / ref) < 1.05e-4


def test_masked_inputs_give_zero():
    assert exp2_poly(np.array([-np.inf, -127.0, -200.0], np.float32)).tolist() == [0.0, 0.0, 0.0]
    assert exp2_poly(np.array([0.0], np.float32))[0] == 1.0
