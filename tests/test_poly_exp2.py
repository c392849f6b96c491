"""The FMA-pipe 2^x used for part of the prefill softmax: range reduction to
f in [-1/2, 1/2] plus a degree-3 minimax polynomial.  Emulated step by step in float32 and
checked against numpy's exp2: relative error below 1e-4 (the fit's bound is 7.5e-5, under
the rounding of the 16-bit P it feeds), and ~0 for very negative arguments."""
import re
import os

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "paged_kv_varlen_flashattention_gb300", "csrc", "device_common.cuh")


def coefficients():
    body = open(SRC).read()
    body = body[body.index("poly_exp2(float x)"):]
    body = body[:body.index("}")]
    c = [float(v) for v in re.findall(r"fmaf\([^;]*?([0-9]\.[0-9]+)f\)", body)]
    lead = float(re.search(r"fmaf\(([0-9.]+)f, f,", body).group(1))
    return lead, c


def emulate(x):
    f32 = np.float32
    lead, (c2, c1, c0) = coefficients()
    x = np.maximum(x.astype(f32), f32(-126.0))
    t = (x + f32(12582912.0)).astype(f32)
    n = (t - f32(12582912.0)).astype(f32)
    f = (x - n).astype(f32)
    p = (f32(lead) * f + f32(c2)).astype(f32)
    p = (p * f + f32(c1)).astype(f32)
    p = (p * f + f32(c0)).astype(f32)
    bits = p.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)
    return ((bits + (1 << 31)) % (1 << 32) - (1 << 31)).astype(np.int32).view(np.float32)


def test_relative_error_bound():
    x = np.linspace(-30.0, 8.0, 400001, dtype=np.float32)
    got = emulate(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got - want) / want
    assert rel.max() < 1e-4, rel.max()


def test_very_negative_and_masked_arguments_vanish():
    x = np.array([-126.5, -200.0, -1e30, -np.inf], dtype=np.float32)
    got = emulate(x)
    assert np.all(np.abs(got) < 1e-37)
