"""The FMA-pipe 2^x of the head-dim-128 backward kernel (exp2_fma), emulated step by step in
float32 with the constants read from the kernel source, against numpy's exp2:
relative error far below a bf16 half-ulp on the range P takes, exact powers of two at the
integers, and the clamp keeping the result a normal float."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(__file__), "..", "reproducible_deterministic_attn_gb300",
                   "csrc", "kernels_tc128.cuh")


def _consts():
    text = open(SRC).read()
    body = text[text.index("float exp2_fma(float x)"):]
    body = body[:body.index("}")]
    vals = dict(re.findall(r"(c[0-3]) = ([0-9.eE+-]+)f", body))
    kround = float(re.search(r"kRound = ([0-9.]+)f", body).group(1))
    return [np.float32(vals["c%d" % k]) for k in range(4)], np.float32(kround)


def exp2_fma(x):
    (c0, c1, c2, c3), kround = _consts()
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-126.0))
    t = (x + kround).astype(np.float32)
    f = (x - (t - kround)).astype(np.float32)
    p = (((c3 * f + c2) * f + c1) * f + c0).astype(np.float32)
    bits = (p.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23))
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def test_kround_is_one_and_a_half_times_two_to_the_23():
    _, kround = _consts()
    assert kround == np.float32(1.5 * 2 ** 23)


def test_relative_error_on_the_range_of_p():
    x = np.linspace(-120.0, 0.5, 400001, dtype=np.float32)
    got = exp2_fma(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got - want) / want
    assert rel.max() < 1e-4, rel.max()          # a bf16 half-ulp is 1.95e-3


def test_integers_and_half_integers():
    n = np.arange(-125, 1, dtype=np.float32)
    got = exp2_fma(n).astype(np.float64)
    assert np.all(np.abs(got / np.exp2(n.astype(np.float64)) - 1) < 1e-4)
    h = n + np.float32(0.5)                     # round-half-even boundary of the reduction
    got = exp2_fma(h).astype(np.float64)
    assert np.all(np.abs(got / np.exp2(h.astype(np.float64)) - 1) < 1e-4)


def test_clamp_keeps_a_tiny_normal_value():
    got = exp2_fma(np.array([-126.0, -200.0, -1e30], dtype=np.float32))
    assert np.all(got > 0) and np.all(got < 2.0 ** -125)
    assert np.all(np.isfinite(got))
