"""The FMA-pipe 2^x used for half of the tensor-core softmax's exponentials.

The coefficients are read from the kernel source and evaluated with float32
arithmetic in the same order as the device code (Horner form, exponent added
to the bit pattern), then checked against exp2 in double precision.  The
tensor-core prefill rounds P to fp16 (2^-11) or to bf16 hi+lo (~2^-17), so a
relative error below 3e-6 is far under what the output can show."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "paged_kv_decode_ns_gb300", "csrc", "ns_common.cuh")


def _coeffs():
    body = open(SRC).read().split("float exp2_fma(float x)")[1].split("return")[0]
    body = body.split("const float f = x - n;")[1]      # the polynomial only
    return [np.float32(v) for v in re.findall(r"([0-9]+\.[0-9]+)f", body)]


def _exp2_fma(x):
    c = _coeffs()
    assert len(c) == 5
    xm = np.maximum(x, np.float32(-127.0))
    n = np.floor(xm).astype(np.float32)
    f = (xm - n).astype(np.float32)
    p = (c[0] * f + c[1]).astype(np.float32)
    for k in c[2:]:
        p = (p * f + k).astype(np.float32)
    return (p.view(np.int32) + (n.astype(np.int32) << 23)).view(np.float32)


def test_relative_error_bound():
    x = np.linspace(-126.0, 8.0, 1_000_001).astype(np.float32)
    got = _exp2_fma(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(got / ref - 1)) < 3e-6


def test_exact_at_integers_and_monotone_near_them():
    x = np.arange(-120, 9, dtype=np.float32)
    got = _exp2_fma(x).astype(np.float64)
    assert np.max(np.abs(got / np.exp2(x.astype(np.float64)) - 1)) < 3e-6
    # across each integer boundary the value does not jump down
    eps = np.float32(1e-6)
    assert np.all(_exp2_fma(x + eps) >= _exp2_fma(x - eps))
