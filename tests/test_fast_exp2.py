"""The FMA-pipe exp2 used by the prefill attention softmax: the header's
coefficients and range reduction, replayed in float32 on the host, must stay
within 5e-6 relative error of 2^x over the range a softmax feeds it."""

import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(__file__), "..", "transformer_decoder_layer_gb300", "csrc",
                   "fast_exp2.cuh")


def _coeffs():
    src = open(HDR).read()
    c = {int(k): np.float32(v) for k, v in re.findall(r"kExp2C(\d) = ([0-9.e+-]+)f;", src)}
    assert sorted(c) == [0, 1, 2, 3, 4]
    return [c[i] for i in range(5)]


def _exp2_fma(x):
    c0, c1, c2, c3, c4 = _coeffs()
    x = np.maximum(x.astype(np.float32), np.float32(-125.0))
    t = (x + np.float32(12582912.0)).astype(np.float32)
    n = (t - np.float32(12582912.0)).astype(np.float32)
    f = (x - n).astype(np.float32)
    # each fmaf rounds once: exact product and sum in float64, one rounding to float32
    p = (np.float64(c4) * f + c3).astype(np.float32)
    p = (p.astype(np.float64) * f + c2).astype(np.float32)
    p = (p.astype(np.float64) * f + c1).astype(np.float32)
    p = (p.astype(np.float64) * f + c0).astype(np.float32)
    bits = p.view(np.int32) + (t.view(np.int32) << 23)
    return bits.astype(np.int32).view(np.float32)


def test_exp2_fma_relative_error():
    x = np.linspace(-124.0, 8.0, 2_000_001, dtype=np.float64).astype(np.float32)
    got = _exp2_fma(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(got / ref - 1.0)) < 5e-6


def test_exp2_fma_integers_and_clamp():
    x = np.arange(-125, 9, dtype=np.float32)
    got = _exp2_fma(x).astype(np.float64)
    assert np.allclose(got, np.exp2(x.astype(np.float64)), rtol=5e-6, atol=0)
    # far below the range the result is 2^-125 (zero once rounded to FP16)
    low = _exp2_fma(np.array([-200.0, -np.inf], dtype=np.float32)).astype(np.float64)
    assert np.allclose(low, 2.0 ** -125, rtol=5e-6)
