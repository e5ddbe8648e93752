"""The FMA-pipe exp2 of the prefill kernel (exp2_fma2 in csrc/ptx.cuh), checked on
the CPU against its stated error bound: the coefficients in the CUDA source,
evaluated the way the kernel evaluates them (range reduction to [-1/2, 1/2],
fp32 Horner steps, exponent added to the bits), against numpy's exp2."""

import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PTX = os.path.join(ROOT, "attention_flashattention_fwd_03_gb300", "csrc", "ptx.cuh")


def _coefficients():
    with open(PTX) as fh:
        src = fh.read()
    body = src[src.index("float2 exp2_fma2("):]
    body = body[:body.index("\n}\n")]
    vals = [float(v.rstrip("f")) for v in re.findall(r"make_float2\((-?\d\.\d+f?), \1\)", body)
            if abs(float(v.rstrip("f"))) < 2]
    c3, c2, c1, c0 = vals[-4:]
    return np.float32(c0), np.float32(c1), np.float32(c2), np.float32(c3)


def _exp2_like_kernel(x):
    c0, c1, c2, c3 = _coefficients()
    x = np.maximum(x.astype(np.float32), np.float32(-126.0))
    t = (x + np.float32(12582912.0)).astype(np.float32)
    n = (t - np.float32(12582912.0)).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = (c3 * f + c2).astype(np.float32)
    p = (p * f + c1).astype(np.float32)
    p = (p * f + c0).astype(np.float32)
    bits = p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.view(np.float32)


def test_exp2_poly_relative_error_bound():
    x = np.linspace(-125.9, 8.0, 400001).astype(np.float32)
    got = _exp2_like_kernel(x).astype(np.float64)
    exp = np.exp2(x.astype(np.float64))
    rel = np.abs(got - exp) / exp
    assert rel.max() <= 1.0e-4, rel.max()  # far below bf16's 2^-9 relative rounding


def test_exp2_poly_is_exact_at_integers_and_monotone():
    x = np.arange(-120, 9, dtype=np.float32)
    got = _exp2_like_kernel(x)
    assert np.all(np.abs(got / np.exp2(x) - 1) <= 1e-4)
    y = _exp2_like_kernel(np.linspace(-20, 8, 100001).astype(np.float32))
    assert np.all(np.diff(y) >= 0)
