"""The FMA-pipe exp2 used for a share of the softmax's exponentials: its cubic's
coefficients in vdit_ptx.cuh are the ones the committed generator fits, and the
float32 evaluation (range reduction r = round(x), f = x - r in [-1/2, 1/2], 2^r
added to the exponent field) stays within the stated relative error against
float64 2^x over the whole input range the kernel uses."""
import importlib.util
import os
import re

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "block_sparse_video_frame_gb300", "csrc")


def _gen():
    spec = importlib.util.spec_from_file_location("gen_exp2_poly", os.path.join(CSRC, "gen_exp2_poly.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _header_coeffs():
    text = open(os.path.join(CSRC, "vdit_ptx.cuh")).read()
    m = re.search(r"kC1 = ([0-9.e+-]+)f, kC2 = ([0-9.e+-]+)f, kC3 = ([0-9.e+-]+)f", text)
    return np.array([1.0] + [float(x) for x in m.groups()], dtype=np.float32)


def emulate_exp2_fma(x):
    """float32 emulation of exp2_fma: the same operations in the same order."""
    c = _header_coeffs()
    x = np.maximum(np.asarray(x, dtype=np.float32), np.float32(-126.0))
    t = (x + np.float32(12582912.0)).astype(np.float32)
    f = (x - (t - np.float32(12582912.0)).astype(np.float32)).astype(np.float32)
    p = np.float32(c[3])
    for ci in (c[2], c[1], c[0]):
        p = (p * f + np.float32(ci)).astype(np.float32)
    bits = (p.view(np.int32).astype(np.int64) + (t.view(np.int32).astype(np.int64) << 23)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(np.float32)


def test_header_matches_generator():
    gen = _gen()
    np.testing.assert_array_equal(_header_coeffs(), gen.COEFFS)
    assert gen.max_rel_error(gen.COEFFS) < gen.MAX_REL_ERR


def test_full_range_relative_error():
    x = np.linspace(-100.0, 8.0, 400001).astype(np.float32)
    got = emulate_exp2_fma(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(got - want) / want) < _gen().MAX_REL_ERR
    assert emulate_exp2_fma(np.float32(0.0)) == np.float32(1.0)


def test_clamp_below_normal_range():
    y = emulate_exp2_fma(np.array([-126.0, -200.0, -1e30], dtype=np.float32))
    assert np.all(y >= 0) and np.all(y <= np.float32(2.0 ** -125))
