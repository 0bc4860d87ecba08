"""The kernels' softplus: max(x,0) + m·P(m²), m = e/(2+e), e = 2^(-|x|·log2 e), i.e. the identity
log1p(e) = 2·atanh(m).  Emulated here in fp32 with the coefficients read from the CUDA header,
against numpy.logaddexp(0, x) in fp64 (CPU only)."""
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HDR = os.path.join(ROOT, "selective_state_space_scan_gb300", "csrc", "device_common.cuh")


def _coeffs():
    text = open(HDR).read()
    c = [float(re.search(rf"kLog1pP{k}\s*=\s*([0-9.eE+-]+)f", text).group(1)) for k in range(5)]
    return np.array(c, np.float32)


def _softplus_fp32(x):
    f = np.float32
    c = _coeffs()
    x = x.astype(np.float32)
    e = np.exp2((-np.abs(x) * f(1.4426950408889634)).astype(np.float32)).astype(np.float32)
    m = (e * (f(1) / (f(2) + e)).astype(np.float32)).astype(np.float32)
    w = (m * m).astype(np.float32)
    p = c[4]
    for k in (3, 2, 1, 0):
        p = (p * w + c[k]).astype(np.float32)
    return (m.astype(np.float64) * p + np.maximum(x, 0)).astype(np.float32)


def test_polynomial_matches_atanh_series():
    w = np.linspace(0.0, 1.0 / 9.0, 10001)
    c = _coeffs().astype(np.float64)
    P = sum(c[k] * w ** k for k in range(5))
    m = np.sqrt(w[1:])
    exact = np.concatenate([[2.0], 2 * np.arctanh(m) / m])
    assert np.max(np.abs(P - exact) / exact) < 1e-8


def test_fp32_softplus_accuracy():
    xs = np.concatenate([np.linspace(-8, 2, 200001), np.linspace(-30, 30, 60001)]).astype(np.float32)
    ref = np.logaddexp(0.0, xs.astype(np.float64))
    got = _softplus_fp32(xs)
    rel = np.abs(got - ref) / ref
    core = (xs > -8) & (xs < 2)
    assert rel[core].max() < 7e-7
    assert rel.max() < 2e-6
    assert _softplus_fp32(np.array([0.0]))[0] == np.float32(np.log(2.0))
