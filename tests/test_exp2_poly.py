"""The FMA-pipe exp2 of the forward softmax, evaluated step for step in fp32
(numpy) as the device code does, against numpy's exp2 in float64: its
relative error must stay below the fp16 rounding of P (2^-11)."""
import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "attention_learnable_head_gb300", "csrc", "sm103_ptx.cuh")


def _coeffs():
    text = open(HDR).read()
    m = re.search(r"kExp2C0 = ([\d.e-]+)f, kExp2C1 = ([\d.e-]+)f, kExp2C2 = ([\d.e-]+)f,\s*"
                  r"kExp2C3 = ([\d.e-]+)f", text)
    return [np.float32(float(g)) for g in m.groups()]


def _exp2_poly(x):
    c0, c1, c2, c3 = _coeffs()
    x0 = x.astype(np.float32)
    x = np.maximum(x0, np.float32(-125.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    n = (t - magic).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = np.float32(c3) * f + c2
    p = (p.astype(np.float32) * f + c1).astype(np.float32)
    p = (p * f + c0).astype(np.float32)
    bits = p.view(np.int32) + (t.view(np.int32) << 23)
    return np.where(x0 < -125.0, np.float32(0.0), bits.astype(np.int32).view(np.float32))


def test_relative_error_bound():
    x = np.linspace(-40.0, 8.0, 400001, dtype=np.float32)
    got = _exp2_poly(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    rel = np.abs(got / ref - 1.0)
    assert rel.max() < 1e-4, rel.max()


def test_integers_and_clamp():
    x = np.arange(-120, 9, dtype=np.float32)
    got = _exp2_poly(x).astype(np.float64)
    assert np.allclose(got, np.exp2(x.astype(np.float64)), rtol=1e-4, atol=0)
    assert _exp2_poly(np.array([-1e9, -np.inf], dtype=np.float32)).tolist() == [0.0, 0.0]
