"""Pins for the oracle's online INT8 row quantizer ("[Feature] TurboMind support
W8A8 or FP8 KV Cache", lmdeploy issue 1463: online KV-cache INT8; symmetric reading
with one fp32 scale amax / 127 per (token, kv-head) row)."""
import numpy as np

import oracle
from tests.conftest import golden


def test_hand_row():
    rows = golden("int8_row.txt")
    x = np.array([float(r[0]) for r in rows], np.float32)
    q, s = oracle.int8_quant_row(x)
    assert s == np.float32(0.125)
    assert list(q) == [int(r[1]) for r in rows]


def test_zero_row():
    q, s = oracle.int8_quant_row(np.zeros(128, np.float32))
    assert s == 0 and not q.any()


def test_properties_random_rows():
    rng = np.random.default_rng(7)
    for i in range(2000):
        d = 128 if i % 2 else 64
        x = (rng.standard_normal(d) * rng.choice([1e-4, 1.0, 20.0, 3000.0])).astype(np.float16)
        x32 = x.astype(np.float32)
        q, s = oracle.int8_quant_row(x32)
        amax = np.abs(x32).max()
        # the scale maps the row maximum onto +-127 and nothing leaves [-127, 127]
        assert s > 0 and abs(float(s) * 127.0 - float(amax)) <= float(amax) * 2.0 ** -23
        assert q.min() >= -127 and q.max() <= 127
        j = int(np.argmax(np.abs(x32)))
        assert q[j] == (127 if x32[j] > 0 else -127)
        # nearest integer: |q - x/s| <= 1/2 (+ one fp32 rounding of x/s)
        r = x32.astype(np.float64) / float(s)
        assert np.all(np.abs(q - r) <= 0.5 + 1e-5 * np.maximum(1.0, np.abs(r)))
        # sign preserved, zeros stay zero
        assert np.all(np.sign(q[np.abs(r) > 0.5 + 1e-4]) == np.sign(x32[np.abs(r) > 0.5 + 1e-4]))
