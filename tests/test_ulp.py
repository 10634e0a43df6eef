"""The ulp-distance helper on values whose distances are known by construction."""

import numpy as np

from ulp import max_ulp


def test_neighbours_zeros_and_sign_changes():
    one = np.array([1.0], np.float32)
    assert max_ulp(np.nextafter(one, np.float32(2)), one) == 1
    assert max_ulp(np.array([0.0], np.float32), np.array([-0.0], np.float32)) == 0
    tiny = np.array([1e-45], np.float32)                    # smallest positive subnormal
    assert max_ulp(tiny, -tiny) == 2
    assert max_ulp(np.array([1.5, -2.0], np.float32), np.array([1.5, -2.0], np.float32)) == 0
    # bf16 patterns: 1.0 = 0x3F80, next up 0x3F81; -1.0 = 0xBF80
    b = lambda *v: np.array(v, np.uint16)
    assert max_ulp(b(0x3F81), b(0x3F80)) == 1
    assert max_ulp(b(0x3F80), b(0xBF80)) == 2 * 0x3F80
    assert max_ulp(b(0x0000), b(0x8000)) == 0
    assert max_ulp(b(0x0001, 0x3F80), b(0x8001, 0x3F83)) == 3
    assert max_ulp(np.zeros(0, np.float32), np.zeros(0, np.float32)) == 0
