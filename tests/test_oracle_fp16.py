"""The oracle's FP16 rounding (numpy float64 -> float16) against hand-derived bit patterns."""
import numpy as np

from oracle import lbq_oracle as O


def test_fp16_round_patterns():
    cases = {
        1.0: 0x3C00,
        1.0 + 2.0 ** -11: 0x3C00,              # tie -> even
        1.0 + 3 * 2.0 ** -11: 0x3C02,          # tie -> even (up)
        1.0 + 2.0 ** -11 + 2.0 ** -40: 0x3C01, # just above the tie
        65504.0: 0x7BFF,
        65519.99: 0x7BFF,
        65520.0: 0x7C00,                       # rounds to infinity
        2.0 ** -24: 0x0001,
        2.0 ** -25: 0x0000,                    # tie between 0 and min subnormal -> 0
        3 * 2.0 ** -25: 0x0002,                # tie -> even subnormal
        1e-8: 0x0000,
        -0.449951171875: 0xB733,
        1.52: 0x3E14,
        0.45: 0x3733,
    }
    for v, bits in cases.items():
        assert int(O.fp16_round(v).view("<u2")) == bits, v
