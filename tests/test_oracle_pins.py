"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""
import numpy as np
import pytest

import oracle
import oracle_checks as oc


@pytest.mark.parametrize("check", oc.ALL_CHECKS, ids=lambda f: f.__name__)
def test_oracle_pin(check):
    check(oracle.default())


# ------------------------------------------------------------------ gated-MLP input (silu(gate) * up)

def _bits(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_silu_mul_special_values():
    """silu(0) = 0; silu(g) -> g for large g and -> 0 for very negative g; up = 1 gives silu(g)
    itself, up = 0 gives 0."""
    g = np.array([[0.0, 20.0, -60.0, 1.0, 2.0, -1.0]], np.float32)
    one = np.ones_like(g)
    x = oracle.silu_mul_bf16(np.concatenate([_bits(g), _bits(one)], axis=1), g.shape[1])
    v = (x.astype(np.uint32) << 16).view(np.float32)[0]
    assert v[0] == 0.0
    assert v[1] == 20.0                       # 20 / (1 + e^-20) rounds to 20 in bfloat16
    assert v[2] == 0.0 or abs(v[2]) < 1e-20   # -60 e^-60: vanishingly small
    # closed forms: silu(1) = 1 / (1 + e^-1) = 0.7310586, silu(2) = 1.7615942, silu(-1) = -0.2689414
    for got, want in zip(v[3:], (0.7310586, 1.7615942, -0.2689414)):
        assert abs(got - want) <= 2.0 ** -8 * abs(want)
    zero = np.zeros_like(g)
    x0 = oracle.silu_mul_bf16(np.concatenate([_bits(g), _bits(zero)], axis=1), g.shape[1])
    assert not x0.any() or np.all((x0 & 0x7FFF) == 0)


def test_silu_mul_odd_part_identity():
    """silu(g) - silu(-g) = g for every g (sigma(g) + sigma(-g) = 1), and the rounding to
    bfloat16 moves each side by at most half an ulp of its value."""
    rng = np.random.default_rng(5)
    g = rng.standard_normal((4, 64)).astype(np.float32) * 3
    g = ((g.view(np.uint32) >> 16) << 16).view(np.float32)   # exact bfloat16 inputs
    one = np.ones_like(g)
    pos = oracle.silu_mul_bf16(np.concatenate([_bits(g), _bits(one)], axis=1), g.shape[1])
    neg = oracle.silu_mul_bf16(np.concatenate([_bits(-g), _bits(one)], axis=1), g.shape[1])
    fp = (pos.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    fn = (neg.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    err = np.abs((fp - fn) - g.astype(np.float64))
    assert np.all(err <= 2.0 ** -8 * (np.abs(fp) + np.abs(fn)) + 1e-30)
