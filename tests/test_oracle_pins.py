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


# ------------------------------------------------------------------ BF16 -> NVFP4 quantizer

def _to_bf16_bits(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_quantizer_e2m1_rounding_brute_force():
    """Every E2M1 rounding decision against exact rationals: the nearest of the eight
    magnitudes, ties to the even code, saturation above 6 (one element per block, so the
    block scale is fixed by a second element of magnitude 6)."""
    from fractions import Fraction
    vals = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]
    probes = sorted({Fraction(i, 16) for i in range(0, 97)})  # 0 .. 6 in steps of 1/16: every tie
    x = np.zeros((len(probes), 16), np.float32)
    x[:, 0] = [float(p) for p in probes]
    x[:, 1] = 6.0  # amax = 6 -> scale 1 with gs = 1
    codes, scales = oracle.quantize_nvfp4(_to_bf16_bits(x), 1.0)
    assert np.all(scales == 0x38)  # E4M3 1.0
    got = codes[:, 0] & 0xF
    for p, c in zip(probes, got):
        best = min(range(8), key=lambda i: (abs(vals[i] - p), i % 2))
        assert c == best, (p, c, best)
    # the same magnitudes negated carry the sign bit, except those that round to 0
    codes_n, _ = oracle.quantize_nvfp4(_to_bf16_bits(-x), 1.0)
    for c, cn in zip(got, codes_n[:, 0] & 0xF):
        assert cn == (c | 8 if c else 0)


def test_quantizer_round_trip_of_representable_blocks():
    """Blocks built as code x E4M3 scale x gs with a +-6 in every block (so the block's amax
    fixes the same scale) quantize back to the same codes and scales."""
    rng = np.random.default_rng(21)
    rows, K = 6, 64
    for gs in (1.0, 0.25):
        sc = rng.integers(0x20, 0x60, (rows, K // 16)).astype(np.uint8)
        code = rng.integers(0, 16, (rows, K)).astype(np.uint8)
        code[code == 8] = 0                                  # -0 comes back as +0
        code[:, ::16] = np.where(rng.random((rows, K // 16)) < 0.5, 7, 15)  # a +-6 per block
        sv = np.array([oracle.e4m3(int(b)) for b in sc.ravel()]).reshape(sc.shape)
        cv = np.array([oracle.e2m1(int(c)) for c in code.ravel()]).reshape(code.shape)
        w = (cv.reshape(rows, K // 16, 16) * sv[:, :, None] * gs).reshape(rows, K).astype(np.float32)
        packed, scales = oracle.quantize_nvfp4(_to_bf16_bits(w), gs)
        assert np.array_equal(scales, sc)
        unpacked = np.empty((rows, K), np.uint8)
        unpacked[:, 0::2] = packed & 0xF
        unpacked[:, 1::2] = packed >> 4
        assert np.array_equal(unpacked, code)


def test_quantizer_special_blocks():
    """An all-zero block: scale 0 and codes 0.  A block far above the E4M3 range saturates
    its scale at 448.  Error bound: every element is within one scale step (the largest gap
    of the E2M1 grid is 2) of its dequantized value when the scale does not saturate."""
    x = np.zeros((3, 32), np.float32)
    x[1, :16] = 1e30
    x[2, 16:] = np.linspace(-3, 5, 16)
    codes, scales = oracle.quantize_nvfp4(_to_bf16_bits(x), 1.0)
    assert scales[0, 0] == 0 and not codes[0].any()
    assert scales[1, 0] == 0x7E and np.all(codes[1, :8] == 0x77)  # saturated scale and codes
    sv = oracle.e4m3(int(scales[2, 1]))
    deq = np.array([oracle.e2m1(int((codes[2, 8 + i // 2] >> (4 * (i % 2))) & 0xF)) for i in range(16)]) * sv
    xb = (_to_bf16_bits(x[2, 16:]).astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.abs(deq - xb) <= sv * 1.0 + 1e-12)


# ------------------------------------------------------------------ quantizer: E4M3 scale rounding

def _e4m3_table():
    """(values, bytes) of the finite non-negative E4M3 bytes, from the OCP definition written out
    with exact rationals (independent of the oracle's decoders)."""
    from fractions import Fraction
    out = []
    for b in range(0x7F):
        e, m = b >> 3, b & 7
        v = Fraction(m, 8) * Fraction(2) ** -6 if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        out.append((v, b))
    return out


def _rational_nearest_even(table, s):
    """Byte of the E4M3 value nearest to the rational s (s >= 0), ties to the even byte, saturating
    at 448."""
    from fractions import Fraction
    if s >= table[-1][0]:
        return table[-1][1]
    best = None
    for v, b in table:
        d = abs(v - s)
        if best is None or d < best[0] or (d == best[0] and b % 2 == 0):
            best = (d, b)
    return best[1]


def _scale_cases():
    """Block maxima (bf16) whose amax / 6 lands exactly on every midpoint between adjacent E4M3
    values that bf16 can reach, on both sides of it by one bf16 step of amax, and past 448."""
    from fractions import Fraction
    table = _e4m3_table()
    amaxes = set()
    for (a, _), (b, _) in zip(table, table[1:]):
        mid = (a + b) / 2
        am = 6 * mid
        bits = int(np.float32(float(am)).view(np.uint32)) >> 16
        for db in (-1, 0, 1):
            v = np.array([(bits + db) << 16], np.uint32).view(np.float32)[0]
            if v > 0:
                amaxes.add(float(v))
    amaxes.update([448.0 * 6, 460.0 * 6, 1.0e4, 6.0 * 2.0 ** -10])
    return sorted(amaxes)


def _check_scale_rounding(quantize):
    """quantize(w_bits, gs) -> (codes, scales); every block's scale must be the rational
    nearest-even E4M3 value of the fp32 quotient (amax / 6) / gs, saturating at 448."""
    from fractions import Fraction
    table = _e4m3_table()
    amaxes = _scale_cases()
    w = np.zeros((len(amaxes), 16), np.float32)
    w[:, 3] = amaxes                       # the block maximum
    w[:, 7] = -np.float32(0.25) * w[:, 3]  # smaller elements do not change the scale
    _, scales = quantize(_to_bf16_bits(w), 1.0)
    for i, am in enumerate(amaxes):
        s32 = np.float32(np.float32(am) / np.float32(6.0)) / np.float32(1.0)
        want = _rational_nearest_even(table, Fraction(float(s32)))
        assert int(scales[i, 0]) == want, (am, float(s32), int(scales[i, 0]), want)


def test_quantizer_scale_rounding_exact_rationals():
    """The oracle's E4M3 scale choice against exact rationals: midpoints between adjacent E4M3
    values (ties to the even byte), one bf16 step to either side, and saturation at 448."""
    _check_scale_rounding(oracle.quantize_nvfp4)


@pytest.mark.parametrize("mutant", ["ceil", "floor", "ties_away", "ties_odd"])
def test_quantizer_scale_rounding_mutants_are_caught(mutant, monkeypatch):
    """Plausible rounding mistakes planted in the oracle's nearest-value search must fail the
    exact-rational pin above."""
    real = oracle._nearest_even

    def planted(values_sorted, codes_sorted, v):
        v = np.asarray(v, np.float64)
        hi = np.clip(np.searchsorted(values_sorted, v, side="left"), 0, len(values_sorted) - 1)
        lo = np.clip(hi - 1, 0, len(values_sorted) - 1)
        exact = values_sorted[hi] == v
        dl, dh = np.abs(v - values_sorted[lo]), np.abs(values_sorted[hi] - v)
        if mutant == "ceil":
            pick_hi = np.ones_like(exact)
        elif mutant == "floor":
            pick_hi = exact
        elif mutant == "ties_away":
            pick_hi = dh <= dl
        else:  # ties to the odd code
            pick_hi = (dh < dl) | ((dh == dl) & (codes_sorted[hi] % 2 == 1))
        return np.where(pick_hi, codes_sorted[hi], codes_sorted[lo])

    # only the E4M3 search (the 127-entry table) is planted; the E2M1 one stays the real one
    def routed(values_sorted, codes_sorted, v):
        return planted(values_sorted, codes_sorted, v) if len(values_sorted) > 8 else real(values_sorted, codes_sorted, v)

    monkeypatch.setattr(oracle, "_nearest_even", routed)
    with pytest.raises(AssertionError):
        _check_scale_rounding(oracle.quantize_nvfp4)


# ------------------------------------------------------------------ gated-MLP input: one bf16 ulp

def test_silu_mul_within_one_bf16_ulp_of_fp64():
    """x = bf16(silu(g) * u) against silu(g) * u computed in binary64 from the closed form
    g / (1 + e^-g): the oracle's fp32 steps may move the bf16 result by at most one ulp, and
    only next to a rounding boundary."""
    import math
    rng = np.random.default_rng(11)
    g = (rng.standard_normal((8, 256)) * 4).astype(np.float32)
    u = (rng.standard_normal((8, 256)) * 2).astype(np.float32)
    g = ((g.view(np.uint32) >> 16) << 16).view(np.float32)
    u = ((u.view(np.uint32) >> 16) << 16).view(np.float32)
    got = oracle.silu_mul_bf16(np.concatenate([_bits(g), _bits(u)], axis=1), g.shape[1])
    gv = (got.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = np.vectorize(lambda a, b: a / (1.0 + math.exp(-a)) * b)(g.astype(np.float64), u.astype(np.float64))
    ulp = np.array([2.0 ** (math.frexp(abs(r))[1] - 8) if r != 0 else 2.0 ** -133 for r in ref.ravel()]).reshape(ref.shape)
    err = np.abs(gv - ref)
    assert np.all(err <= 1.0 * ulp), float(np.max(err / ulp))
    assert np.mean(err <= 0.5 * ulp) > 0.97   # almost every element is the correctly rounded one
