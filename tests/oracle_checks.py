"""Pins for the CPU oracle, written against an oracle object so the same checks
can be run on deliberately broken copies of it (see test_oracle_mutants.py).

Every expected value here comes from outside the oracle:
  * the cited fixtures in tests/golden/ (OCP E2M1 table, E4M3 specials,
    E4M3_MAX = 448 from "Module ops");
  * library decoders (torch's float8_e4m3fn and bfloat16 casts);
  * exact rational arithmetic (fractions.Fraction) on tiny cases;
  * closed forms and invariants (one-hot inputs, power-of-two scaling, zero
    codes, integer inputs, numpy's float64 matmul on a dequantised matrix).
"""
import math
from fractions import Fraction

import numpy as np
import torch

from golden_tables import e2m1_table, e4m3_specials


def torch_e4m3(byte_array):
    """Library decode of E4M3 bytes -> float64 (torch float8_e4m3fn)."""
    b = torch.as_tensor(np.asarray(byte_array, np.uint8))
    return b.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_bf16(bits_array):
    """Library decode of bfloat16 bit patterns -> float64."""
    b = torch.as_tensor(np.asarray(bits_array, np.uint16).astype(np.int16))
    return b.view(torch.bfloat16).to(torch.float64).numpy()


def bf16_bits(values):
    """Round float values to bfloat16 (torch, RNE) and return the bit patterns."""
    t = torch.as_tensor(np.asarray(values, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().astype(np.uint16)


def test_side_dequant(codes, scales, gs):
    """Dequantise with the test's own decoders: golden E2M1 table, torch E4M3,
    low nibble = even k ("Module ops", nvfp4_mmq_repack)."""
    tab = np.array([e2m1_table()[c] for c in range(16)], np.float64)
    lo = codes & 0x0F
    hi = codes >> 4
    N, Kh = codes.shape
    q = np.empty((N, 2 * Kh), np.uint8)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    s = torch_e4m3(scales.reshape(-1)).reshape(scales.shape)
    return tab[q] * np.repeat(s, 16, axis=1) * float(np.float32(gs))


def random_case(rng, M, N, K, scale_lo=0x28, scale_hi=0x48):
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = rng.integers(scale_lo, scale_hi, size=(N, K // 16), dtype=np.uint8)
    x = bf16_bits(rng.standard_normal((M, K)))
    return x, codes, scales


# ----------------------------------------------------------------------------- formats

def check_e2m1_table(orc):
    for c, v in e2m1_table().items():
        got = orc.e2m1(c)
        assert got == v and math.copysign(1.0, got) == math.copysign(1.0, v), (c, got, v)


def check_e2m1_negation(orc):
    for c in range(8):
        assert orc.e2m1(c | 8) == -orc.e2m1(c)
    assert [orc.e2m1(c) for c in range(8)] == sorted(orc.e2m1(c) for c in range(8))


def check_e4m3_vs_library(orc):
    ref = torch_e4m3(np.arange(256))
    got = np.array([orc.e4m3(b) for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def check_e4m3_specials(orc):
    for b, v in e4m3_specials().items():
        got = orc.e4m3(b)
        if math.isnan(v):
            assert math.isnan(got), b
        else:
            assert got == v and math.copysign(1.0, got) == math.copysign(1.0, v), (hex(b), got, v)
    finite = [abs(orc.e4m3(b)) for b in range(256) if not math.isnan(orc.e4m3(b))]
    assert max(finite) == 448.0  # E4M3_MAX ("Module ops", Constants)


def check_bf16_vs_library(orc):
    bits = np.arange(65536)
    ref = torch_bf16(bits)
    got = np.array([orc.bf16(int(b)) for b in bits])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def check_product_table_exact(orc):
    """"10 Kernels" 10.2: e2m1 x e4m3 needs six significant bits, so every product
    is exact in fp16 (11 bits) -- and in bf16 (8 bits)."""
    n_finite = 0
    for c in range(16):
        for b in range(256):
            p = orc.e2m1(c) * orc.e4m3(b)
            if math.isnan(p):
                assert b in (0x7F, 0xFF)
                continue
            n_finite += 1
            assert float(np.float16(p)) == p, (c, b, p)
            assert float(torch.tensor(p, dtype=torch.float64).to(torch.bfloat16).double()) == p, (c, b, p)
            if p != 0.0:
                m, _ = math.frexp(abs(p))
                assert Fraction(m).denominator <= 64  # at most six significant bits
    assert n_finite == 16 * 254


# ----------------------------------------------------------------------------- layout

def check_layout_nibbles_and_blocks(orc):
    """Low nibble = even k; scale index = k // 16; row stride K/2 and K/16."""
    N, K = 3, 64
    codes = np.zeros((N, K // 2), np.uint8)
    scales = np.full((N, K // 16), 0x38, np.uint8)  # 1.0
    codes[1, 0] = 0x21   # k=0 -> code 1 (0.5), k=1 -> code 2 (1.0)
    codes[1, 8] = 0x7F   # k=16 -> code 15 (-6), k=17 -> code 7 (6)
    scales[1, 1] = 0x40  # block 1 (k = 16..31) -> 2.0
    scales[2, 3] = 0x30  # row 2, block 3 -> 0.5
    codes[2, 31] = 0x50  # k=62 -> 0, k=63 -> code 5 (3.0)
    gs = 0.25
    w = lambda n, k: orc.weight(codes, scales, gs, K, n, k)
    assert w(1, 0) == 0.5 * 0.25 and w(1, 1) == 1.0 * 0.25
    assert w(1, 16) == -6.0 * 2.0 * 0.25 and w(1, 17) == 6.0 * 2.0 * 0.25
    assert w(1, 15) == 0.0 and w(0, 0) == 0.0
    assert w(2, 62) == 0.0 and w(2, 63) == 3.0 * 0.5 * 0.25
    # one-hot rows of x pick these columns out through linear()
    x = np.zeros((4, K), np.float32)
    x[0, 0] = 1.0
    x[1, 1] = 1.0
    x[2, 17] = 1.0
    x[3, 63] = 1.0
    y, _ = orc.linear(bf16_bits(x), codes, scales, gs)
    assert y.shape == (4, N)
    assert y[0, 1] == 0.125 and y[1, 1] == 0.25 and y[2, 1] == 3.0 and y[3, 2] == 0.375
    assert y[0, 0] == 0.0 and y[3, 1] == 0.0 and y[2, 2] == 0.0


# ----------------------------------------------------------------------------- dot products

def check_brute_force_exact(orc, seed=11):
    """fp64 oracle vs exact rationals on tiny shapes (M, N <= 4, K in {16, 32, 64})."""
    rng = np.random.default_rng(seed)
    tab = e2m1_table()
    for M, N, K in ((1, 1, 16), (2, 3, 32), (4, 4, 64), (3, 2, 64)):
        x, codes, scales = random_case(rng, M, N, K, 0x01, 0x7F)
        gs = float(np.float32(rng.uniform(0.001, 3.0)))
        xs = torch_bf16(x.reshape(-1)).reshape(M, K)
        ss = torch_e4m3(scales.reshape(-1)).reshape(N, K // 16)
        y, a = orc.linear(x, codes, scales, gs)
        for m in range(M):
            for n in range(N):
                exact = Fraction(0)
                aexact = Fraction(0)
                for k in range(K):
                    byte = int(codes[n, k // 2])
                    c = (byte >> 4) if (k & 1) else (byte & 15)
                    t = Fraction(tab[c]) * Fraction(float(ss[n, k // 16])) * Fraction(gs) * Fraction(float(xs[m, k]))
                    exact += t
                    aexact += abs(t)
                bound = K * 2.0 ** -52 * float(aexact)
                assert abs(Fraction(y[m, n]) - exact) <= Fraction(bound), (M, N, K, m, n)
                assert abs(Fraction(a[m, n]) - aexact) <= Fraction(bound), (M, N, K, m, n)


def check_one_hot_columns(orc, seed=12):
    """x = e_k gives y[:, n] = W[n, k] exactly."""
    rng = np.random.default_rng(seed)
    N, K = 5, 96
    _, codes, scales = random_case(rng, 1, N, K)
    gs = 0.375
    W = test_side_dequant(codes, scales, gs)
    ks = [0, 1, 15, 16, 17, 50, 95]
    x = np.zeros((len(ks), K), np.float32)
    for i, k in enumerate(ks):
        x[i, k] = 1.0
    y, a = orc.linear(bf16_bits(x), codes, scales, gs)
    for i, k in enumerate(ks):
        assert np.array_equal(y[i], W[:, k]), k
        assert np.array_equal(a[i], np.abs(W[:, k])), k


def check_integer_exact(orc, seed=13):
    """Scales 1.0, gs = 1, integer x: y is an exact multiple of 1/2 computed in int64."""
    rng = np.random.default_rng(seed)
    M, N, K = 3, 6, 128
    codes = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    scales = np.full((N, K // 16), 0x38, np.uint8)
    xi = rng.integers(-100, 101, size=(M, K))
    twice = {c: int(2 * v) for c, v in e2m1_table().items()}
    q = np.empty((N, K), np.int64)
    q[:, 0::2] = np.vectorize(twice.get)(codes & 15)
    q[:, 1::2] = np.vectorize(twice.get)(codes >> 4)
    exact2 = xi @ q.T  # = 2 * y
    y, _ = orc.linear(bf16_bits(xi), codes, scales, 1.0)
    assert np.array_equal(y * 2, exact2.astype(np.float64))


def check_pow2_global_scale(orc, seed=14):
    rng = np.random.default_rng(seed)
    x, codes, scales = random_case(rng, 2, 7, 64)
    y1, a1 = orc.linear(x, codes, scales, 1.0)
    y8, a8 = orc.linear(x, codes, scales, 0.125)
    assert np.array_equal(y8, y1 * 0.125) and np.array_equal(a8, a1 * 0.125)
    y0, _ = orc.linear(x, codes, scales, 0.0)
    assert np.all(y0 == 0.0)


def check_zero_codes(orc, seed=15):
    rng = np.random.default_rng(seed)
    x, _, scales = random_case(rng, 3, 4, 64)
    for byte in (0x00, 0x88, 0x08, 0x80):
        codes = np.full((4, 32), byte, np.uint8)
        y, a = orc.linear(x, codes, scales, 1.0)
        assert np.all(y == 0.0) and np.all(a == 0.0)


def check_library_matmul(orc, seed=16):
    """Same product as numpy's float64 matmul of the test-side dequantised matrix."""
    rng = np.random.default_rng(seed)
    M, N, K = 5, 33, 256
    x, codes, scales = random_case(rng, M, N, K, 0x20, 0x50)
    gs = 0.01
    W = test_side_dequant(codes, scales, gs)
    X = torch_bf16(x.reshape(-1)).reshape(M, K)
    ref = X @ W.T
    y, a = orc.linear(x, codes, scales, gs)
    aref = np.abs(X) @ np.abs(W).T
    bound = K * 2.0 ** -52 * aref * 2
    assert np.all(np.abs(y - ref) <= bound)
    assert np.all(np.abs(a - aref) <= bound)


def check_sampled_matches_full(orc, seed=17):
    rng = np.random.default_rng(seed)
    M, N, K = 4, 20, 128
    x, codes, scales = random_case(rng, M, N, K)
    y, a = orc.linear(x, codes, scales, 0.5)
    ms = rng.integers(0, M, 30)
    ns = rng.integers(0, N, 30)
    ys, as_ = orc.linear_at(x, codes, scales, 0.5, ms, ns)
    assert np.array_equal(ys, y[ms, ns]) and np.array_equal(as_, a[ms, ns])


def check_bf16_ulp(orc):
    """ulp from consecutive bfloat16 values (torch decode of adjacent bit patterns)."""
    for v in (1.0, 1.5, 1.9921875, 2.0, 0.75, 3.0e-3, 1234.0, 6.0e30):
        b = int(bf16_bits([v])[0])
        lo, hi = torch_bf16([b, b + 1])
        assert orc.bf16_ulp(v) == hi - lo, v
        assert orc.bf16_ulp(-v) == hi - lo, v
    assert orc.bf16_ulp(0.0) == 2.0 ** -133


ALL_CHECKS = [
    check_e2m1_table, check_e2m1_negation, check_e4m3_vs_library, check_e4m3_specials,
    check_bf16_vs_library, check_product_table_exact, check_layout_nibbles_and_blocks,
    check_brute_force_exact, check_one_hot_columns, check_integer_exact, check_pow2_global_scale,
    check_zero_codes, check_library_matmul, check_sampled_matches_full, check_bf16_ulp,
]
