"""CPU oracle for y = x . dequant(W)^T with an NVFP4 weight (binary64).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA path (``nvfp4_skinny_gb300``) and neither imports the other.

The arithmetic lives in ``nvfp4_oracle.c`` (plain C, binary64, ascending-k
sums, formats decoded from their bit fields).  This module only marshals
numpy arrays into it.

Sources: "10 Kernels" section 10.2 (E2M1 weight, E4M3 group scale per 16
along K, 16-bit activations); "Module ops", Functions dequant_nvfp4_to_bf16,
nvfp4_mmq_repack (E2M1 [n, k/2] with the low nibble = even k, E4M3
[n, k/16]), w4a16_gemm (FP32 per-tensor scale, BF16 A [M, K]) and
w4a16_tc_rows (output [m, n] = input [m, :] . W[n, :]^T).

Tolerance: |y - y_ref| <= 4e-3 * sum_k |w_k x_k| + one bfloat16 ulp of
|y_ref| per element (the stated acceptance bound for the GPU path).
"""
import ctypes
import numpy as np

from . import build as _build

class Oracle:
    """Marshalling wrapper around one build of the oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        d, i64, p = ctypes.c_double, ctypes.c_int64, ctypes.c_void_p
        lib.nvfp4_oracle_e2m1.restype = d
        lib.nvfp4_oracle_e2m1.argtypes = [ctypes.c_uint]
        lib.nvfp4_oracle_e4m3.restype = d
        lib.nvfp4_oracle_e4m3.argtypes = [ctypes.c_uint]
        lib.nvfp4_oracle_bf16.restype = d
        lib.nvfp4_oracle_bf16.argtypes = [ctypes.c_uint]
        lib.nvfp4_oracle_weight.restype = d
        lib.nvfp4_oracle_weight.argtypes = [p, p, ctypes.c_float, i64, i64, i64]
        lib.nvfp4_oracle_linear.restype = None
        lib.nvfp4_oracle_linear.argtypes = [i64, i64, i64, p, p, p, ctypes.c_float, p, p, ctypes.c_int]
        lib.nvfp4_oracle_linear_at.restype = None
        lib.nvfp4_oracle_linear_at.argtypes = [i64, i64, p, p, p, p, p, ctypes.c_float, p, p, ctypes.c_int]
        lib.nvfp4_oracle_bf16_ulp.restype = d
        lib.nvfp4_oracle_bf16_ulp.argtypes = [d]
        lib.nvfp4_oracle_max_threads.restype = ctypes.c_int
        lib.nvfp4_oracle_max_threads.argtypes = []
        self.lib = lib
        self.path = path

    def e2m1(self, code: int) -> float:
        """E2M1 value of a 4-bit code (OCP MX FP4)."""
        return self.lib.nvfp4_oracle_e2m1(int(code))

    def e4m3(self, byte: int) -> float:
        """E4M3 value of one byte (OCP FP8 E4M3FN; 0x7F/0xFF are NaN)."""
        return self.lib.nvfp4_oracle_e4m3(int(byte))

    def bf16(self, bits: int) -> float:
        """Value of a bfloat16 bit pattern."""
        return self.lib.nvfp4_oracle_bf16(int(bits))

    def weight(self, codes, scales, gs: float, K: int, n: int, k: int) -> float:
        """Dequantised W[n, k] = E2M1(code) * E4M3(scale[n, k // 16]) * gs."""
        codes, scales = _u8(codes), _u8(scales)
        return self.lib.nvfp4_oracle_weight(_ptr(codes), _ptr(scales), float(np.float32(gs)), int(K), int(n), int(k))

    def linear(self, x_bits, codes, scales, gs: float, threads: int = 0):
        """Full product.  x_bits: uint16 [M, K] (bfloat16 bits); codes: uint8 [N, K/2];
        scales: uint8 [N, K/16]; gs: float32 per-tensor scale.

        Returns (y_ref, absdot), both float64 [M, N]."""
        x_bits, codes, scales = _u16(x_bits), _u8(codes), _u8(scales)
        M, K = x_bits.shape
        N = codes.shape[0]
        assert codes.shape == (N, K // 2) and scales.shape == (N, K // 16) and K % 16 == 0
        y = np.empty((M, N), np.float64)
        a = np.empty((M, N), np.float64)
        self.lib.nvfp4_oracle_linear(M, N, K, _ptr(x_bits), _ptr(codes), _ptr(scales), float(np.float32(gs)),
                                     _ptr(y), _ptr(a), int(threads))
        return y, a

    def linear_at(self, x_bits, codes, scales, gs: float, ms, ns, threads: int = 0):
        """Sampled outputs (ms[i], ns[i]); returns (y_ref, absdot), float64 [count]."""
        x_bits, codes, scales = _u16(x_bits), _u8(codes), _u8(scales)
        M, K = x_bits.shape
        N = codes.shape[0]
        assert codes.shape == (N, K // 2) and scales.shape == (N, K // 16) and K % 16 == 0
        ms = np.ascontiguousarray(ms, dtype=np.int64)
        ns = np.ascontiguousarray(ns, dtype=np.int64)
        assert ms.shape == ns.shape and ms.ndim == 1
        assert (ms >= 0).all() and (ms < M).all() and (ns >= 0).all() and (ns < N).all()
        y = np.empty(ms.shape, np.float64)
        a = np.empty(ms.shape, np.float64)
        self.lib.nvfp4_oracle_linear_at(K, ms.size, _ptr(ms), _ptr(ns), _ptr(x_bits), _ptr(codes), _ptr(scales),
                                        float(np.float32(gs)), _ptr(y), _ptr(a), int(threads))
        return y, a

    def bf16_ulp(self, a) -> np.ndarray:
        """One bfloat16 ulp at magnitude |a| (elementwise)."""
        f = np.vectorize(self.lib.nvfp4_oracle_bf16_ulp, otypes=[np.float64])
        return f(np.asarray(a, np.float64))

    def tolerance(self, y_ref, absdot) -> np.ndarray:
        """Per-element acceptance bound 4e-3 * sum|w x| + ulp_bf16(|y_ref|)."""
        return 4e-3 * np.asarray(absdot, np.float64) + self.bf16_ulp(y_ref)

    def max_threads(self) -> int:
        """Threads the oracle's OpenMP runtime uses by default."""
        return int(self.lib.nvfp4_oracle_max_threads())


def _u8(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint8
    return a


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "x must be given as bfloat16 bit patterns (uint16)"
    return a


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


_default = None


def default() -> Oracle:
    """The oracle built from oracle/nvfp4_oracle.c (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default


def e2m1(code):
    return default().e2m1(code)


def e4m3(byte):
    return default().e4m3(byte)


def bf16(bits):
    return default().bf16(bits)


def weight(codes, scales, gs, K, n, k):
    return default().weight(codes, scales, gs, K, n, k)


def linear(x_bits, codes, scales, gs, threads: int = 0):
    return default().linear(x_bits, codes, scales, gs, threads)


def linear_at(x_bits, codes, scales, gs, ms, ns, threads: int = 0):
    return default().linear_at(x_bits, codes, scales, gs, ms, ns, threads)


def bf16_ulp(a):
    return default().bf16_ulp(a)


def tolerance(y_ref, absdot):
    return default().tolerance(y_ref, absdot)


def max_threads():
    return default().max_threads()


def silu_mul_bf16(gate_up_bits, K: int) -> np.ndarray:
    """Input of the gated-MLP down projection: x[m, k] = bf16(silu(g) * u) with g = row[k] and
    u = row[K + k] of a [gate | up] bfloat16 row ("Module ops", the SiLU-times-up input of the
    fused MLP launchers).  silu(g) = g / (1 + e^-g).

    The bfloat16 rounding of x is a decision taken in the GPU path's precision (fp32 operations,
    each rounded to nearest), so it is taken here in fp32 too; only the exponential may differ
    from the GPU's by an ulp, which can move x by at most one bfloat16 ulp.

    gate_up_bits: uint16 [M, >= 2K] (bfloat16 bits).  Returns uint16 [M, K] (bfloat16 bits)."""
    gu = np.ascontiguousarray(gate_up_bits, dtype=np.uint16)
    g = (gu[:, :K].astype(np.uint32) << 16).view(np.float32)
    u = (gu[:, K:2 * K].astype(np.uint32) << 16).view(np.float32)
    with np.errstate(over="ignore"):
        den = np.float32(1.0) + np.exp(-g, dtype=np.float32)
    x = (g / den).astype(np.float32) * u
    bits = x.astype(np.float32).view(np.uint32)
    rounded = (bits + np.uint32(0x7FFF) + ((bits >> 16) & np.uint32(1))) >> 16   # nearest-even (finite x)
    return rounded.astype(np.uint16)


def _nearest_even(values_sorted, codes_sorted, v):
    """Index into codes_sorted of the value nearest to each v (v within [min, max] of the table);
    ties go to the even code.  Distances are compared in binary64, exact for these operands."""
    v = np.asarray(v, np.float64)
    hi = np.clip(np.searchsorted(values_sorted, v, side="left"), 0, len(values_sorted) - 1)
    lo = np.clip(hi - 1, 0, len(values_sorted) - 1)
    dl = np.abs(v - values_sorted[lo])
    dh = np.abs(values_sorted[hi] - v)
    pick_hi = (dh < dl) | ((dh == dl) & (codes_sorted[hi] % 2 == 0) & (codes_sorted[lo] % 2 == 1))
    return np.where(pick_hi, codes_sorted[hi], codes_sorted[lo])


def quantize_nvfp4(w_bits, gs: float):
    """BF16 weight -> NVFP4 ("Module ops", quantize_bf16_to_nvfp4), the plainest reading of the
    unprinted rules: per 16-element block, scale = E4M3(amax / 6 / gs) and code = E2M1(x /
    (scale * gs)), each the nearest representable value with ties to the even code, saturating
    at 448 and 6; a zero scale gives codes 0; a code whose magnitude is 0 is +0.  The divisions
    and the product are fp32 operations rounded to nearest, the precision in which the GPU path
    takes the same rounding decisions; the nearest-value searches run over the formats' value
    tables, decoded by this oracle.

    w_bits: uint16 [rows, K] (bfloat16 bits), K a multiple of 16.  Returns (codes uint8
    [rows, K/2] with the low nibble the even k, scales uint8 [rows, K/16])."""
    w_bits = np.ascontiguousarray(w_bits, dtype=np.uint16)
    rows, K = w_bits.shape
    assert K % 16 == 0
    x = (w_bits.astype(np.uint32) << 16).view(np.float32).reshape(rows, K // 16, 16)
    gs32 = np.float32(gs)
    amax = np.abs(x).max(axis=2)
    s = (amax / np.float32(6.0)).astype(np.float32) / gs32
    # E4M3 table of the finite non-negative bytes 0x00..0x7E, in increasing order
    e4_codes = np.arange(0x7F)
    e4_vals = np.array([e4m3(int(c)) for c in e4_codes], np.float64)
    s64 = np.minimum(s.astype(np.float64), 448.0)
    sc = _nearest_even(e4_vals, e4_codes, s64).astype(np.uint8)
    d = (e4_vals[sc].astype(np.float32) * gs32).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (x / d[:, :, None]).astype(np.float32)
    e2_codes = np.arange(8)
    e2_vals = np.array([e2m1(int(c)) for c in e2_codes], np.float64)
    mag = _nearest_even(e2_vals, e2_codes, np.minimum(np.abs(q.astype(np.float64)), 6.0))
    code = np.where((mag != 0) & (q < 0), mag | 8, mag)
    code = np.where(d[:, :, None] > 0, code, 0).astype(np.uint8).reshape(rows, K)
    packed = (code[:, 0::2] | (code[:, 1::2] << 4)).astype(np.uint8)
    return packed, sc


__all__ = ["Oracle", "default", "e2m1", "e4m3", "bf16", "weight", "linear", "linear_at", "bf16_ulp", "tolerance",
           "max_threads", "silu_mul_bf16", "quantize_nvfp4"]
