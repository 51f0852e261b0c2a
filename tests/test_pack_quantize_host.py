"""The host BF16 -> NVFP4 quantizer of the packer library ("Module ops", quantize_bf16_to_nvfp4),
bit for bit against the oracle's quantizer (whose E4M3 and E2M1 rounding is pinned in
test_oracle_pins.py), on random weights and on the blocks where the rounding rules decide:
midpoints of both formats with either sign, zero and tiny blocks, saturation, bf16 subnormals,
and strided rows; plus its refusals.  No GPU."""
import ctypes

import numpy as np
import pytest

import oracle
from nvfp4_skinny_gb300 import binding as nb
from nvfp4_skinny_gb300 import build


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build_pack()


def bits_of(a):
    """float32 values that are bfloat16-representable -> their bfloat16 bits."""
    a = np.ascontiguousarray(a, np.float32)
    assert np.all((a.view(np.uint32) & 0xFFFF) == 0), "not a bfloat16 value"
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def to_bf16(a):
    """Round float32 values to bfloat16 (nearest even), as float32."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16).astype(np.uint32)
    return r.view(np.float32)


def check_same(w_bits, gs):
    c, s = nb.nvfp4_quantize_bf16_host(w_bits, w_global_scale=gs)
    c_ref, s_ref = oracle.quantize_nvfp4(w_bits, gs)
    assert np.array_equal(s, s_ref), np.argwhere(s != s_ref)[:5]
    assert np.array_equal(c, c_ref), np.argwhere(c != c_ref)[:5]
    return c, s


@pytest.mark.parametrize("gs", [1.0, 0.37, 1.0e-3, 7.5, 2.0 ** -20])
@pytest.mark.parametrize("dist", ["normal", "heavy", "wide"])
def test_random_weights_match_oracle(gs, dist):
    rng = np.random.default_rng(hash((gs, dist)) % 2 ** 32)
    if dist == "normal":
        w = rng.standard_normal((48, 512)) * 0.05
    elif dist == "heavy":
        w = rng.standard_t(2, (48, 512))
    else:  # magnitudes spread over 2^-40 .. 2^40
        w = rng.standard_normal((48, 512)) * np.exp2(rng.uniform(-40, 40, (48, 512)))
    check_same(bits_of(to_bf16(w)), gs)


def test_rounding_midpoints_both_signs():
    """Blocks whose amax is 6 (scale exactly 1 with gs = 1), so every element is its own E2M1
    quotient: the midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5 and values just beside them,
    with both signs; ties go to the even code (0.25 -> 0, 0.75 -> 1.0, 5 -> 4 ...)."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    vals = []
    for m in mids:  # the midpoint, its negative, and the bfloat16 neighbours on either side
        b = int(bits_of(np.array([m], np.float32))[0])
        up, down = (np.array([b + 1, b - 1], np.uint32) << 16).view(np.float32)
        vals += [m, -m, float(up), -float(down)]
    vals = np.array(vals, np.float32)
    assert np.array_equal(to_bf16(vals), vals)
    blocks = []
    for i in range(0, len(vals), 15):
        b = np.zeros(16, np.float32)
        chunk = vals[i:i + 15]
        b[:len(chunk)] = chunk
        b[15] = 6.0
        blocks.append(b)
    w = np.stack(blocks).reshape(1, -1)
    c, s = check_same(bits_of(w), 1.0)
    assert np.all(s == 0x38)  # E4M3 1.0
    codes = nb.nvfp4_unpack_codes(c, w.shape[1])[0]
    want = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for j, v in enumerate(w[0]):
        if float(abs(v)) in want and v != 0:
            mag = want[float(abs(v))]
            assert codes[j] == mag | (8 if v < 0 and mag else 0), (v, codes[j])  # magnitude 0 is +0


def test_zero_tiny_saturated_and_subnormal_blocks():
    rows = []
    rows.append(np.zeros(64, np.float32))                                   # zero blocks: scale 0, codes 0
    r = np.zeros(64, np.float32); r[3] = -0.0; r[20] = 2.0 ** -133; rows.append(r)  # -0 and a bf16 subnormal
    rows.append(np.full(64, 3.0e38, np.float32) * np.tile([1, -1], 32))       # saturates at 448 and 6
    rows.append(np.float32(2.0 ** -12) * np.arange(1, 65, dtype=np.float32))  # E4M3 subnormal scales
    rows.append(np.full(64, np.inf, np.float32) * np.tile([1, -1, 1, 1], 16))  # infinities saturate
    w = np.stack([to_bf16(r) for r in rows])
    c, s = check_same(bits_of(w), 1.0)
    assert np.all(s[0] == 0) and np.all(c[0] == 0)
    assert np.all(s[2] == 0x7E) and np.all(s[4] == 0x7E)


def test_strided_rows():
    rng = np.random.default_rng(5)
    w = bits_of(to_bf16(rng.standard_normal((9, 384))))
    c, s = nb.nvfp4_quantize_bf16_host(w, K=256, w_global_scale=0.5)
    c_ref, s_ref = oracle.quantize_nvfp4(np.ascontiguousarray(w[:, :256]), 0.5)
    assert np.array_equal(c, c_ref) and np.array_equal(s, s_ref)


def test_refusals():
    lib = nb.pack_lib()
    w = np.zeros((4, 32), np.uint16)
    c = np.zeros((4, 16), np.uint8)
    s = np.zeros((4, 2), np.uint8)
    q = lambda wp, rows, K, ldw, gs, cp, sp: lib.nvfp4_quantize_bf16_host(wp, rows, K, ldw, gs, cp, sp)
    W, C, S = w.ctypes.data, c.ctypes.data, s.ctypes.data
    assert q(W, 4, 32, 32, 1.0, C, S) == nb.NVFP4_PACK_OK
    assert q(None, 4, 32, 32, 1.0, C, S) == nb.NVFP4_PACK_ERR_ARG
    assert q(W, 4, 32, 32, 1.0, None, S) == nb.NVFP4_PACK_ERR_ARG
    assert q(W, 0, 32, 32, 1.0, C, S) == nb.NVFP4_PACK_ERR_ARG
    assert q(W, 4, 24, 32, 1.0, C, S) == nb.NVFP4_PACK_ERR_ARG     # K not a multiple of 16
    assert q(W, 4, 32, 16, 1.0, C, S) == nb.NVFP4_PACK_ERR_ARG     # ldw < K
    for gs in (0.0, -1.0, float("inf"), float("nan")):
        c[:] = 0xAB
        assert q(W, 4, 32, 32, gs, C, S) == nb.NVFP4_PACK_ERR_VALUE
        assert np.all(c == 0xAB), "a refused call wrote its output"
