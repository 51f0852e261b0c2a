"""Host-side checks that need no GPU: the C-ABI libraries load and export every
symbol include/*.h declares, argument and shape refusals that happen before any
CUDA call, and the work split the kernels use."""
import ctypes
import os
import re

import numpy as np
import pytest

from nvfp4_skinny_gb300 import binding as nb
from nvfp4_skinny_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _declared_functions(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.mark.parametrize("header,getter,listed", [
    ("nvfp4_skinny.h", nb.cuda_lib, nb.CUDA_SYMBOLS),
    ("nvfp4_pack.h", nb.pack_lib, nb.PACK_SYMBOLS),
    ("nvfp4_prefill.h", nb.cuda_lib, nb.PREFILL_SYMBOLS),
])
def test_every_declared_symbol_is_exported(header, getter, listed):
    names = _declared_functions(header)
    assert names, header
    lib = getter()
    for n in names:
        assert hasattr(lib, n), "%s declares %s but the library does not export it" % (header, n)
    assert sorted(listed) == names


def test_status_strings_and_version():
    assert nb.nvfp4_abi_version() == nb.NVFP4_ABI_VERSION == 4
    for s in range(9):
        assert nb.nvfp4_status_string(s).startswith("NVFP4_")


@pytest.mark.parametrize("N,K", [(0, 512), (-1, 512), (256, 0), (256, 128), (256, 300), (256, 512 + 64)])
def test_plan_shape_refused_without_gpu(N, K):
    h = ctypes.c_void_p(123)
    st = nb.cuda_lib().nvfp4_plan_create_ex(N, K, 0, ctypes.byref(h))
    assert st == nb.NVFP4_ERR_SHAPE and h.value is None


def test_plan_bad_enum_and_null_out():
    h = ctypes.c_void_p()
    assert nb.cuda_lib().nvfp4_plan_create_ex(256, 512, 7, ctypes.byref(h)) == nb.NVFP4_ERR_ARG
    assert nb.cuda_lib().nvfp4_plan_create_ex(256, 512, 0, None) == nb.NVFP4_ERR_ARG


def test_linear_null_plan_refused():
    buf = np.zeros(64, np.uint8)
    p = buf.ctypes.data
    st = nb.cuda_lib().nvfp4_skinny_linear(None, p, 1, p, p, ctypes.c_float(1.0), p, None)
    assert st == nb.NVFP4_ERR_ARG
    assert nb.cuda_lib().nvfp4_plan_get_info(None, None) == nb.NVFP4_ERR_ARG
    assert nb.cuda_lib().nvfp4_plan_check(None, None) == nb.NVFP4_ERR_ARG
    nb.cuda_lib().nvfp4_plan_destroy(None)  # ignored


# ----------------------------------------------------------------------------- work split
# The kernels split units u = row_block * S + k_step into `grid` contiguous ranges
# [p*T/G, (p+1)*T/G); block_of_unit(u) = ((u+1)*G - 1) / T; partial slot 2p or 2p+1.

def _split(T, G):
    return [(p * T // G, (p + 1) * T // G) for p in range(G)]


def _block_of(u, T, G):
    return ((u + 1) * G - 1) // T


@pytest.mark.parametrize("B,S,sms", [(1, 2, 152), (20, 20, 152), (28, 20, 152), (20, 68, 152), (136, 20, 152),
                                     (594, 20, 152), (3, 1, 152), (7, 3, 4), (5, 7, 5), (2, 9, 11), (40, 2, 152)])
@pytest.mark.parametrize("aligned", [False, True])
def test_work_split_invariants(B, S, sms, aligned):
    T = B * S
    G = min(T, sms)
    if aligned:  # the tcgen05 plan's grid: ranges that never straddle a row block, where it can
        us = [u for u in range(1, 5) if T % u == 0 and S % u == 0 and T // u <= sms]
        ks = [k for k in range(1, B + 1) if B % k == 0 and B // k <= sms][:1]
        if us:  # u <= 4 units of one row block per range
            G = T // us[0]
            assert all((b // S) == ((e - 1) // S) for b, e in _split(T, G))
        elif ks and 20 * (B // ks[0]) >= 17 * sms:  # whole row blocks per range
            G = B // ks[0]
            assert all(b % S == 0 and e % S == 0 for b, e in _split(T, G))
    ranges = _split(T, G)
    assert ranges[0][0] == 0 and ranges[-1][1] == T
    sizes = [e - b for b, e in ranges]
    assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    for p, (b, e) in enumerate(ranges):
        for u in range(b, e):
            assert _block_of(u, T, G) == p
    slots = set()
    for rb in range(B):
        pf, pl = _block_of(rb * S, T, G), _block_of(rb * S + S - 1, T, G)
        covered = []
        for p in range(pf, pl + 1):
            b, e = ranges[p]
            lo, hi = max(b, rb * S), min(e, rb * S + S)
            assert lo < hi
            covered.append((lo, hi))
            if pl > pf:
                slot = 2 * p + (0 if rb == b // S else 1)
                assert slot not in slots
                slots.add(slot)
        # the parts of one row block are contiguous and cover its whole K, in block order
        assert covered[0][0] == rb * S and covered[-1][1] == rb * S + S
        assert all(covered[i][1] == covered[i + 1][0] for i in range(len(covered) - 1))
    assert all(s < 2 * G for s in slots)


# ----------------------------------------------------------------------------- packer

def test_pack_roundtrip_and_nibble_order():
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 16, size=(5, 64), dtype=np.uint8)
    packed = nb.nvfp4_pack_codes(codes)
    assert packed.shape == (5, 32)
    assert np.array_equal(packed, codes[:, 0::2] | (codes[:, 1::2] << 4))
    assert np.array_equal(nb.nvfp4_unpack_codes(packed, 64), codes)
    one = np.zeros((1, 4), np.uint8)
    one[0, 0] = 3
    assert nb.nvfp4_pack_codes(one)[0, 0] == 0x03   # k = 0 -> low nibble
    one[0, 0], one[0, 1] = 0, 3
    assert nb.nvfp4_pack_codes(one)[0, 0] == 0x30   # k = 1 -> high nibble


def test_pack_refuses_bad_codes_and_shapes():
    with pytest.raises(ValueError):
        nb.nvfp4_pack_codes(np.full((2, 4), 16, np.uint8))
    bad = np.zeros((2, 3), np.uint8)
    assert nb.pack_lib().nvfp4_pack_codes(bad.ctypes.data, 2, 3, bad.ctypes.data) == nb.NVFP4_PACK_ERR_ARG


def _torch_e4m3(values):
    import torch
    return torch.as_tensor(np.asarray(values, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encoder_matches_library_cast():
    """Round to nearest even, as torch's float8_e4m3fn cast does, over many magnitudes."""
    rng = np.random.default_rng(1)
    v = np.concatenate([np.exp2(rng.uniform(-12, 8.8, 200000)).astype(np.float32),
                        np.array([0.0, 2.0 ** -9, 2.0 ** -10, 1.5 * 2.0 ** -10, 2.0 ** -6, 448.0, 1.0625,
                                  1.1875, 0.0029296875, 0.0009765625 * 3], np.float32)])
    v = v[v <= 448.0]
    assert np.array_equal(nb.nvfp4_e4m3_encode(v), _torch_e4m3(v))


def test_e4m3_encoder_roundtrips_every_finite_nonnegative_byte():
    import torch
    b = np.arange(0x7F, dtype=np.uint8)                  # 0x00..0x7E: every finite value >= 0
    vals = torch.as_tensor(b).view(torch.float8_e4m3fn).to(torch.float32).numpy()
    assert np.array_equal(nb.nvfp4_e4m3_encode(vals), b)


def test_e4m3_encoder_saturates_and_refuses():
    assert list(nb.nvfp4_e4m3_encode(np.array([448.0, 449.0, 464.0, 1.0e6, np.inf], np.float32))) == [0x7E] * 5
    assert list(nb.nvfp4_e4m3_encode(np.array([-0.0, 0.0], np.float32))) == [0, 0]
    for bad in (-1.0, -1.0e-30, np.nan, -np.inf):
        with pytest.raises(ValueError):
            nb.nvfp4_e4m3_encode(np.array([1.0, bad], np.float32))


# ----------------------------------------------------------------------------- prefill geometry
# nvfp4_prefill_geometry is host-only: the tiles must cover [M, N], the split must give every
# block at least one 256-k unit, and the choice must be a function of (N, K, M, SMs) alone.

@pytest.mark.parametrize("N,K", [(17, 256), (640, 512), (5120, 5120), (34816, 5120), (5120, 17408), (152064, 5120)])
@pytest.mark.parametrize("sms", [1, 8, 152])
def test_prefill_geometry_invariants(N, K, sms):
    U = K // 256
    for M in list(range(1, 70)) + [96, 100, 127, 128, 129, 255, 256, 257, 300, 511, 512, 1000, 1024, 4096]:
        g = nb.nvfp4_prefill_geometry(N, K, M, sms)
        assert g == nb.nvfp4_prefill_geometry(N, K, M, sms)
        bm, mt = g["bm"], g["m_tiles"]
        assert bm % 32 == 0 and 32 <= bm <= (192 if g["k_step"] == 64 else 128), g
        assert g["k_step"] in (64, 128) and 4 <= g["load_stages"] <= 8, g
        assert mt * bm >= M and (mt - 1) * bm < M, g
        assert g["n_tiles"] == -(-N // 256)
        assert 1 <= g["splits"] <= min(U, 32)
        assert g["grid"] == mt * g["n_tiles"] * g["splits"]
        assert g["launches_per_call"] == (3 if g["splits"] > 1 else 2)
        assert g["threads"] == 416 and g["sm_count"] == sms
        assert 0 < g["smem_bytes"] <= 232448
        assert g["M"] == M and g["N"] == N and g["K"] == K


def test_prefill_geometry_refusals():
    info = nb.PrefillInfo()
    lib = nb.cuda_lib()
    assert lib.nvfp4_prefill_geometry(512, 512, 8, 152, None) == nb.NVFP4_ERR_ARG
    assert lib.nvfp4_prefill_geometry(512, 512, 8, 0, ctypes.byref(info)) == nb.NVFP4_ERR_ARG
    for N, K in [(0, 512), (512, 0), (512, 300), (512, 128)]:
        assert lib.nvfp4_prefill_geometry(N, K, 8, 152, ctypes.byref(info)) == nb.NVFP4_ERR_SHAPE
    for M in (0, -3, nb.NVFP4_PREFILL_MAX_ROWS + 1):
        assert lib.nvfp4_prefill_geometry(512, 512, M, 152, ctypes.byref(info)) == nb.NVFP4_ERR_M_RANGE
    h = ctypes.c_void_p(5)
    assert lib.nvfp4_prefill_plan_create(512, 300, 8, ctypes.byref(h)) == nb.NVFP4_ERR_SHAPE and h.value is None
    assert lib.nvfp4_prefill_plan_create(512, 512, 8, None) == nb.NVFP4_ERR_ARG
    buf = np.zeros(64, np.uint8)
    p = buf.ctypes.data
    assert lib.nvfp4_prefill_linear(None, p, 40, p, p, ctypes.c_float(1.0), p, None) == nb.NVFP4_ERR_ARG
    assert lib.nvfp4_prefill_plan_check(None, None) == nb.NVFP4_ERR_ARG
    assert lib.nvfp4_prefill_plan_get_info(None, 40, None) == nb.NVFP4_ERR_ARG
    lib.nvfp4_prefill_plan_destroy(None)  # ignored


# the geometry the cost model picks for the stated projection shapes; each was measured on GB300
# as the fastest or within a few percent of the fastest explicit geometry tried
@pytest.mark.parametrize("N,K,M,want", [
    (5120, 5120, 64, (128, 64, 1, 7)),
    (5120, 5120, 256, (128, 128, 2, 3)),
    (5120, 5120, 1024, (64, 160, 7, 1)),
    (34816, 5120, 128, (128, 128, 1, 1)),
    (34816, 5120, 1024, (128, 128, 8, 1)),
    (5120, 17408, 1024, (64, 160, 7, 1)),
])
def test_prefill_geometry_choices_for_the_stated_shapes(N, K, M, want):
    g = nb.nvfp4_prefill_geometry(N, K, M, 152)
    assert (g["k_step"], g["bm"], g["m_tiles"], g["splits"]) == want, g
