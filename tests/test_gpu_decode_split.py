"""The decode and the work split of both projection kernels, through the C ABI.

- The whole E2M1 x E4M3 product table ("10 Kernels" 10.2: four-bit weights times an eight-bit
  group scale, at most six significant bits, so exact in fp16 and bf16) decoded by the real
  kernels: every code against every finite scale byte, one product per output element, compared
  exactly with the product of the OCP definitions.
- Shapes that force the tcgen05 kernel's two-launch mode (activation preparation, then the
  projection), blocks whose unit range spans three row-block segments, and ragged last row
  blocks, checked on every element against the oracle at M = 1, 16, 17 and 32.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import Case, to_f64, within_tolerance
from nvfp4_skinny_gb300 import binding as nb

pytestmark = pytest.mark.gpu

KERNELS = {"tcgen05": nb.NVFP4_PLAN_KERNEL_TCGEN05, "mma": nb.NVFP4_PLAN_KERNEL_MMA_SYNC,
           "cluster": nb.NVFP4_PLAN_KERNEL_CLUSTER}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_skinny_gb300 import build
    build.build()
    torch.cuda.init()


# every finite E4M3 byte: 0x00..0x7E and their negatives 0x80..0xFE (0x7F and 0xFF are NaN)
SCALE_BYTES = [b for b in range(256) if (b & 0x7F) != 0x7F]


@pytest.mark.parametrize("kernel", list(KERNELS))
@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("M,stride", [(16, 1), (32, 1), (16, 17), (12, 21)])
def test_decode_table_exhaustive(kernel, out, M, stride):
    """Row n of the weight has scale byte SCALE_BYTES[n] in every block and code k % 16 at k;
    activation row m is one-hot at k_m = stride m mod K; gs = 1.  Then y[m, n] =
    e2m1(k_m % 16) * e4m3(s_n) exactly: each element is a single product, which fp16, fp32 and
    bf16 all hold.  Strides 17 and 21 put the one-hot positions in both 128-k halves of the unit
    and every 16-byte chunk of a row (all 16 codes at stride 17), and M = 12 runs the tcgen05
    kernel's 16-decoder-warp layout, whose warps each convert one half."""
    N, K = len(SCALE_BYTES), 256
    code_k = np.arange(K) % 16
    codes = np.tile((code_k[0::2] | (code_k[1::2] << 4)).astype(np.uint8), (N, 1))
    scales = np.repeat(np.array(SCALE_BYTES, np.uint8)[:, None], K // 16, axis=1)
    x = torch.zeros((M, K), dtype=torch.float32)
    k_m = (stride * np.arange(M)) % K
    x[torch.arange(M), torch.from_numpy(k_m)] = 1.0
    x = x.to(torch.bfloat16)
    f32 = out == "f32"
    plan = nb.nvfp4_plan_create_flags(N, K, nb.NVFP4_OUT_F32 if f32 else nb.NVFP4_OUT_BF16, KERNELS[kernel])
    y = torch.empty((M, N), dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
    nb.nvfp4_skinny_linear(plan, x.cuda(), M, torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), 1.0,
                           y)
    torch.cuda.synchronize()
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK
    want = np.array([[oracle.e2m1(int(k_m[m]) % 16) * oracle.e4m3(s) for s in SCALE_BYTES] for m in range(M)],
                    np.float64)
    assert np.all(want.astype(np.float32).astype(np.float64) == want)          # exact in fp32
    got = y.float().cpu().numpy().astype(np.float64)
    if not f32:
        bf = torch.from_numpy(want.astype(np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)
        assert np.all(bf == want)                                                  # exact in bf16
    bad = np.argwhere(got != want)   # +0 and -0 compare equal
    assert bad.size == 0, [(int(m), hex(SCALE_BYTES[n]), got[m, n], want[m, n]) for m, n in bad[:8]]


@pytest.mark.parametrize("kernel", ["tcgen05", "mma"])
@pytest.mark.parametrize("N,K,Ms", [(100000, 512, (1, 17)), (100000, 1024, (16, 32)), (2000, 32768, (1, 17))])
def test_split_modes_every_element(kernel, N, K, Ms):
    """Many units per block (the tcgen05 kernel's two-launch mode), blocks covering up to three
    row-block segments (K = 512), a ragged last row block (N = 100000) and a deep k-split
    (K = 32768): every element within the tolerance of the oracle."""
    plan = nb.nvfp4_plan_create_flags(N, K, nb.NVFP4_OUT_BF16, KERNELS[kernel])
    info = nb.nvfp4_plan_get_info(plan)
    if kernel == "tcgen05":
        assert info["launches_per_call"] == 2
    assert info["units"] > 2 * info["grid"] or K == 32768
    case = Case(N, K, max(Ms), seed=N % 1000 + K, outlier_frac=0.01)
    y_ref, absdot = case.oracle_full()
    for M in Ms:
        y = case.run(plan, M, x=case.d_x[:M].contiguous())
        torch.cuda.synchronize()
        ok, ratio = within_tolerance(to_f64(y), y_ref[:M], absdot[:M])
        assert ok, (M, ratio)
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK


@pytest.mark.parametrize("N,K", [(5120, 5120), (4000, 6144), (2000, 3072), (999, 1536), (2500, 2048), (160, 1280)])
def test_cluster_split_every_element(N, K):
    """The cluster kernel's work split on every element: clusters of 8, 4 and 2 blocks (K / C of
    6, 3, 3, 2, 1 and 5 units of 128), tiles shared by two or more warps, warps with no tile-unit,
    panels of unequal tile counts and a ragged last tile."""
    plan = nb.nvfp4_plan_create_flags(N, K, nb.NVFP4_OUT_BF16, nb.NVFP4_PLAN_KERNEL_CLUSTER)
    info = nb.nvfp4_plan_get_info(plan)
    assert info["kernel"] == nb.NVFP4_KERNEL_CLUSTER and info["launches_per_call"] == 1
    assert K % (info["cluster_size"] * 128) == 0 and K // (info["cluster_size"] * 128) <= 6
    case = Case(N, K, 32, seed=N % 1000 + K, outlier_frac=0.01)
    y_ref, absdot = case.oracle_full()
    for M in (1, 9, 17, 32):
        y = case.run(plan, M, x=case.d_x[:M].contiguous())
        torch.cuda.synchronize()
        ok, ratio = within_tolerance(to_f64(y), y_ref[:M], absdot[:M])
        assert ok, (M, ratio)
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK
