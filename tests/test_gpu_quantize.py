"""Device BF16 -> NVFP4 quantizer (through the C ABI) against the CPU oracle, bit for bit:
every code and scale is a rounding decision taken in the same fp32 precision on both sides."""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import bf16_bits
from nvfp4_skinny_gb300 import binding as nb
from nvfp4_skinny_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_skinny_gb300 import build
    build.build()
    torch.cuda.init()


def _weights(rows, K, seed):
    gen = torch.Generator().manual_seed(seed)
    w = torch.randn((rows, K), generator=gen)
    w = w * torch.exp2(torch.randint(-12, 6, (rows, K // 16), generator=gen).float()).repeat_interleave(16, dim=1)
    w[0, :16] = 0.0                        # an all-zero block
    w[1, 16:32] = 3.0e30                   # a block far above the E4M3 range
    w[2, 32:48] = 1.0e-30                  # a block that needs a subnormal (or zero) scale
    w[3, 48:64] = torch.tensor([0.25, -0.25, 0.75, -0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -6.0, 7.0, 0.0, -0.0,
                                1.0, -1.0])  # ties of the E2M1 grid under scale 1
    return w.to(torch.bfloat16)


def _device_quantize(w, gs, ldw=None):
    rows, K = w.shape
    ldw = K if ldw is None else ldw
    wd = torch.zeros((rows, ldw), dtype=torch.bfloat16, device="cuda")
    wd[:, :K] = w.cuda()
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, K // 16), dtype=torch.uint8, device="cuda")
    nb.nvfp4_quantize_bf16(wd, rows, K, ldw, gs, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("gs", [1.0, 0.0625, 7.5])
@pytest.mark.parametrize("ldw_pad", [0, 24])
def test_quantizer_matches_oracle_bitwise(gs, ldw_pad):
    w = _weights(300, 1024, seed=int(gs * 16) + ldw_pad)
    codes, scales = _device_quantize(w, gs, ldw=1024 + ldw_pad)
    codes_ref, scales_ref = oracle.quantize_nvfp4(bf16_bits(w), gs)
    assert np.array_equal(scales, scales_ref)
    assert np.array_equal(codes, codes_ref)


@pytest.mark.parametrize("gs", [1.0, 0.0625, 7.5])
def test_device_and_host_quantizers_agree_bitwise(gs):
    """The device kernel and the packer library's host quantizer take every rounding decision
    alike: the same codes and scales, byte for byte, on the special blocks and on random ones."""
    w = _weights(257, 2048, seed=int(gs * 32) + 5)
    codes, scales = _device_quantize(w, gs)
    from nvfp4_skinny_gb300 import build
    build.build_pack()
    codes_h, scales_h = nb.nvfp4_quantize_bf16_host(bf16_bits(w), w_global_scale=gs)
    assert np.array_equal(scales, scales_h)
    assert np.array_equal(codes, codes_h)


def test_quantizer_round_trip_of_representable_blocks():
    rng = np.random.default_rng(33)
    rows, K = 64, 512
    sc = rng.integers(0x20, 0x60, (rows, K // 16)).astype(np.uint8)
    code = rng.integers(0, 16, (rows, K)).astype(np.uint8)
    code[code == 8] = 0
    code[:, ::16] = 7
    sv = np.array([oracle.e4m3(int(b)) for b in sc.ravel()]).reshape(sc.shape)
    cv = np.array([oracle.e2m1(int(c)) for c in code.ravel()]).reshape(code.shape)
    w = torch.from_numpy((cv.reshape(rows, K // 16, 16) * sv[:, :, None]).reshape(rows, K).astype(np.float32))
    codes, scales = _device_quantize(w.to(torch.bfloat16), 1.0)
    assert np.array_equal(scales, sc)
    assert np.array_equal(codes[:, :] & 0xF, code[:, 0::2]) and np.array_equal(codes >> 4, code[:, 1::2])


def test_quantize_then_project_matches_oracle():
    """A bf16 weight quantized on the device feeds the projection; the projection matches the
    oracle applied to those codes and scales."""
    from gpu_cases import Case, to_f64, within_tolerance
    rows, K, M = 768, 1024, 4
    w = _weights(rows, K, seed=5)
    codes, scales = _device_quantize(w, 0.5)
    case = Case(rows, K, M, seed=6, codes=torch.from_numpy(codes), scales=torch.from_numpy(scales), gs=0.5)
    y = case.run(nb.nvfp4_plan_create(rows, K))
    torch.cuda.synchronize()
    y_ref, absdot = case.oracle_full()
    ok, ratio = within_tolerance(to_f64(y), y_ref, absdot)
    assert ok, ratio


def test_quantizer_refusals():
    w = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    codes = torch.empty((4, 32), dtype=torch.uint8, device="cuda")
    scales = torch.empty((4, 4), dtype=torch.uint8, device="cuda")
    q = lambda K, ldw, gs: nb.nvfp4_quantize_bf16(w, 4, K, ldw, gs, codes, scales, check=False)
    assert q(40, 64, 1.0) == nb.NVFP4_ERR_SHAPE       # K not a multiple of 16
    assert q(64, 48, 1.0) == nb.NVFP4_ERR_SHAPE       # ldw < K
    assert q(64, 64, 0.0) == nb.NVFP4_ERR_ARG         # the global scale must be positive
    assert q(64, 64, float("nan")) == nb.NVFP4_ERR_ARG
    assert q(64, 68, 1.0) == nb.NVFP4_ERR_ALIGN       # ldw not a multiple of 8
    assert q(64, 64, 1.0) == nb.NVFP4_OK


@pytest.mark.parametrize("kernel", [nb.NVFP4_PLAN_KERNEL_TCGEN05, nb.NVFP4_PLAN_KERNEL_MMA_SYNC])
def test_weights_written_on_the_stream_then_projected(kernel):
    """Weights produced on the same stream, with no host synchronisation before the projection,
    by plans created with NVFP4_PLAN_WEIGHTS_AFTER_WAIT:
    - by the library's quantizer (device BF16 -> NVFP4);
    - by a kernel that lets its dependents launch early: one of the library's own projections,
      whose bf16 output bytes are then used as the next projection's codes.
    Each projection must read the weights as written, which the oracle on the final bytes
    checks."""
    from gpu_cases import Case, to_f64, within_tolerance
    flags = kernel | nb.NVFP4_PLAN_WEIGHTS_AFTER_WAIT
    s = torch.cuda.Stream()
    # 1) quantize -> project
    rows, K, M = 768, 1024, 4
    w = _weights(rows, K, seed=15).cuda()
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, K // 16), dtype=torch.uint8, device="cuda")
    x = synth.activations(M, K, 16).cuda()
    y = torch.empty((M, rows), dtype=torch.bfloat16, device="cuda")
    plan = nb.nvfp4_plan_create_flags(rows, K, nb.NVFP4_OUT_BF16, flags)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        nb.nvfp4_quantize_bf16(w, rows, K, K, 0.5, codes, scales, stream=s)
        nb.nvfp4_skinny_linear(plan, x, M, codes, scales, 0.5, y, stream=s)
    s.synchronize()
    case = Case(rows, K, M, seed=16, x=x.cpu(), codes=codes.cpu(), scales=scales.cpu(), gs=0.5)
    y_ref, absdot = case.oracle_full()
    ok, ratio = within_tolerance(to_f64(y), y_ref, absdot)
    assert ok, ratio
    assert nb.nvfp4_plan_check(plan, s) == nb.NVFP4_OK
    # 2) projection A writes y_a; projection B reads y_a's bytes as its codes
    Na, Ka, Ma = 1024, 512, 16   # y_a: 16 x 1024 bf16 = 32 KB = codes of a [64, 1024] weight
    Nb, Kb, Mb = 64, 1024, 3
    ca, sa, gsa = synth.weights(Na, Ka, 17, device="cuda")
    xa = synth.activations(Ma, Ka, 18, device="cuda")
    y_a = torch.empty((Ma, Na), dtype=torch.bfloat16, device="cuda")
    sb = torch.full((Nb, Kb // 16), 0x30, dtype=torch.uint8, device="cuda")  # E4M3 0.5
    xb = synth.activations(Mb, Kb, 19, device="cuda")
    y_b = torch.empty((Mb, Nb), dtype=torch.bfloat16, device="cuda")
    plan_a = nb.nvfp4_plan_create_flags(Na, Ka, nb.NVFP4_OUT_BF16, kernel)
    plan_b = nb.nvfp4_plan_create_flags(Nb, Kb, nb.NVFP4_OUT_BF16, flags)
    y_a.zero_()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        nb.nvfp4_skinny_linear(plan_a, xa, Ma, ca, sa, gsa, y_a, stream=s)
        nb.nvfp4_skinny_linear(plan_b, xb, Mb, y_a.view(torch.uint8).view(Nb, Kb // 2), sb, 1.0, y_b, stream=s)
    s.synchronize()
    cb = y_a.view(torch.uint8).view(Nb, Kb // 2).cpu()
    assert bool((cb != 0).any())
    case = Case(Nb, Kb, Mb, seed=20, x=xb.cpu(), codes=cb, scales=sb.cpu(), gs=1.0)
    y_ref, absdot = case.oracle_full()
    ok, ratio = within_tolerance(to_f64(y_b), y_ref, absdot)
    assert ok, ratio
