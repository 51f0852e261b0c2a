"""CUDA path (through the C ABI) against the CPU oracle, element by element.

Tolerance (stated acceptance bound): |y - y_ref| <= 4e-3 * sum_k |w_k x_k| + one bfloat16
ulp of |y_ref|, per element.  Row invariance ("10 Kernels" 10.1) is a separate, bitwise gate.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_cases import Case, bf16_bits, to_f64, within_tolerance
from nvfp4_skinny_gb300 import binding as nb
from nvfp4_skinny_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_skinny_gb300 import build
    build.build()
    torch.cuda.init()


# the three projection kernels: tcgen05, the register-direct mma.sync one and the cluster-split
# mma.sync one (which takes only the shapes whose K splits over a cluster, see cluster_takes)
KERNELS = {"tcgen05": nb.NVFP4_PLAN_KERNEL_TCGEN05, "mma": nb.NVFP4_PLAN_KERNEL_MMA_SYNC,
           "cluster": nb.NVFP4_PLAN_KERNEL_CLUSTER}
kernel_param = pytest.mark.parametrize("kernel", list(KERNELS))
KERNEL_IDS = {"tcgen05": nb.NVFP4_KERNEL_TCGEN05, "mma": nb.NVFP4_KERNEL_MMA_SYNC, "cluster": nb.NVFP4_KERNEL_CLUSTER}


def cluster_takes(N, K):
    """Whether the cluster kernel plans (N, K): refused with NVFP4_ERR_SHAPE otherwise."""
    try:
        nb.nvfp4_plan_create_flags(N, K, nb.NVFP4_OUT_BF16, nb.NVFP4_PLAN_KERNEL_CLUSTER).destroy()
        return True
    except nb.Nvfp4Error as e:
        assert e.status == nb.NVFP4_ERR_SHAPE
        return False


def _plan(N, K, f32=False, kernel=None):
    out = nb.NVFP4_OUT_F32 if f32 else nb.NVFP4_OUT_BF16
    if kernel is None:
        return nb.nvfp4_plan_create_ex(N, K, out)
    if kernel == "cluster" and not cluster_takes(N, K):
        pytest.skip("the cluster kernel does not take N=%d K=%d" % (N, K))
    return nb.nvfp4_plan_create_flags(N, K, out, KERNELS[kernel])


def _full_check(case, plan, M=None):
    M = case.M if M is None else M
    y = case.run(plan, M)
    torch.cuda.synchronize()
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK
    y_ref, absdot = case.oracle_full()
    ok, ratio = within_tolerance(to_f64(y), y_ref[:M], absdot[:M])
    assert ok, "max |err|/tol = %.3g" % ratio
    return y


# ------------------------------------------------------------------ small shapes, every element

def test_tiny_workload():
    """The tiny workload: N=256, K=512, M=1, gs=0.01."""
    w = synth.WORKLOADS["tiny"].projections[0]
    case = Case(w.N, w.K, 1, w.seed)
    _full_check(case, _plan(w.N, w.K))


@kernel_param
@pytest.mark.parametrize("N,K", [(256, 256), (300, 768), (1000, 2048), (17, 512), (513, 1280)])
@pytest.mark.parametrize("M", [1, 5, 8, 9, 16, 17, 31, 32])
def test_small_shapes_all_elements(N, K, M, kernel):
    """Several row blocks and k-steps, ragged last row block, every M band."""
    case = Case(N, K, M, seed=100 + N + K + M, outlier_frac=0.01)
    _full_check(case, _plan(N, K, kernel=kernel))


@kernel_param
def test_f32_output_small(kernel):
    case = Case(640, 1024, 7, seed=7)
    plan = _plan(640, 1024, f32=True, kernel=kernel)
    y = case.run(plan)
    torch.cuda.synchronize()
    assert y.dtype == torch.float32
    y_ref, absdot = case.oracle_full()
    ok, ratio = within_tolerance(to_f64(y), y_ref, absdot)
    assert ok, ratio


@kernel_param
def test_split_k_fixup_path_every_element(kernel):
    """More units than blocks with row blocks split across blocks: N=4096, K=8192 (every element)."""
    N, K, M = 4096, 8192, 9
    plan = _plan(N, K, kernel=kernel)
    info = nb.nvfp4_plan_get_info(plan)
    assert info["units"] > info["grid"]
    case = Case(N, K, M, seed=21)
    _full_check(case, plan)


# ------------------------------------------------------------------ edge cases

def _case_with_x(N, K, xf32, seed=5, gs=None):
    x = torch.as_tensor(np.asarray(xf32, np.float32)).to(torch.bfloat16)
    return Case(N, K, x.shape[0], seed, x=x, gs=gs)


@kernel_param
def test_zero_rows_and_mixed_magnitudes(kernel):
    K = 1024
    rng = np.random.default_rng(3)
    x = np.zeros((6, K), np.float32)
    x[1] = rng.standard_normal(K) * 2.0 ** -100     # tiny row
    x[2] = rng.standard_normal(K) * 2.0 ** 100      # huge row
    x[3] = rng.standard_normal(K)
    x[3, 7] = 3.0e4                                 # one large outlier
    x[4] = rng.standard_normal(K) * 2.0 ** -120     # bf16 subnormal-range row
    x[5, ::3] = 1.0
    case = _case_with_x(384, K, x)
    y = _full_check(case, _plan(384, K, kernel=kernel))
    assert torch.all(y[0] == 0)


@kernel_param
def test_extreme_scales_and_codes(kernel):
    N, K = 256, 512
    codes = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, generator=torch.Generator().manual_seed(9))
    scales = torch.full((N, K // 16), 0x7E, dtype=torch.uint8)   # 448, the E4M3 maximum
    scales[::2] = 0x01                                           # 2^-9, the smallest subnormal
    scales[5] = 0x00                                             # zero scale
    codes[7] = 0x88                                              # -0 codes
    x = synth.activations(4, K, 11)
    case = Case(N, K, 4, 0, x=x, codes=codes, scales=scales, gs=1.0)
    _full_check(case, _plan(N, K, kernel=kernel))


@pytest.mark.parametrize("gs", [0.0, -1.0, 1.0e-3, 7.5])
def test_global_scale_values(gs):
    case = Case(256, 512, 3, seed=12, gs=gs)
    _full_check(case, _plan(256, 512))


# ------------------------------------------------------------------ row invariance (bitwise)

def _row_invariance(N, K, seed, Ms=range(1, 33), f32=False, kernel=None):
    plan = _plan(N, K, f32, kernel=kernel)
    x_all = synth.activations(32, K, seed, outlier_frac=0.01).cuda()
    case = Case(N, K, 32, seed, x=x_all.cpu())
    singles = []
    for r in range(32):
        singles.append(case.run(plan, 1, x=x_all[r:r + 1].contiguous()))
    for M in Ms:
        y = case.run(plan, M, x=x_all[:M].contiguous())
        for r in range(M):
            assert torch.equal(y[r], singles[r][0]), "row %d differs at M=%d" % (r, M)
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK


@kernel_param
def test_row_invariance_square(kernel):
    _row_invariance(5120, 5120, seed=2, kernel=kernel)


@kernel_param
@pytest.mark.parametrize("N,K", [(7168, 5120), (5120, 17408), (34816, 5120), (300, 768)])
def test_row_invariance_other_shapes(N, K, kernel):
    # M = 12 / 13 is where the tcgen05 kernel changes its decoder layout (16 / 8 decoder warps)
    _row_invariance(N, K, seed=N % 97, Ms=(1, 2, 8, 9, 12, 13, 16, 17, 24, 32), kernel=kernel)


@kernel_param
def test_row_invariance_head_f32(kernel):
    _row_invariance(152064, 5120, seed=6, Ms=(1, 16, 17, 32), f32=True, kernel=kernel)


# ------------------------------------------------------------------ determinism, graphs

@kernel_param
def test_repeat_and_graph_bit_identical(kernel):
    N, K, M = 5120, 5120, 17
    plan = _plan(N, K, kernel=kernel)
    case = Case(N, K, M, seed=33)
    y0 = case.run(plan)
    y1 = case.run(plan)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    s = torch.cuda.Stream()
    yg = torch.empty_like(y0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        nb.nvfp4_skinny_linear(plan, case.d_x, M, case.d_codes, case.d_scales, case.gs, yg, stream=s)  # warm
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            nb.nvfp4_skinny_linear(plan, case.d_x, M, case.d_codes, case.d_scales, case.gs, yg, stream=s)
    yg.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(yg, y0)
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK


@kernel_param
def test_back_to_back_different_plans(kernel):
    """Calls of several plans queued on one stream (the decode-round pattern) give the
    same bits as the same calls made one at a time."""
    shapes = [(7168, 5120), (5120, 5120), (34816, 5120), (5120, 17408)]
    if kernel == "cluster":
        shapes = [s for s in shapes if cluster_takes(*s)] + [(300, 768)]
    plans = [_plan(N, K, kernel=kernel) for N, K in shapes]
    cases = [Case(N, K, 16, seed=40 + i) for i, (N, K) in enumerate(shapes)]
    alone = []
    for pl, c in zip(plans, cases):
        alone.append(c.run(pl))
        torch.cuda.synchronize()
    queued = [c.run(pl) for pl, c in zip(plans, cases)] * 1
    queued += [c.run(pl) for pl, c in zip(plans, cases)]
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        assert torch.equal(queued[i], alone[i])
        assert torch.equal(queued[i + len(shapes)], alone[i])


# ------------------------------------------------------------------ row strides (pitched x and y)

@kernel_param
@pytest.mark.parametrize("N,K,M", [(5120, 5120, 3), (34816, 5120, 17), (300, 768, 32)])
def test_strided_slices_match_contiguous_bitwise(N, K, M, kernel):
    """x and y as column slices of wider row-major buffers: the same bits as the contiguous
    call for every row, and nothing outside the slices is written."""
    plan = _plan(N, K, kernel=kernel)
    case = Case(N, K, M, seed=N + M)
    y_ref = case.run(plan)
    lda, ldc, x_off, y_off = K + 264, -(-N // 8) * 8 + 136, 8, 16  # row strides (lda + x_off, ldc + y_off) % 8 == 0
    xw = torch.zeros((M, lda + x_off), dtype=torch.bfloat16, device="cuda")
    xw[:, x_off:x_off + K] = case.d_x
    sentinel = torch.tensor(-7.0, dtype=torch.bfloat16)
    yw = torch.full((M, ldc + y_off), float(sentinel), dtype=torch.bfloat16, device="cuda")
    row = lda + x_off
    nb.nvfp4_skinny_linear_strided(plan, xw.view(-1)[x_off:], row, M, case.d_codes, case.d_scales, case.gs,
                                   yw.view(-1)[y_off:], ldc + y_off)
    torch.cuda.synchronize()
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK
    assert torch.equal(yw[:, y_off:y_off + N], y_ref)
    assert bool((yw[:, :y_off] == sentinel).all()) and bool((yw[:, y_off + N:] == sentinel).all())


def test_strided_argument_errors():
    plan = _plan(256, 512)
    case = Case(256, 512, 2, seed=3)
    y = torch.empty((2, 512), dtype=torch.bfloat16, device="cuda")
    xw = torch.zeros((2, 1024), dtype=torch.bfloat16, device="cuda")
    call = lambda lda, ldc, xx=xw: nb.nvfp4_skinny_linear_strided(plan, xx, lda, 2, case.d_codes, case.d_scales,
                                                                 case.gs, y, ldc, check=False)
    assert call(256, 512) == nb.NVFP4_ERR_SHAPE        # lda < K
    assert call(512, 128) == nb.NVFP4_ERR_SHAPE        # ldc < N
    assert call(516, 512) == nb.NVFP4_ERR_ALIGN        # lda not a multiple of 8
    assert call(512, 260) == nb.NVFP4_ERR_ALIGN        # ldc not a multiple of 8
    assert call(1024, 512) == nb.NVFP4_OK


# ------------------------------------------------------------------ gated-MLP input (silu(gate) * up)

def _gate_up(M, K, seed):
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn((M, 2 * K), generator=gen) * 2).to(torch.bfloat16)


@kernel_param
@pytest.mark.parametrize("N,K,M", [(256, 512, 5), (640, 1024, 17), (5120, 17408, 8)])
def test_silu_mul_input(N, K, M, kernel):
    """The down projection fed by a [gate | up] row: every sampled element within the
    tolerance of the oracle applied to x = bf16(silu(gate) * up)."""
    gu = _gate_up(M, K, seed=N + M)
    x_bits = oracle.silu_mul_bf16(bf16_bits(gu), K)
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16)
    case = Case(N, K, M, seed=N + K, x=x)
    plan = _plan(N, K, kernel=kernel)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    nb.nvfp4_skinny_linear_silu_mul(plan, gu.cuda(), 2 * K, M, case.d_codes, case.d_scales, case.gs, y, N)
    torch.cuda.synchronize()
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK
    if N * K <= 1 << 20:
        y_ref, absdot = case.oracle_full()
        ok, ratio = within_tolerance(to_f64(y), y_ref, absdot)
    else:
        rng = np.random.default_rng(M)
        ms, ns = rng.integers(0, M, 256), rng.integers(0, N, 256)
        y_ref, absdot = case.oracle_at(ms, ns)
        ok, ratio = within_tolerance(to_f64(y)[ms, ns], y_ref, absdot)
    assert ok, ratio


@kernel_param
def test_silu_mul_row_invariance_and_refusals(kernel):
    N, K = 5120, 5120
    plan = _plan(N, K, kernel=kernel)
    case = Case(N, K, 1, seed=8)
    gu = _gate_up(32, K, seed=9).cuda()
    y32 = torch.empty((32, N), dtype=torch.bfloat16, device="cuda")
    nb.nvfp4_skinny_linear_silu_mul(plan, gu, 2 * K, 32, case.d_codes, case.d_scales, case.gs, y32, N)
    for r in (0, 7, 31):
        y1 = torch.empty((1, N), dtype=torch.bfloat16, device="cuda")
        nb.nvfp4_skinny_linear_silu_mul(plan, gu[r:r + 1].contiguous(), 2 * K, 1, case.d_codes, case.d_scales,
                                        case.gs, y1, N)
        torch.cuda.synchronize()
        assert torch.equal(y1[0], y32[r])
    call = lambda ld, ldc: nb.nvfp4_skinny_linear_silu_mul(plan, gu, ld, 2, case.d_codes, case.d_scales, case.gs,
                                                           y32, ldc, check=False)
    assert call(K, N) == nb.NVFP4_ERR_SHAPE           # the row holds gate and up: ld >= 2 K
    assert call(2 * K + 4, N) == nb.NVFP4_ERR_ALIGN
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK


# ------------------------------------------------------------------ grouped expert projections

@kernel_param
def test_grouped_experts_match_single_calls_and_oracle(kernel):
    """Eight experts of one (N, K) with their own weights, global scales and row counts: each
    item's bits equal a single call's, and sampled elements meet the oracle's tolerance."""
    N, K = 2048, 1024
    plan = _plan(N, K, kernel=kernel)
    cases = [Case(N, K, M, seed=70 + e, gs=0.01 * (e + 1)) for e, M in enumerate((1, 3, 8, 16, 17, 24, 32, 2))]
    ys = [torch.empty((c.M, N), dtype=torch.bfloat16, device="cuda") for c in cases]
    nb.nvfp4_skinny_linear_grouped(plan, [(c.d_x, c.M, c.d_codes, c.d_scales, c.gs, y) for c, y in zip(cases, ys)])
    torch.cuda.synchronize()
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK
    for c, y in zip(cases, ys):
        assert torch.equal(y, c.run(plan))
        rng = np.random.default_rng(c.M)
        ms, ns = rng.integers(0, c.M, 128), rng.integers(0, N, 128)
        y_ref, absdot = c.oracle_at(ms, ns)
        ok, ratio = within_tolerance(to_f64(y)[ms, ns], y_ref, absdot)
        assert ok, ratio
    torch.cuda.synchronize()
    bad = [(c.d_x, c.M, c.d_codes, c.d_scales, c.gs, y) for c, y in zip(cases, ys)]
    bad[5] = (cases[5].d_x, 33, cases[5].d_codes, cases[5].d_scales, cases[5].gs, ys[5])
    assert nb.nvfp4_skinny_linear_grouped(plan, bad, check=False) == nb.NVFP4_ERR_M_RANGE


# ------------------------------------------------------------------ N-sharding (replicas path)

@pytest.mark.parametrize("cuts", [(2560,), (2000, 3100)])
def test_n_shards_of_one_weight(cuts):
    """The projection shards along N with no exchange: each shard is a plain call on a row
    slice of the same weight (views into the packed arrays, no copies), and its output meets
    the tolerance against the oracle on the whole slice.  Bitwise equality with the unsharded
    call is not claimed: how K is split among blocks follows (N, K), so a shard of another N
    may sum the same terms in another order."""
    N, K, M = 5120, 5120, 16
    case = Case(N, K, M, seed=12)
    y_full = case.run(_plan(N, K))
    bounds = (0,) + tuple(cuts) + (N,)
    y_ref, absdot = case.oracle_full()
    for n0, n1 in zip(bounds[:-1], bounds[1:]):
        plan = _plan(n1 - n0, K)
        y = torch.empty((M, n1 - n0), dtype=torch.bfloat16, device="cuda")
        nb.nvfp4_skinny_linear(plan, case.d_x, M, case.d_codes[n0:n1], case.d_scales[n0:n1], case.gs, y)
        torch.cuda.synchronize()
        assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK
        ok, ratio = within_tolerance(to_f64(y), y_ref[:, n0:n1], absdot[:, n0:n1])
        assert ok, (n0, n1, ratio)
    ok, ratio = within_tolerance(to_f64(y_full), y_ref, absdot)
    assert ok, ratio


# ------------------------------------------------------------------ full-size workloads, sampled

def _sampled(case, plan, M, n_samples=384, seed=0):
    y = case.run(plan, M)
    torch.cuda.synchronize()
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK
    rng = np.random.default_rng(seed)
    ms = np.concatenate([rng.integers(0, M, n_samples), np.full(4, M - 1)])
    ns = np.concatenate([rng.integers(0, case.N, n_samples), [0, case.N - 1, case.N - 2, case.N // 2]])
    y_ref, absdot = case.oracle_at(ms, ns)
    yg = to_f64(y)[ms, ns]
    ok, ratio = within_tolerance(yg, y_ref, absdot)
    assert ok, "max |err|/tol = %.3g" % ratio


@kernel_param
@pytest.mark.parametrize("wl", ["square", "qkv_down", "wide_head"])
def test_full_size_workloads_sampled(wl, kernel):
    w = synth.WORKLOADS[wl]
    for pj in w.projections:
        if kernel == "cluster" and not cluster_takes(pj.N, pj.K):
            continue
        plan = _plan(pj.N, pj.K, pj.f32_out, kernel=kernel)
        x = synth.activations(32, pj.K, pj.seed, outlier_frac=w.outlier_frac)
        case = Case(pj.N, pj.K, 32, pj.seed, x=x)
        for M in w.Ms:
            xm = case.d_x[:M].contiguous()
            y = case.run(plan, M, x=xm)
            torch.cuda.synchronize()
            rng = np.random.default_rng(M)
            ms = rng.integers(0, M, 256)
            ns = rng.integers(0, pj.N, 256)
            y_ref, absdot = case.oracle_at(ms, ns)
            ok, ratio = within_tolerance(to_f64(y)[ms, ns], y_ref, absdot)
            assert ok, (pj.name, M, ratio)
        assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK


@kernel_param
def test_round_workload_first_layer_sampled(kernel):
    """The decode-round shapes with their per-(layer, projection) seeds, layer 0."""
    for pj in synth.WORKLOADS["round"].projections[:4]:
        if kernel == "cluster" and not cluster_takes(pj.N, pj.K):
            continue
        plan = _plan(pj.N, pj.K, kernel=kernel)
        case = Case(pj.N, pj.K, 32, pj.seed)
        _sampled(case, plan, 32, seed=pj.seed)


# ------------------------------------------------------------------ argument errors (nothing launched)

def test_argument_errors():
    plan = _plan(256, 512)
    case = Case(256, 512, 2, seed=1)
    y = torch.empty((2, 256), dtype=torch.bfloat16, device="cuda")
    lin = lambda **kw: nb.nvfp4_skinny_linear(
        kw.get("plan", plan), kw.get("x", case.d_x), kw.get("M", 2), kw.get("codes", case.d_codes),
        kw.get("scales", case.d_scales), 1.0, kw.get("y", y), check=False)
    assert lin(M=0) == nb.NVFP4_ERR_M_RANGE
    assert lin(M=33) == nb.NVFP4_ERR_M_RANGE
    assert lin(x=0) == nb.NVFP4_ERR_ARG
    assert lin(codes=0) == nb.NVFP4_ERR_ARG
    assert lin(y=0) == nb.NVFP4_ERR_ARG
    assert lin(plan=0) == nb.NVFP4_ERR_ARG
    assert lin(x=case.d_x.data_ptr() + 2) == nb.NVFP4_ERR_ALIGN
    assert lin(codes=case.d_codes.data_ptr() + 8) == nb.NVFP4_ERR_ALIGN
    assert lin() == nb.NVFP4_OK
    torch.cuda.synchronize()
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK


@kernel_param
def test_plan_info_independent_of_M(kernel):
    for N, K in [(5120, 5120), (152064, 5120), (256, 512), (5120, 17408)]:
        if kernel == "cluster" and not cluster_takes(N, K):
            continue
        info = nb.nvfp4_plan_get_info(_plan(N, K, kernel=kernel))
        assert info["N"] == N and info["K"] == K
        assert info["kernel"] == KERNEL_IDS[kernel]
        if kernel == "cluster":  # clusters of C blocks over 16-row tiles, K / C per block
            C = info["cluster_size"]
            assert C in (2, 4, 8) and info["grid"] % C == 0 and info["grid"] <= 2 * info["sm_count"]
            assert info["rows_per_block"] == 16 and info["row_blocks"] == -(-N // 16)
            assert info["k_steps"] * info["k_step"] == K and info["launches_per_call"] == 1
            continue
        assert info["row_blocks"] == -(-N // info["rows_per_block"])
        assert info["units"] == info["row_blocks"] * (K // info["k_step"])
        if kernel == "tcgen05":
            # min(units, SMs), or fewer blocks of u <= 4 units whose ranges never straddle a row block
            steps, units, sms = K // info["k_step"], info["units"], info["sm_count"]
            aligned = [units // u for u in range(1, 5) if units % u == 0 and steps % u == 0 and units // u <= sms]
            rb = units // steps
            whole = [rb // k for k in range(1, rb + 1) if rb % k == 0 and rb // k <= sms][:1]
            whole = [g for g in whole if 20 * g >= 17 * sms]  # whole row blocks, >= 85 % of the SMs
            assert info["grid"] == (aligned or whole or [min(units, sms)])[0]
            # the block size of calls with M > 12: 16 decoder warps (768 threads) on plans whose
            # blocks stream at least 40 units, else 8 (512); M <= 12 always runs 16
            wide = -(-units // info["grid"]) >= 40
            assert info["threads"] == (768 if wide else 512)
        else:  # the register-direct kernel runs two blocks per SM
            assert info["grid"] == min(info["units"], 2 * info["sm_count"])
        assert info["warps_rows"] * info["warps_k"] * 32 == (info["threads"] if kernel == "mma" else 32)
