"""One-launch variants of the projection ("Module ops"): two weights over one input
(w4a16_gemv_dual), interleaved weight rows stored deinterleaved (w4a16_gemv_qg, w4a16_gemv_qkvz),
and grouped experts over device tables (Nvfp4ExpertTables), through the C ABI, against the
oracle and against the plain call."""
import numpy as np
import pytest
import torch

from gpu_cases import Case, to_f64, within_tolerance
from nvfp4_skinny_gb300 import binding as nb

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_skinny_gb300 import build
    build.build()
    torch.cuda.init()


# ------------------------------------------------------------------ dual

@pytest.mark.parametrize("kernel_flag", [0, nb.NVFP4_PLAN_KERNEL_MMA_SYNC])
@pytest.mark.parametrize("N,K", [(1000, 2048), (5120, 5120), (700, 17408)])
def test_dual_matches_oracle_and_is_row_invariant(N, K, kernel_flag):
    """Both outputs of a dual call within the oracle's tolerance on every element, at M = 1, 9,
    17 and 32, and each activation row's bits the same at every M."""
    plan = nb.nvfp4_plan_create_flags(N, K, nb.NVFP4_OUT_BF16, nb.NVFP4_PLAN_DUAL | kernel_flag)
    info = nb.nvfp4_plan_get_info(plan)
    assert info["kernel"] in (nb.NVFP4_KERNEL_CLUSTER, nb.NVFP4_KERNEL_MMA_SYNC)
    if kernel_flag:
        assert info["kernel"] == nb.NVFP4_KERNEL_MMA_SYNC
    c0 = Case(N, K, 32, seed=N + K, outlier_frac=0.01)
    c1 = Case(N, K, 32, seed=N + K + 1, x=c0.x, gs=0.25)
    r0, a0 = c0.oracle_full() if N * K <= 1 << 24 else (None, None)
    r1, a1 = c1.oracle_full() if N * K <= 1 << 24 else (None, None)
    ys = {}
    for M in (1, 9, 17, 32):
        xm = c0.d_x[:M].contiguous()
        y0 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        y1 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        nb.nvfp4_skinny_linear_dual(plan, xm, M, (c0.d_codes, c0.d_scales, c0.gs), (c1.d_codes, c1.d_scales, c1.gs),
                                    y0, y1)
        torch.cuda.synchronize()
        ys[M] = (y0, y1)
        if r0 is not None:
            for y, r, a in ((y0, r0, a0), (y1, r1, a1)):
                ok, ratio = within_tolerance(to_f64(y), r[:M], a[:M])
                assert ok, (M, ratio)
        else:
            rng = np.random.default_rng(M)
            ms, ns = rng.integers(0, M, 256), rng.integers(0, N, 256)
            for y, c in ((y0, c0), (y1, c1)):
                r, a = c.oracle_at(ms, ns)
                ok, ratio = within_tolerance(to_f64(y)[ms, ns], r, a)
                assert ok, (M, ratio)
    for M in (1, 9, 17):
        for o in range(2):
            assert torch.equal(ys[M][o], ys[32][o][:M]), (M, o)
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK


def test_dual_refusals():
    plan = nb.nvfp4_plan_create_flags(512, 1024, nb.NVFP4_OUT_BF16, nb.NVFP4_PLAN_DUAL)
    c = Case(512, 1024, 2, seed=3)
    y = torch.empty((2, 512), dtype=torch.bfloat16, device="cuda")
    # a dual plan takes only dual calls
    assert nb.nvfp4_skinny_linear(plan, c.d_x, 2, c.d_codes, c.d_scales, 1.0, y, check=False) == nb.NVFP4_ERR_ARG
    plain = nb.nvfp4_plan_create(512, 1024)
    assert nb.nvfp4_skinny_linear_dual(plain, c.d_x, 2, (c.d_codes, c.d_scales, 1.0), (c.d_codes, c.d_scales, 1.0),
                                       y, y, check=False) == nb.NVFP4_ERR_ARG
    with pytest.raises(nb.Nvfp4Error):  # the tcgen05 kernel has no dual form
        nb.nvfp4_plan_create_flags(512, 1024, nb.NVFP4_OUT_BF16, nb.NVFP4_PLAN_DUAL | nb.NVFP4_PLAN_KERNEL_TCGEN05)
    torch.cuda.synchronize()


# ------------------------------------------------------------------ deinterleaved output

def _deinterleave_order(N, part_rows):
    """Output position of every weight row (the definition, written out)."""
    S = sum(part_rows)
    G = N // S
    out = np.empty(N, np.int64)
    offs = np.concatenate([[0], np.cumsum(part_rows)[:-1]])
    for n in range(N):
        g, o = divmod(n, S)
        q = int(np.searchsorted(np.cumsum(part_rows), o, side="right"))
        out[n] = G * offs[q] + g * part_rows[q] + (o - offs[q])
    return out


@pytest.mark.parametrize("kernel", [nb.NVFP4_PLAN_KERNEL_TCGEN05, nb.NVFP4_PLAN_KERNEL_MMA_SYNC,
                                    nb.NVFP4_PLAN_KERNEL_CLUSTER])
@pytest.mark.parametrize("N,K,parts", [(2048, 1024, (128, 128)),            # Q | gate per head
                                       (3072, 1024, (256, 64, 64, 128)),   # Q | K | V | Z per group
                                       (5120, 5120, (128, 128)),
                                       (1152, 512, (48, 24, 24, 48))])     # parts off the 16-row tiles
def test_deinterleaved_is_the_plain_result_permuted(N, K, parts, kernel):
    plan = nb.nvfp4_plan_create_flags(N, K, nb.NVFP4_OUT_BF16, kernel)
    case = Case(N, K, 17, seed=N + len(parts))
    order = torch.from_numpy(_deinterleave_order(N, parts)).cuda()
    for M in (1, 17):
        xm = case.d_x[:M].contiguous()
        y = case.run(plan, M, x=xm)
        yd = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        nb.nvfp4_skinny_linear_deinterleaved(plan, xm, M, case.d_codes, case.d_scales, case.gs, yd, parts)
        torch.cuda.synchronize()
        want = torch.empty_like(y)
        want[:, order] = y
        assert torch.equal(yd, want), M
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK


def test_deinterleaved_refusals():
    plan = nb.nvfp4_plan_create(1000, 512)
    c = Case(1000, 512, 1, seed=1)
    y = torch.empty((1, 1000), dtype=torch.bfloat16, device="cuda")
    call = lambda parts: nb.nvfp4_skinny_linear_deinterleaved(plan, c.d_x, 1, c.d_codes, c.d_scales, 1.0, y, parts,
                                                              check=False)
    assert call((100, 100)) == nb.NVFP4_OK          # 5 groups of 200 rows
    assert call((300, 100)) == nb.NVFP4_ERR_SHAPE   # 1000 % 400 != 0
    assert call((600, 600)) == nb.NVFP4_ERR_SHAPE   # one group is more than N
    assert call((10, 0)) == nb.NVFP4_ERR_ARG
    assert call((10,)) == nb.NVFP4_ERR_ARG
    assert call((10, 10, 10, 10, 10)) == nb.NVFP4_ERR_ARG
    torch.cuda.synchronize()


# ------------------------------------------------------------------ grouped experts over device tables

def _tables(cases, ys):
    ptr = lambda ts: torch.tensor([t.data_ptr() for t in ts], dtype=torch.int64, device="cuda")
    return {
        "w_codes": ptr([c.d_codes for c in cases]),
        "w_block_scales": ptr([c.d_scales for c in cases]),
        "w_global_scales": torch.tensor([c.gs for c in cases], dtype=torch.float32, device="cuda"),
        "x": ptr([c.d_x for c in cases]),
        "M": torch.tensor([c.M for c in cases], dtype=torch.int32, device="cuda"),
        "y": ptr(ys),
    }


@pytest.mark.parametrize("N,K", [(2048, 1024), (5120, 5120)])
def test_grouped_tables_equal_single_calls(N, K):
    """Experts with their own weights, scales and row counts in one launch: each expert's bits
    equal a single call's on the same plan."""
    plan = nb.nvfp4_plan_create_flags(N, K, nb.NVFP4_OUT_BF16, nb.NVFP4_PLAN_KERNEL_CLUSTER)
    Ms = (1, 3, 8, 17, 32, 2)
    cases = [Case(N, K, M, seed=90 + e, gs=0.01 * (e + 1)) for e, M in enumerate(Ms)]
    ys = [torch.full((max(c.M, 1), N), -7.0, dtype=torch.bfloat16, device="cuda") for c in cases]
    t = _tables(cases, ys)
    nb.nvfp4_skinny_linear_grouped_tables(plan, t, len(cases), 32)
    torch.cuda.synchronize()
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK
    for c, y in zip(cases, ys):
        single = c.run(plan)
        torch.cuda.synchronize()
        assert torch.equal(y[:c.M], single), c.M
    # sampled elements of one expert against the oracle
    c, y = cases[3], ys[3]
    rng = np.random.default_rng(0)
    ms, ns = rng.integers(0, c.M, 128), rng.integers(0, N, 128)
    r, a = c.oracle_at(ms, ns)
    ok, ratio = within_tolerance(to_f64(y)[ms, ns], r, a)
    assert ok, ratio


def test_grouped_tables_rows_out_of_range_and_refusals():
    N, K = 1024, 1024
    plan = nb.nvfp4_plan_create_flags(N, K, nb.NVFP4_OUT_BF16, nb.NVFP4_PLAN_KERNEL_CLUSTER)
    cases = [Case(N, K, 4, seed=1), Case(N, K, 4, seed=2), Case(N, K, 4, seed=3)]
    ys = [torch.full((4, N), -7.0, dtype=torch.bfloat16, device="cuda") for _ in cases]
    t = _tables(cases, ys)
    t["M"] = torch.tensor([4, 9, 0], dtype=torch.int32, device="cuda")  # 9 > max_M = 8; 0 rows
    nb.nvfp4_skinny_linear_grouped_tables(plan, t, 3, 8)
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_ERR_M_RANGE
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK            # the word was cleared
    assert torch.all(ys[1] == -7.0)                              # the refused entry wrote nothing
    assert torch.all(ys[2] == -7.0)                              # an entry of no rows writes nothing
    assert torch.equal(ys[0], cases[0].run(plan))
    other = nb.nvfp4_plan_create(N, K)                           # tcgen05 plan: no device-table form
    assert nb.nvfp4_skinny_linear_grouped_tables(other, t, 2, 8, check=False) == nb.NVFP4_ERR_ARG
    assert nb.nvfp4_skinny_linear_grouped_tables(plan, t, 0, 8, check=False) == nb.NVFP4_ERR_ARG
    assert nb.nvfp4_skinny_linear_grouped_tables(plan, t, 2, 33, check=False) == nb.NVFP4_ERR_M_RANGE
    torch.cuda.synchronize()


# ------------------------------------------------------------------ fp32 outputs of the variants

def test_variants_fp32_output():
    """Dual, deinterleaved and grouped-table calls on fp32-output plans: the same values as the
    bf16 plans before rounding, within the oracle's tolerance, and the grouped bits equal to
    single calls."""
    N, K, M = 768, 1024, 5
    c0 = Case(N, K, M, seed=71)
    c1 = Case(N, K, M, seed=72, x=c0.x, gs=0.5)
    r0, a0 = c0.oracle_full()
    r1, a1 = c1.oracle_full()
    dual = nb.nvfp4_plan_create_flags(N, K, nb.NVFP4_OUT_F32, nb.NVFP4_PLAN_DUAL)
    y0 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    y1 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    nb.nvfp4_skinny_linear_dual(dual, c0.d_x, M, (c0.d_codes, c0.d_scales, c0.gs), (c1.d_codes, c1.d_scales, c1.gs),
                                y0, y1)
    torch.cuda.synchronize()
    for y, r, a in ((y0, r0, a0), (y1, r1, a1)):
        ok, ratio = within_tolerance(to_f64(y), r, a)
        assert ok, ratio
    parts = (64, 32, 32, 64)
    order = torch.from_numpy(_deinterleave_order(N, parts)).cuda()
    for kernel in (nb.NVFP4_PLAN_KERNEL_TCGEN05, nb.NVFP4_PLAN_KERNEL_MMA_SYNC, nb.NVFP4_PLAN_KERNEL_CLUSTER):
        plan = nb.nvfp4_plan_create_flags(N, K, nb.NVFP4_OUT_F32, kernel)
        y = c0.run(plan)
        yd = torch.empty_like(y)
        nb.nvfp4_skinny_linear_deinterleaved(plan, c0.d_x, M, c0.d_codes, c0.d_scales, c0.gs, yd, parts)
        torch.cuda.synchronize()
        want = torch.empty_like(y)
        want[:, order] = y
        assert torch.equal(yd, want), kernel
        ok, ratio = within_tolerance(to_f64(y), r0, a0)
        assert ok, (kernel, ratio)
    plan = nb.nvfp4_plan_create_flags(N, K, nb.NVFP4_OUT_F32, nb.NVFP4_PLAN_KERNEL_CLUSTER)
    ys = [torch.empty((M, N), dtype=torch.float32, device="cuda") for _ in range(2)]
    nb.nvfp4_skinny_linear_grouped_tables(plan, _tables([c0, c1], ys), 2, M)
    torch.cuda.synchronize()
    assert nb.nvfp4_plan_check(plan) == nb.NVFP4_OK
    assert torch.equal(ys[0], c0.run(plan)) and torch.equal(ys[1], c1.run(plan))
