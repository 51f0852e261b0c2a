"""Prefill projection (activation rows above the skinny band, "10.2 NVFP4 matrix products")
through the C ABI against the CPU oracle.

Same acceptance bound as the skinny path: |y - y_ref| <= 4e-3 * sum_k |w_k x_k| + one bfloat16
ulp of |y_ref|, per element.  The shapes are chosen so that the launch geometry covers one and
several activation tiles with a ragged last tile, tile heights from 32 to 192, both pipeline
steps (64 and 128 k), weight row counts below one tile and with a ragged last tile, and one and
several k-splits (the reduction launch).
"""
import numpy as np
import pytest
import torch

from gpu_cases import Case, to_f64, within_tolerance
from nvfp4_skinny_gb300 import binding as nb
from nvfp4_skinny_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_skinny_gb300 import build
    build.build()
    torch.cuda.init()


def _run(plan, case, M=None, x=None):
    M = case.M if M is None else M
    dx = case.d_x if x is None else x
    y = torch.empty((M, case.N), dtype=torch.bfloat16, device="cuda")
    nb.nvfp4_prefill_linear(plan, dx, M, case.d_codes, case.d_scales, case.gs, y)
    return y


def _geometry(plan, M):
    return nb.nvfp4_prefill_plan_get_info(plan, M)


@pytest.mark.parametrize("N,K,M", [
    (640, 512, 33),      # two activation tiles of 32, three weight tiles (ragged)
    (300, 768, 100),     # N between one and two weight tiles
    (17, 256, 40),       # N below one weight tile, one 256-k unit
    (513, 1280, 257),    # nine activation tiles, ragged in both dimensions
    (1024, 4096, 64),    # k split sixteen ways: the reduction launch
    (1024, 8192, 100),   # k split eight ways, four activation tiles
])
def test_small_shapes_every_element(N, K, M):
    case = Case(N, K, M, seed=900 + N + K + M, outlier_frac=0.01)
    plan = nb.nvfp4_prefill_plan_create(N, K, M)
    y = _run(plan, case)
    torch.cuda.synchronize()
    assert nb.nvfp4_prefill_plan_check(plan) == nb.NVFP4_OK
    y_ref, absdot = case.oracle_full()
    ok, ratio = within_tolerance(to_f64(y), y_ref, absdot)
    assert ok, ("geometry", _geometry(plan, M), "max |err|/tol = %.3g" % ratio)


def test_geometry_of_the_small_shapes_covers_the_paths():
    """The shapes above reach the paths they are meant to reach."""
    g = [nb.nvfp4_prefill_geometry(N, K, M, 152) for N, K, M in
         [(640, 512, 33), (513, 1280, 257), (1024, 4096, 64), (1024, 8192, 100)]]
    assert g[0]["m_tiles"] > 1 and g[0]["n_tiles"] == 3
    assert g[1]["m_tiles"] * g[1]["bm"] > 257
    assert g[2]["splits"] > 1 and g[3]["splits"] > 1 and g[3]["bm"] > 16


def _sampled(plan, case, M, n_samples=512, seed=0):
    y = _run(plan, case, M)
    torch.cuda.synchronize()
    assert nb.nvfp4_prefill_plan_check(plan) == nb.NVFP4_OK
    rng = np.random.default_rng(seed)
    ms = np.concatenate([rng.integers(0, M, n_samples), [0, M - 1, M - 1, M // 2]])
    ns = np.concatenate([rng.integers(0, case.N, n_samples), [0, case.N - 1, 0, case.N - 1]])
    y_ref, absdot = case.oracle_at(ms, ns)
    ok, ratio = within_tolerance(to_f64(y)[ms, ns], y_ref, absdot)
    assert ok, ("geometry", _geometry(plan, M), "max |err|/tol = %.3g" % ratio)
    return y


@pytest.mark.parametrize("N,K,M", [
    (34816, 512, 160),   # one 160-row activation tile, 136 weight tiles
    (38400, 256, 250),   # two 128-row tiles, 6 rows past M
    (20000, 1024, 200),  # three 80-row tiles, ragged weight tile
])
def test_tall_tiles_sampled(N, K, M):
    case = Case(N, K, M, seed=N + M)
    plan = nb.nvfp4_prefill_plan_create(N, K, M)
    _sampled(plan, case, M, seed=M)


@pytest.mark.parametrize("M", [33, 64, 256, 1024])
def test_square_workload_sampled(M):
    """The square 5120 x 5120 projection at prefill row counts (sampled outputs)."""
    w = synth.WORKLOADS["square"].projections[0]
    case = Case(w.N, w.K, M, seed=w.seed + M, outlier_frac=0.001)
    plan = nb.nvfp4_prefill_plan_create(w.N, w.K, 1024)
    _sampled(plan, case, M, seed=M)


def test_deterministic_and_graph_replay_bit_identical():
    """Two calls, and a CUDA-graph replay of the call, give the same bits."""
    N, K, M = 1024, 4096, 96
    case = Case(N, K, M, seed=5)
    plan = nb.nvfp4_prefill_plan_create(N, K, M)
    y1 = _run(plan, case)
    y2 = _run(plan, case)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    s = torch.cuda.Stream()
    y3 = torch.empty_like(y1)
    with torch.cuda.stream(s):
        nb.nvfp4_prefill_linear(plan, case.d_x, M, case.d_codes, case.d_scales, case.gs, y3, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            nb.nvfp4_prefill_linear(plan, case.d_x, M, case.d_codes, case.d_scales, case.gs, y3, stream=s)
        y3.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))
    assert nb.nvfp4_prefill_plan_check(plan) == nb.NVFP4_OK


def test_rows_of_smaller_calls_match_the_oracle_and_plan_reuse():
    """One plan serves every M up to max_M, calls with different M back to back."""
    N, K = 768, 2048
    case = Case(N, K, 200, seed=11)
    plan = nb.nvfp4_prefill_plan_create(N, K, 200)
    y_ref, absdot = case.oracle_full()
    for M in (200, 1, 37, 128, 200):
        xm = case.d_x[:M].contiguous()
        y = _run(plan, case, M, x=xm)
        torch.cuda.synchronize()
        ok, ratio = within_tolerance(to_f64(y), y_ref[:M], absdot[:M])
        assert ok, (M, ratio)
    assert nb.nvfp4_prefill_plan_check(plan) == nb.NVFP4_OK


def test_argument_errors():
    N, K = 512, 512
    plan = nb.nvfp4_prefill_plan_create(N, K, 64)
    case = Case(N, K, 64, seed=3)
    y = torch.full((64, N), 7.0, dtype=torch.bfloat16, device="cuda")

    def call(x=case.d_x, M=64, codes=case.d_codes, scales=case.d_scales, yy=y):
        return nb.nvfp4_prefill_linear(plan, x, M, codes, scales, 1.0, yy, check=False)

    assert call(M=0) == nb.NVFP4_ERR_M_RANGE
    assert call(M=65) == nb.NVFP4_ERR_M_RANGE
    assert call(x=None) == nb.NVFP4_ERR_ARG
    assert call(codes=case.d_codes.view(-1)[1:]) == nb.NVFP4_ERR_ALIGN
    assert call(yy=y.view(-1)[3:]) == nb.NVFP4_ERR_ALIGN
    torch.cuda.synchronize()
    assert bool((y == 7.0).all()), "a refused call wrote y"
    for bad in [(0, 512, 8), (512, 100, 8), (512, 512, 0), (512, 512, nb.NVFP4_PREFILL_MAX_ROWS + 1)]:
        with pytest.raises(nb.Nvfp4Error):
            nb.nvfp4_prefill_plan_create(*bad)
    info = nb.nvfp4_prefill_plan_get_info(plan, 64)
    assert info["max_M"] == 64 and info["workspace_bytes"] > 0


@pytest.mark.parametrize("bm,splits,k_step", [(32, 1, 64), (32, 3, 128), (64, 8, 64), (64, 1, 128), (96, 5, 64),
                                              (96, 2, 128), (128, 2, 128), (128, 4, 64), (160, 4, 64), (192, 1, 64)])
def test_forced_geometries_every_element(bm, splits, k_step):
    """Every tile height band, split and pipeline step through the explicit-geometry entry point:
    each one is within the tolerance on every element (N = 1024, K = 4096, M = 100)."""
    N, K, M = 1024, 4096, 100
    case = _forced_case()
    plan = nb.nvfp4_prefill_plan_create(N, K, M)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    nb.nvfp4_prefill_linear_ex(plan, case.d_x, M, case.d_codes, case.d_scales, case.gs, y, bm=bm, splits=splits,
                               k_step=k_step)
    torch.cuda.synchronize()
    assert nb.nvfp4_prefill_plan_check(plan) == nb.NVFP4_OK
    y_ref, absdot = _forced_ref()
    ok, ratio = within_tolerance(to_f64(y), y_ref, absdot)
    assert ok, (bm, splits, k_step, "max |err|/tol = %.3g" % ratio)


_FORCED = {}


def _forced_case():
    if "case" not in _FORCED:
        _FORCED["case"] = Case(1024, 4096, 100, seed=77, outlier_frac=0.01)
    return _FORCED["case"]


def _forced_ref():
    if "ref" not in _FORCED:
        _FORCED["ref"] = _forced_case().oracle_full()
    return _FORCED["ref"]


def test_forced_geometry_refusals():
    N, K, M = 512, 512, 40
    plan = nb.nvfp4_prefill_plan_create(N, K, M)
    case = Case(N, K, M, seed=4)
    y = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")

    def call(bm, splits, k_step=0):
        return nb.nvfp4_prefill_linear_ex(plan, case.d_x, M, case.d_codes, case.d_scales, 1.0, y, bm=bm,
                                          splits=splits, k_step=k_step, check=False)

    for bm, splits in [(16, 1), (48, 1), (208, 1), (256, 1), (-32, 1), (32, -1), (32, 3), (32, 33)]:
        assert call(bm, splits) == nb.NVFP4_ERR_ARG, (bm, splits)
    for bm, k_step in [(160, 128), (192, 128), (64, 96), (64, 256), (64, -64)]:
        assert call(bm, 1, k_step) == nb.NVFP4_ERR_ARG, (bm, k_step)
    # a split the plan's part buffer was not sized for
    info = nb.nvfp4_prefill_plan_get_info(plan, M)
    if info["workspace_bytes"] < 2 * M * N * 4:
        assert call(32, 2) == nb.NVFP4_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert bool((y == 3.0).all()), "a refused call wrote y"
