"""The allocation-free entry point, nvfp4_skinny_linear_noalloc, against the plan-based one.

Some callers cannot allocate device memory while they run: code inside another framework's
memory pool, engines that reserve all device memory up front, or paths where a cudaMalloc
would synchronise the device.  For them the library keeps its scratch in one fixed device
array.  This test checks that such calls give the same answer as nvfp4_skinny_linear, within
the tolerance the other GPU tests use, for two calls in a row that share that scratch.  It
sits in a file of its own that pytest collects last.
"""
import numpy as np
import pytest
import torch

import oracle

from gpu_cases import Case, to_f64, within_tolerance
from nvfp4_skinny_gb300 import binding as nb

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from nvfp4_skinny_gb300 import build
    build.build()
    torch.cuda.init()


def _both(case, f32=False):
    out = nb.NVFP4_OUT_F32 if f32 else nb.NVFP4_OUT_BF16
    plan = nb.nvfp4_plan_create_ex(case.N, case.K, out)
    y_plan = case.run(plan)
    y_free = torch.empty_like(y_plan)
    nb.nvfp4_skinny_linear_noalloc(case.N, case.K, out, case.d_x, case.M, case.d_codes, case.d_scales, case.gs,
                                   y_free)
    torch.cuda.synchronize()
    return y_plan, y_free


def _check(case, y_plan, y_free):
    y_ref, absdot = case.oracle_full()
    # the tolerance every GPU test uses, applied between the two entry points ...
    tol = oracle.tolerance(y_ref, absdot)
    assert np.all(np.abs(to_f64(y_free) - to_f64(y_plan)) <= tol)
    # ... and both against the oracle
    assert within_tolerance(to_f64(y_free), y_ref, absdot)[0]


def test_noalloc_matches_plan_entry_two_calls_in_a_row():
    # split row blocks (counters and parts in the shared scratch), then a different shape and M
    first = Case(2048, 8192, 9, seed=21, outlier_frac=0.01)
    second = Case(5120, 5120, 17, seed=2)
    y1_plan, y1_free = _both(first)
    y2_plan, y2_free = _both(second)
    _check(first, y1_plan, y1_free)
    _check(second, y2_plan, y2_free)
    # same kernels and the same work split on a GPU with at most 160 SMs: the same bits
    if torch.cuda.get_device_properties(0).multi_processor_count <= 160:
        assert torch.equal(y1_plan, y1_free) and torch.equal(y2_plan, y2_free)


def test_noalloc_fp32_output():
    case = Case(640, 1024, 3, seed=7)
    y_plan, y_free = _both(case, f32=True)
    _check(case, y_plan, y_free)


def test_noalloc_allocates_nothing_and_reports_no_error():
    """After a first call (the per-device set-up), calls of several shapes leave the device's
    free memory unchanged, and the error word reads clear."""
    cases = [Case(2048, 8192, 9, seed=31), Case(640, 1024, 32, seed=32), Case(5120, 5120, 1, seed=33)]
    ys = [torch.empty((c.M, c.N), dtype=torch.bfloat16, device="cuda") for c in cases]
    c0 = cases[0]
    nb.nvfp4_skinny_linear_noalloc(c0.N, c0.K, nb.NVFP4_OUT_BF16, c0.d_x, c0.M, c0.d_codes, c0.d_scales, c0.gs, ys[0])
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        for c, y in zip(cases, ys):
            nb.nvfp4_skinny_linear_noalloc(c.N, c.K, nb.NVFP4_OUT_BF16, c.d_x, c.M, c.d_codes, c.d_scales, c.gs, y)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    assert nb.nvfp4_noalloc_check() == nb.NVFP4_OK
    for c, y in zip(cases, ys):
        y_ref, absdot = c.oracle_full()
        assert within_tolerance(to_f64(y), y_ref, absdot)[0]


def test_noalloc_refuses_beyond_its_scratch():
    dev = torch.empty(64, dtype=torch.uint8, device="cuda")
    y = torch.empty(64, dtype=torch.uint8, device="cuda")
    call = lambda N, K: nb.nvfp4_skinny_linear_noalloc(N, K, nb.NVFP4_OUT_BF16, dev, 1, dev, dev, 1.0, y,
                                                       check=False)
    assert call(256, nb.NVFP4_NOALLOC_MAX_K + 256) == nb.NVFP4_ERR_SCRATCH_LIMIT
    assert call(nb.NVFP4_NOALLOC_MAX_N + 1, 512) == nb.NVFP4_ERR_SCRATCH_LIMIT
    assert call(256, 300) == nb.NVFP4_ERR_SHAPE
    torch.cuda.synchronize()
