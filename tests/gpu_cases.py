"""Helpers shared by the GPU tests: seeded inputs on both sides, one call through the
C ABI, and the element-wise acceptance check against the CPU oracle."""
import numpy as np
import torch

import oracle
from nvfp4_skinny_gb300 import binding as nb
from nvfp4_skinny_gb300 import synth


def bf16_bits(t):
    """bfloat16 torch tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Case:
    """One seeded weight + activation set, resident on the CPU (for the oracle) and the GPU."""

    def __init__(self, N, K, M, seed, outlier_frac=0.0, x=None, codes=None, scales=None, gs=None):
        if codes is None:
            codes, scales, gs0 = synth.weights(N, K, seed)
            gs = gs0 if gs is None else gs
        if x is None:
            x = synth.activations(M, K, seed, outlier_frac=outlier_frac)
        self.N, self.K, self.M, self.gs = N, K, M, float(np.float32(gs))
        self.codes, self.scales, self.x = codes, scales, x
        self.codes_np = codes.numpy()
        self.scales_np = scales.numpy()
        self.x_bits = bf16_bits(x)
        self.d_codes = codes.cuda()
        self.d_scales = scales.cuda()
        self.d_x = x.cuda()

    def run(self, plan, M=None, x=None, stream=None):
        M = self.M if M is None else M
        dx = self.d_x if x is None else x
        dtype = torch.float32 if plan.out_dtype == nb.NVFP4_OUT_F32 else torch.bfloat16
        y = torch.empty((M, self.N), dtype=dtype, device="cuda")
        nb.nvfp4_skinny_linear(plan, dx, M, self.d_codes, self.d_scales, self.gs, y, stream=stream)
        return y

    def oracle_full(self):
        return oracle.linear(self.x_bits, self.codes_np, self.scales_np, self.gs)

    def oracle_at(self, ms, ns):
        return oracle.linear_at(self.x_bits, self.codes_np, self.scales_np, self.gs, ms, ns)


def within_tolerance(y_gpu, y_ref, absdot):
    """|y - y_ref| <= 4e-3 * sum|w x| + ulp_bf16(|y_ref|), element-wise.  Returns (ok, worst ratio)."""
    y = np.asarray(y_gpu, np.float64)
    tol = oracle.tolerance(y_ref, absdot)
    err = np.abs(y - y_ref)
    ok = bool(np.all(err <= tol)) and bool(np.all(np.isfinite(y)))
    ratio = float(np.max(err / tol)) if err.size else 0.0
    return ok, ratio


def to_f64(y):
    return y.float().cpu().numpy().astype(np.float64)
