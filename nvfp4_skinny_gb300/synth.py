"""Seeded synthetic inputs for the NVFP4 skinny projection.

This module draws random numbers and casts them with torch's own dtype
conversions.  It holds none of the projection's arithmetic (no E2M1 or E4M3
decoding, no dot products), so the oracle and the CUDA path can both consume
what it produces.

Recipe (the same on every device; only the random stream differs between a
CPU and a CUDA generator):
  * E2M1 codes: independent uniform bytes.  Each byte holds two codes (low
    nibble = even k), so every code is uniform over all 16 values.
  * E4M3 block scales, one per 16 elements along K: u ~ U[-4, 2) in fp32,
    s = 2**u, rounded to E4M3 by torch's float8_e4m3fn cast (round to
    nearest even).  Every value lands in [1/16, 4].
  * Per-tensor scale: a fixed fp32 value (0.01 by default).
  * Activations: x ~ N(0, 1) in fp32; optionally each entry independently,
    with probability `outlier_frac`, is multiplied by `outlier_scale` in fp32;
    then cast to bfloat16 (round to nearest even).
"""
from dataclasses import dataclass, field
from typing import List, Tuple

import torch

DEFAULT_GLOBAL_SCALE = 0.01
_X_SEED_OFFSET = 100003


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def weights(N: int, K: int, seed: int, device="cpu", global_scale: float = DEFAULT_GLOBAL_SCALE):
    """Random NVFP4 weight [N, K]: (codes uint8 [N, K/2], scales uint8 [N, K/16], gs float)."""
    if K % 16 != 0:
        raise ValueError("K must be a multiple of 16")
    g = _gen(seed, device)
    codes = torch.randint(0, 256, (N, K // 2), generator=g, dtype=torch.uint8, device=device)
    u = torch.rand((N, K // 16), generator=g, dtype=torch.float32, device=device) * 6.0 - 4.0
    scales = torch.exp2(u).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scales, float(global_scale)


def activations(M: int, K: int, seed: int, device="cpu", outlier_frac: float = 0.0,
                outlier_scale: float = 30.0) -> torch.Tensor:
    """Random bfloat16 activations [M, K] ~ N(0, 1), with optional sparse outliers."""
    g = _gen(int(seed) + _X_SEED_OFFSET, device)
    x = torch.randn((M, K), generator=g, dtype=torch.float32, device=device)
    if outlier_frac > 0.0:
        hit = torch.rand((M, K), generator=g, dtype=torch.float32, device=device) < outlier_frac
        x = torch.where(hit, x * float(outlier_scale), x)
    return x.to(torch.bfloat16)


@dataclass(frozen=True)
class Projection:
    """One weight shape of a workload."""
    name: str
    N: int
    K: int
    seed: int
    f32_out: bool = False


@dataclass(frozen=True)
class Workload:
    """A named synthetic workload: projections, row counts and activation recipe."""
    name: str
    projections: Tuple[Projection, ...]
    Ms: Tuple[int, ...]
    outlier_frac: float = 0.0
    layers: int = 1


def _round_projections() -> Tuple[Projection, ...]:
    out: List[Projection] = []
    shapes = (("qkv", 7168, 5120), ("o", 5120, 5120), ("gate_up", 34816, 5120), ("down", 5120, 17408))
    for layer in range(64):
        for p, (nm, N, K) in enumerate(shapes):
            out.append(Projection("L%d.%s" % (layer, nm), N, K, 1000 + 4 * layer + p))
    return tuple(out)


WORKLOADS = {
    "tiny": Workload("tiny", (Projection("tiny", 256, 512, 1),), (1,)),
    "square": Workload("square", (Projection("square", 5120, 5120, 2),), (1, 2, 4, 8, 16, 17, 24, 32)),
    "qkv_down": Workload("qkv_down", (Projection("qkv", 7168, 5120, 3), Projection("down", 5120, 17408, 4)),
                         (1, 8, 16, 32), outlier_frac=0.01),
    "wide_head": Workload("wide_head", (Projection("gate_up", 34816, 5120, 5),
                                        Projection("head", 152064, 5120, 6, f32_out=True)), (1, 16, 32)),
    "round": Workload("round", _round_projections(), (1, 16, 32), layers=64),
}
