"""Helpers shared by the GPU parity tests: device transfer, and the error
measure of the float parity bar (max |gpu - exact| normalised by
sqrt(K) * max|a| * max|b|, K = contraction length of the result)."""
import numpy as np
import torch

import oracle as O
from comm_gemm_tile_gb300 import inputs as I

TOL = {"bf16": 2e-2, "f32": 1e-3}


def dev(ts):
    return [t.cuda() for t in ts]


def gpu_values(t: torch.Tensor) -> np.ndarray:
    """Device output -> float64 values (bf16 via its exact bits)."""
    if t.dtype == torch.bfloat16:
        return O.bf16_to_f64(I.bits(t))
    return t.detach().cpu().numpy().astype(np.float64)


def gpu_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return I.bits(t)
    return t.detach().cpu().numpy().view(np.uint32)


def absmax(ts) -> float:
    return max(float(t.float().abs().max()) for t in ts)


def norm_err(got: np.ndarray, exact: np.ndarray, K: int, amax: float, bmax: float) -> float:
    scale = O.norm_scale(K, amax, bmax)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - exact)) / scale) if scale > 0 else float(np.max(np.abs(got - exact)))


def oracle_bits(exact: np.ndarray, out: str) -> np.ndarray:
    r = O.round_out(exact, out)
    return r if out == "bf16" else r.view(np.uint32)


def bf16_ulps(got_bits: np.ndarray, want_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 units in the last place between two arrays of bf16 bit
    patterns (finite values): the bit patterns mapped to a monotone integer
    line (negative values mirrored below zero) and subtracted."""
    def line(b):
        b = np.asarray(b, dtype=np.uint16).astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(line(got_bits) - line(want_bits))


def check_bf16_ulps(got_bits: np.ndarray, exact: np.ndarray, floor_frac: float = 2.0 ** -6,
                    max_ulps: int = 2) -> int:
    """Diagnostic beside the normalised bar for bf16 outputs: distance in bf16
    ulps between the GPU bits and the oracle's one rounding of the exact
    result.  Asserted (<= max_ulps) where |exact| is at least floor_frac of
    max|exact|, since near zero the fp32 accumulation error of a long sum can
    exceed the bf16 spacing of a cancelled value.  Returns the largest
    distance seen anywhere (reported, not asserted)."""
    want = O.f64_to_bf16_bits(exact)
    d = bf16_ulps(got_bits, want)
    if d.size == 0:
        return 0
    big = np.abs(exact) >= floor_frac * float(np.max(np.abs(exact)))
    worst = int(d[big].max()) if big.any() else 0
    assert worst <= max_ulps, f"{worst} bf16 ulps from the oracle above the floor"
    return int(d.max())
