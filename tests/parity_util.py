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
