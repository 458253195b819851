"""Seeded synthetic inputs for the fused collective + GEMM ops.

This module only draws random numbers and packs them as bf16; it holds none of
the arithmetic of the ops themselves, so both the CUDA path and the CPU oracle
can be fed from it.  Everything is CPU-side (numpy PCG64 + torch CPU for the
fp32 -> bf16 round-to-nearest-even packing).

Workload shapes follow the five fused kernels listed in the mKernel write-up
(news.chathome.org, "五种融合内核" table): AllGather+GEMM, GEMM+ReduceScatter,
GEMM+AllReduce and MoE Dispatch+GEMM, sized like tensor-parallel (TP=8) MLP and
MoE layers of an LLM.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """fp32 samples -> bf16 tensor (round to nearest even, done by torch)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> its raw uint16 bit patterns (what the oracle consumes)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def normal_bf16(shape, std: float, seed: int) -> torch.Tensor:
    x = rng(seed).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return to_bf16(x)


def int_bf16(shape, seed: int, lo: int = -2, hi: int = 2) -> torch.Tensor:
    """Integers uniform in [lo, hi]: exact in bf16, so every fp32 sum of their
    products stays exact while |sum| < 2**24."""
    x = rng(seed).integers(lo, hi + 1, size=shape, dtype=np.int32).astype(np.float32)
    return to_bf16(x)


def normal_fp8(shape, std: float, seed: int) -> torch.Tensor:
    """N(0, std) samples converted by torch to fp8 e4m3 (CPU tensor)."""
    x = rng(seed).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return torch.from_numpy(x).to(torch.float8_e4m3fn)


def int_fp8(shape, seed: int, lo: int = -2, hi: int = 2) -> torch.Tensor:
    """Integers uniform in [lo, hi] as fp8 e4m3 (exact for |x| <= 16)."""
    x = rng(seed).integers(lo, hi + 1, size=shape, dtype=np.int32).astype(np.float32)
    return torch.from_numpy(x).to(torch.float8_e4m3fn)


def fp8_bytes(t: torch.Tensor) -> np.ndarray:
    """Raw bytes of an fp8 tensor (any device) as a uint8 array."""
    return t.detach().cpu().view(torch.uint8).numpy()


def zipf_logits(tokens: int, experts: int, seed: int, s: float = 1.1) -> torch.Tensor:
    """Router logits whose top-k picks expert e with popularity ~ (e+1)^-s.

    logits[t, e] = ln p_e + Gumbel(0, 1); the top-k of these is a draw of k
    distinct experts without replacement, proportional to p (Gumbel-top-k).
    Expert 0 is the most popular (identity popularity ranking).
    """
    e = np.arange(experts, dtype=np.float64)
    p = (e + 1.0) ** (-s)
    p /= p.sum()
    u = rng(seed).random(size=(tokens, experts))
    u = np.clip(u, np.finfo(np.float64).tiny, 1.0 - 1e-16)
    g = -np.log(-np.log(u))
    return torch.from_numpy((np.log(p)[None, :] + g).astype(np.float32))


# --------------------------------------------------------------------------
# Workload definitions (shapes, distributions, seeds)
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class GemmWorkload:
    name: str
    op: str              # "ag", "rs", "ar"
    R: int               # virtual ranks
    m: int               # rows of A per rank (AG: shard rows m_r)
    n: int
    k: int
    out: str             # "bf16" | "f32"
    a_std: float = 1.0
    b_std: float = 0.02
    a_seed: int = 0
    b_seed: int = 0
    integer: bool = False
    local_rank: int = 0

    def flops(self) -> float:
        if self.op == "ag":
            return 2.0 * self.R * self.m * self.n * self.k
        return 2.0 * self.R * self.m * self.n * self.k

    def integer_twin(self) -> "GemmWorkload":
        return dataclasses.replace(self, name=self.name + "_int", integer=True,
                                   a_seed=self.a_seed + 50000, b_seed=self.b_seed + 50000)

    def scaled(self, m: int | None = None, n: int | None = None, k: int | None = None,
               R: int | None = None) -> "GemmWorkload":
        return dataclasses.replace(self, name=self.name + "_small", m=m or self.m, n=n or self.n,
                                   k=k or self.k, R=R or self.R)


@dataclasses.dataclass(frozen=True)
class MoeWorkload:
    name: str
    R: int
    E_loc: int
    T: int               # tokens per rank
    H: int               # hidden (contraction)
    N: int               # expert up-proj width
    topk: int = 2
    zipf_s: float = 1.1
    x_seed: int = 1700
    logit_seed: int = 1800
    w_seed: int = 1900
    integer: bool = False
    cap_rows: int = 0    # 0 -> R*T*topk (every row could land on one rank)

    @property
    def E(self) -> int:
        return self.R * self.E_loc

    @property
    def cap(self) -> int:
        return self.cap_rows or self.R * self.T * self.topk

    def flops(self) -> float:
        return 2.0 * self.R * self.T * self.topk * self.H * self.N

    def integer_twin(self) -> "MoeWorkload":
        return dataclasses.replace(self, name=self.name + "_int", integer=True,
                                   x_seed=self.x_seed + 50000, w_seed=self.w_seed + 50000)


@dataclasses.dataclass(frozen=True)
class MoeCombineWorkload:
    """MoE combine: the expert hidden rows h[d] ([cap x N], in dispatch order,
    routed by the same Zipf logits as the dispatch), the down-projection
    W2[d] ([E_loc x N x H]) and the gate weights gates[r] ([T x topk] fp32)."""
    name: str
    R: int
    E_loc: int
    T: int               # tokens per rank
    H: int               # model width (output)
    N: int               # expert width (contraction)
    topk: int = 2
    zipf_s: float = 1.1
    logit_seed: int = 1800
    h_seed: int = 2100
    w2_seed: int = 2200
    gate_seed: int = 2300
    integer: bool = False
    cap_rows: int = 0

    @property
    def E(self) -> int:
        return self.R * self.E_loc

    @property
    def cap(self) -> int:
        return self.cap_rows or self.R * self.T * self.topk

    def flops(self) -> float:
        return 2.0 * self.R * self.T * self.topk * self.N * self.H

    def integer_twin(self) -> "MoeCombineWorkload":
        return dataclasses.replace(self, name=self.name + "_int", integer=True,
                                   h_seed=self.h_seed + 50000, w2_seed=self.w2_seed + 50000,
                                   gate_seed=self.gate_seed + 50000)


@dataclasses.dataclass(frozen=True)
class MlpWorkload:
    """Tensor-parallel MLP layer: x shards [m x h] per rank, W1_r [h x f_r]
    (column shard of the up-projection), W2_r [f_r x h] (row shard of the
    down-projection)."""
    name: str
    R: int
    m: int               # rows per shard
    h: int               # model width
    f_r: int             # hidden width per rank
    x_seed: int = 2500
    w1_seed: int = 2600
    w2_seed: int = 2700
    w_std: float = 0.02
    integer: bool = False

    def flops(self) -> float:
        M = self.R * self.m
        return 2.0 * M * self.h * self.f_r * self.R * 2

    def integer_twin(self) -> "MlpWorkload":
        return dataclasses.replace(self, name=self.name + "_int", integer=True,
                                   x_seed=self.x_seed + 50000, w1_seed=self.w1_seed + 50000,
                                   w2_seed=self.w2_seed + 50000)


def mlp_inputs(w: MlpWorkload):
    """x[r] (m x h), w1[r] (h x f_r), w2[r] (f_r x h), all bf16."""
    def draw(shape, std, seed):
        return int_bf16(shape, seed) if w.integer else normal_bf16(shape, std, seed)

    x = [draw((w.m, w.h), 1.0, w.x_seed + r) for r in range(w.R)]
    w1 = [draw((w.h, w.f_r), w.w_std, w.w1_seed + r) for r in range(w.R)]
    w2 = [draw((w.f_r, w.h), w.w_std, w.w2_seed + r) for r in range(w.R)]
    return x, w1, w2


@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    """Ring attention: every rank holds a contiguous block of s_r positions of
    the sequence, q/k/v per rank [heads x s_r x d]."""
    name: str
    R: int
    heads: int
    s_r: int
    d: int = 128
    causal: bool = False
    q_seed: int = 2800
    k_seed: int = 2900
    v_seed: int = 3000
    integer: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def flops(self) -> float:
        S = self.R * self.s_r
        full = 4.0 * self.heads * S * S * self.d
        return full / 2 if self.causal else full


def attn_inputs(w: AttnWorkload):
    """q[r], k[r], v[r]: [heads x s_r x d] bf16 (N(0,1), or integers in {-2..2})."""
    def draw(shape, seed):
        return int_bf16(shape, seed) if w.integer else normal_bf16(shape, 1.0, seed)

    shape = (w.heads, w.s_r, w.d)
    q = [draw(shape, w.q_seed + r) for r in range(w.R)]
    k = [draw(shape, w.k_seed + r) for r in range(w.R)]
    v = [draw(shape, w.v_seed + r) for r in range(w.R)]
    return q, k, v


# The five workloads: a tiny bit-exact GEMM+RS, then TP=8 MLP up-proj (AG),
# down-proj (RS), a decode-shaped AR and a 64-expert top-2 MoE layer.
RS_R2_256_INT = GemmWorkload("rs_r2_256_int", "rs", R=2, m=256, n=256, k=256, out="f32",
                             a_seed=1000, b_seed=2000, integer=True)
AG_R8_TP8_UP = GemmWorkload("ag_r8_m1024x8_k8192_n3584", "ag", R=8, m=1024, n=3584, k=8192,
                            out="bf16", a_seed=1100, b_seed=1200)
RS_R8_TP8_DOWN = GemmWorkload("rs_r8_m8192_k3584_n8192", "rs", R=8, m=8192, n=8192, k=3584,
                              out="bf16", a_seed=1300, b_seed=1400)
AR_R8_DECODE = GemmWorkload("ar_r8_m128_k3584_n8192", "ar", R=8, m=128, n=8192, k=3584,
                            out="bf16", a_seed=1500, b_seed=1600)
MOE_R8_E64 = MoeWorkload("moe_r8x8e_t4096_h4096_n1536", R=8, E_loc=8, T=4096, H=4096, N=1536)
# The combine that follows it: down-projection 1536 -> 4096 and the top-2 weighted sum.
MOE_COMBINE_R8_E64 = MoeCombineWorkload("moe_combine_r8x8e_t4096_n1536_h4096", R=8, E_loc=8,
                                        T=4096, H=4096, N=1536)

# The whole TP=8 MLP layer those two GEMMs belong to, as one chained kernel.
MLP_R8_TP8 = MlpWorkload("mlp_r8_m1024x8_h8192_f3584x8", R=8, m=1024, h=8192, f_r=3584)

# Ring attention over 8 ranks x 4096 positions (32768 in all), 8 heads of 128.
RING_R8_H8_S4096 = AttnWorkload("ring_r8_h8_s4096x8_d128", R=8, heads=8, s_r=4096, d=128)
RING_R8_H8_S4096_CAUSAL = AttnWorkload("ring_r8_h8_s4096x8_d128_causal", R=8, heads=8, s_r=4096,
                                       d=128, causal=True)

WORKLOADS = {w.name: w for w in (RS_R2_256_INT, AG_R8_TP8_UP, RS_R8_TP8_DOWN, AR_R8_DECODE,
                                 MOE_R8_E64, MOE_COMBINE_R8_E64, MLP_R8_TP8, RING_R8_H8_S4096,
                                 RING_R8_H8_S4096_CAUSAL)}


def gemm_inputs(w: GemmWorkload):
    """Per-rank operands as bf16 CPU tensors.

    AG: a = [A_r (m x k)] * R, b = [B (k x n)] (one B, seed b_seed).
    RS/AR: a = [A_r (m x k)] * R, b = [B_r (k x n)] * R.
    """
    def draw(shape, std, seed):
        return int_bf16(shape, seed) if w.integer else normal_bf16(shape, std, seed)

    a = [draw((w.m, w.k), w.a_std, w.a_seed + r) for r in range(w.R)]
    if w.op == "ag":
        b = [draw((w.k, w.n), w.b_std, w.b_seed)]
    else:
        b = [draw((w.k, w.n), w.b_std, w.b_seed + r) for r in range(w.R)]
    return a, b


def gemm_inputs_fp8(w: GemmWorkload):
    """Per-rank fp8 e4m3 operands (CPU tensors) of an AG / RS / AR workload,
    B given as its transpose: a = [A_r (m x k)], b = [B^T (n x k)] (AG: one)."""
    def draw(shape, std, seed):
        return int_fp8(shape, seed) if w.integer else normal_fp8(shape, std, seed)

    a = [draw((w.m, w.k), w.a_std, w.a_seed + r) for r in range(w.R)]
    if w.op == "ag":
        b = [draw((w.n, w.k), w.b_std, w.b_seed)]
    else:
        b = [draw((w.n, w.k), w.b_std, w.b_seed + r) for r in range(w.R)]
    return a, b


def moe_inputs(w: MoeWorkload):
    """x[r] (T x H) bf16, logits[r] (T x E) fp32, wexp[d] (E_loc x H x N) bf16."""
    def draw(shape, std, seed):
        return int_bf16(shape, seed) if w.integer else normal_bf16(shape, std, seed)

    x = [draw((w.T, w.H), 1.0, w.x_seed + r) for r in range(w.R)]
    logits = [zipf_logits(w.T, w.E, w.logit_seed + r, w.zipf_s) for r in range(w.R)]
    wexp = []
    for d in range(w.R):
        per = [draw((w.H, w.N), 0.02, w.w_seed + d * w.E_loc + l) for l in range(w.E_loc)]
        wexp.append(torch.stack(per, 0))
    return x, logits, wexp


def combine_inputs(w: MoeCombineWorkload):
    """logits[r] (T x E) fp32 (the routing), h[d] (cap x N) bf16, w2[d]
    (E_loc x N x H) bf16, gates[r] (T x topk) fp32.  Float gates are uniform
    in [0.05, 1) scaled to sum to 1 per token; integer-twin gates are drawn from
    {0.25, 0.5, 0.75, 1} so that every weighted sum is exact in fp32."""
    def draw(shape, std, seed):
        return int_bf16(shape, seed) if w.integer else normal_bf16(shape, std, seed)

    logits = [zipf_logits(w.T, w.E, w.logit_seed + r, w.zipf_s) for r in range(w.R)]
    h = [draw((w.cap, w.N), 1.0, w.h_seed + d) for d in range(w.R)]
    w2 = []
    for d in range(w.R):
        per = [draw((w.N, w.H), 0.02, w.w2_seed + d * w.E_loc + l) for l in range(w.E_loc)]
        w2.append(torch.stack(per, 0))
    gates = []
    for r in range(w.R):
        g = rng(w.gate_seed + r)
        if w.integer:
            v = g.choice(np.array([0.25, 0.5, 0.75, 1.0], dtype=np.float32), size=(w.T, w.topk))
        else:
            u = g.uniform(0.05, 1.0, size=(w.T, w.topk)).astype(np.float32)
            v = u / u.sum(axis=1, keepdims=True, dtype=np.float32)
        gates.append(torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)))
    return logits, h, w2, gates


def sample_rows(M: int, seed: int, per_tile: int = 2, tile: int = 128) -> np.ndarray:
    """A seeded row sample hitting every `tile`-row block `per_tile` times
    (plus the first and last row), sorted and unique."""
    g = rng(seed)
    rows = [0, M - 1]
    for t0 in range(0, M, tile):
        hi = min(t0 + tile, M)
        rows.extend(g.integers(t0, hi, size=per_tile).tolist())
    return np.unique(np.asarray(rows, dtype=np.int64))


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("math", "np", "torch",
                                                                  "dataclasses")]
