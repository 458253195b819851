"""Writes the stored expected values under tests/golden/ from the CPU oracle.

Run from the repository root:  python tests/golden/make_golden.py
Inputs come from the seeded generators; every expected value comes from
``oracle`` alone (never from the CUDA path).
"""
import hashlib
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle as O  # noqa: E402
from comm_gemm_tile_gb300 import inputs as I  # noqa: E402


def sha(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def rs_r2_256_int():
    w = I.RS_R2_256_INT
    a, b = I.gemm_inputs(w)
    blocks = O.gemm_rs([I.bits(x) for x in a], [I.bits(x) for x in b], out="f32")
    return {
        "what": "GEMM+ReduceScatter, R=2, A_r and B_r 256x256 integer-valued bf16 "
                "(U{-2..2}, seeds 1000+r / 2000+r), fp32 out, 2 row blocks of 128x256",
        "cite": "mKernel write-up, news.chathome.org, five-kernel table, row 'GEMM + ReduceScatter'",
        "block_sha256_f32_le": [sha(blk) for blk in blocks],
        "block_sum": [float(blk.astype(np.float64).sum()) for blk in blocks],
        "samples": [[o, i, j, float(blocks[o][i, j])] for o, i, j in
                    [(0, 0, 0), (0, 127, 255), (1, 0, 17), (1, 64, 200), (1, 127, 0)]],
    }


def moe_small_route():
    R, E_loc, T, topk = 4, 4, 256, 2
    logits = [I.zipf_logits(T, R * E_loc, 7000 + r).numpy() for r in range(R)]
    idx = [O.moe_route(lg, topk) for lg in logits]
    counts = O.moe_counts(idx, R * E_loc)
    recv_src, seg = O.moe_dispatch(idx, E_loc)
    return {
        "what": "MoE routing + dispatch permutation, R=4 ranks x 4 experts, T=256 tokens/rank, "
                "top-2, Zipf(1.1) logits with seeds 7000+r",
        "cite": "mKernel write-up, news.chathome.org, five-kernel table, row 'MoE Dispatch + GEMM'",
        "topk_sha256_i32": sha(np.concatenate(idx, 0).astype(np.int32)),
        "counts": counts.tolist(),
        "recv_src_sha256_i32": [sha(s.astype(np.int32)) for s in recv_src],
        "seg": [s.tolist() for s in seg],
    }


def main():
    out = {"rs_r2_256_int": rs_r2_256_int(), "moe_small_route": moe_small_route()}
    with open(os.path.join(HERE, "oracle_golden.json"), "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
