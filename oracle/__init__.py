"""CPU oracle -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The product path never does.
"""
from .mk_oracle import *  # noqa: F401,F403
from .mk_oracle import (ag_gemm, allgather_rows, bf16_to_f64, f64_to_bf16_bits, gemm_ar,  # noqa
                        gemm_rs, mlp_ag_rs, mlp_hidden, moe_combine, moe_counts, moe_dispatch, moe_dispatch_gemm,
                        moe_expert_gemm, moe_gather_rows, moe_return_rows, moe_route,
                        moe_seg_from_counts, moe_weighted_sum, norm_scale, owner_rows,
                        ring_attention, ring_order, round_out, sum_over_ranks, rank_partials,
                        running_sum_bf16_wire, f64_to_f32, e4m3_to_f64, ag_gemm_fp8,
                        sum_over_ranks_fp8)
