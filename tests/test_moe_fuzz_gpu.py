"""MoE dispatch + grouped GEMM over seeded random shapes (GPU).

Every case draws the ranks, experts per rank, tokens, widths, top-k, CTA
pairing and grid size from a fixed seed, runs the fused call on integer-valued
inputs, and checks the routing, counts, dispatch permutation, received rows and
expert outputs bit for bit against the oracle.  Small grids make each copy warp
and compute CTA cover many rows and tiles; top-k above 2 exercises a token's
copy writing all of its slots.
"""
import numpy as np
import pytest
import torch

import oracle as O
import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import inputs as I
from parity_util import gpu_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from comm_gemm_tile_gb300 import build
    build.build()
    torch.cuda.init()


def _case(seed):
    g = np.random.default_rng(seed)
    R = int(g.integers(1, 17))                      # up to 16 ranks
    E_loc = int(g.integers(1, min(6, 256 // R) + 1))
    topk = int(g.integers(1, min(8, R * E_loc) + 1))
    T = int(g.integers(1, 400))
    H = 8 * int(g.integers(1, 40))
    N = 8 * int(g.integers(1, 70))
    pair = [mk.PAIR_OFF, mk.PAIR_ON][int(g.integers(0, 2))]
    max_ctas = [0, 4, 16][int(g.integers(0, 3))]
    return R, E_loc, topk, T, H, N, pair, max_ctas


@pytest.mark.parametrize("seed", list(range(12)))
def test_moe_random_shapes_bit_exact(seed):
    R, E_loc, topk, T, H, N, pair, max_ctas = _case(5000 + seed)
    w = I.MoeWorkload("t", R=R, E_loc=E_loc, T=T, H=H, N=N, topk=topk, integer=True,
                      x_seed=600 + seed, logit_seed=700 + seed, w_seed=800 + seed)
    x, logits, wexp = I.moe_inputs(w)
    ws = mk.Workspace()
    res = mk.moe_dispatch_gemm([t.cuda() for t in x], [t.cuda() for t in logits], [t.cuda() for t in wexp],
                               E_loc=E_loc, topk=topk, cfg=mk.Config(cta_pair=pair, max_ctas=max_ctas),
                               workspace=ws)
    st, detail = mk.device_status(ws)
    assert st == mk.MK_OK, (mk.status_string(st), detail, (R, E_loc, topk, T, H, N, pair, max_ctas))
    idx = [O.moe_route(t.numpy(), topk) for t in logits]
    np.testing.assert_array_equal(res["topk_idx"].cpu().numpy(), np.concatenate(idx, 0))
    np.testing.assert_array_equal(res["counts"].cpu().numpy(), O.moe_counts(idx, w.E))
    recv_src, seg = O.moe_dispatch(idx, E_loc)
    rc = res["recv_counts"].cpu().numpy()
    xb = [I.bits(t) for t in x]
    for d in range(R):
        n = len(recv_src[d])
        assert rc[d] == n
        np.testing.assert_array_equal(res["recv_src"][d][:n].cpu().numpy(), recv_src[d])
        rows = O.moe_gather_rows(xb, recv_src[d], topk)
        np.testing.assert_array_equal(I.bits(res["recv_x"][d][:n]), rows)
        want = O.moe_expert_gemm(rows, seg[d], I.bits(wexp[d]), out="bf16")
        np.testing.assert_array_equal(gpu_bits(res["y"][d][:n]), want)
