"""Chained tensor-parallel MLP (AllGather+GEMM -> ReLU -> GEMM+ReduceScatter):
CUDA path vs the CPU oracle (GPU).

Integer-valued inputs keep every fp32 sum exact (the hidden activations are
rounded to bf16 the same way on both sides), so the gathered input, the
hidden activations of every rank and the output blocks must match bit for
bit.  Shapes cover shard rows that are not a multiple of 128 (chunks straddle
shards and pairs), widths that are not multiples of 64 (two-box B loads) or
of the 256-column block, one and several ranks, CTA pairs on and off, all
three modes, and the full TP=8 layer on a row sample within tolerance.
"""
import numpy as np
import pytest
import torch

import oracle as O
import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import inputs as I
from parity_util import TOL, absmax, dev, gpu_bits, gpu_values, norm_err, oracle_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from comm_gemm_tile_gb300 import build
    build.build()
    torch.cuda.init()


def _ok(ws=None):
    st, detail = mk.device_status(ws)
    assert st == mk.MK_OK, (mk.status_string(st), detail)


SHAPES = [  # R, m, h, f_r
    (2, 128, 256, 256),
    (4, 200, 264, 520),
    (8, 128, 512, 256),
    (1, 300, 256, 264),
]


def _check(w, cfg=None, pre_gather=False):
    x, w1, w2 = I.mlp_inputs(w)
    want = O.mlp_ag_rs([I.bits(t) for t in x], [I.bits(t) for t in w1], [I.bits(t) for t in w2])
    g = None
    if pre_gather:
        g = torch.from_numpy(want["gathered"].view(np.int16)).view(torch.bfloat16).cuda()
    ws = mk.Workspace()
    xg, hid, y = mk.mlp_ag_rs(dev(x), dev(w1), dev(w2), x_gathered=g, cfg=cfg, workspace=ws)
    _ok(ws)
    np.testing.assert_array_equal(I.bits(xg), want["gathered"])
    for r in range(w.R):
        np.testing.assert_array_equal(I.bits(hid[r]), want["hidden"][r])
        np.testing.assert_array_equal(gpu_bits(y[r]), want["blocks"][r])


@pytest.mark.parametrize("pair", [mk.PAIR_OFF, mk.PAIR_ON])
@pytest.mark.parametrize("R,m,h,f_r", SHAPES)
def test_mlp_integer_bit_exact(R, m, h, f_r, pair):
    w = I.MlpWorkload("t", R=R, m=m, h=h, f_r=f_r, integer=True, x_seed=11, w1_seed=21, w2_seed=31)
    _check(w, mk.Config(cta_pair=pair))


@pytest.mark.parametrize("mode", [mk.MODE_GEMM_ONLY, mk.MODE_UNFUSED])
@pytest.mark.parametrize("pair", [mk.PAIR_OFF, mk.PAIR_ON])
def test_mlp_baseline_modes(mode, pair):
    w = I.MlpWorkload("t", R=4, m=200, h=264, f_r=520, integer=True, x_seed=12, w1_seed=22, w2_seed=32)
    _check(w, mk.Config(mode=mode, cta_pair=pair), pre_gather=(mode == mk.MODE_GEMM_ONLY))


@pytest.mark.parametrize("max_ctas", [2, 5])
def test_mlp_few_ctas(max_ctas):
    # one pair / few CTAs walk both phases: down-projection tiles wait across many items
    w = I.MlpWorkload("t", R=4, m=256, h=256, f_r=512, integer=True, x_seed=13, w1_seed=23, w2_seed=33)
    _check(w, mk.Config(max_ctas=max_ctas))


def test_mlp_float_within_tolerance():
    w = I.MlpWorkload("t", R=4, m=256, h=512, f_r=768, x_seed=14, w1_seed=24, w2_seed=34)
    x, w1, w2 = I.mlp_inputs(w)
    want = O.mlp_ag_rs([I.bits(t) for t in x], [I.bits(t) for t in w1], [I.bits(t) for t in w2])
    ws = mk.Workspace()
    xg, hid, y = mk.mlp_ag_rs(dev(x), dev(w1), dev(w2), workspace=ws)
    _ok(ws)
    hmax = max(float(np.abs(O.bf16_to_f64(hh)).max()) for hh in want["hidden"])
    for r in range(w.R):
        assert norm_err(gpu_values(hid[r]), O.bf16_to_f64(want["hidden"][r]), w.h, absmax(x),
                        absmax(w1)) <= TOL["bf16"]
        exact = O.bf16_to_f64(want["blocks"][r])
        assert norm_err(gpu_values(y[r]), exact, w.R * w.f_r, hmax, absmax(w2)) <= TOL["bf16"]


def test_mlp_full_size_row_sample():
    # 8 ranks, 8192 tokens, h = 8192, f = 8 x 3584 (the TP=8 layer of the AG and RS workloads)
    w = I.MLP_R8_TP8
    x, w1, w2 = I.mlp_inputs(w)
    ws = mk.Workspace()
    xg, hid, y = mk.mlp_ag_rs(dev(x), dev(w1), dev(w2), workspace=ws)
    _ok(ws)
    xb = [I.bits(t) for t in x]
    np.testing.assert_array_equal(I.bits(xg), O.allgather_rows(xb))
    rows = I.sample_rows(w.R * w.m, seed=9, per_tile=1)
    want = O.mlp_ag_rs(xb, [I.bits(t) for t in w1], [I.bits(t) for t in w2], rows=rows)
    sel = torch.from_numpy(rows).cuda()
    hmax = max(float(np.abs(O.bf16_to_f64(hh)).max()) for hh in want["hidden"])
    for r in range(w.R):
        assert norm_err(gpu_values(hid[r][sel]), O.bf16_to_f64(want["hidden"][r]), w.h, absmax(x),
                        absmax(w1)) <= TOL["bf16"]
    got = torch.stack([y[int(i) // w.m][int(i) % w.m] for i in rows], 0)
    assert norm_err(gpu_values(got), O.bf16_to_f64(want["rows"]), w.R * w.f_r, hmax, absmax(w2)) \
        <= TOL["bf16"]
