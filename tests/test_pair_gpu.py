"""CTA pairs (GPU): the 256 x 256 tiles computed by two SMs through tcgen05
cta_group::2 against the oracle, with pairs forced on and forced off.

Shapes cover an odd count of 128-row blocks (the second half of the last pair
is empty), a single row block (every pair half-empty: the AllReduce decode
shape), shards that straddle pairs, one and several pairs, both reductions,
the two baseline modes, and the bounded waits of a pair that has to abort.
Integer-valued inputs: every result is exact in fp32, so bits must match.
"""
import numpy as np
import pytest
import torch

import oracle as O
import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import inputs as I
from parity_util import TOL, absmax, dev, gpu_bits, gpu_values, norm_err, oracle_bits

pytestmark = pytest.mark.gpu

PAIRS = [mk.PAIR_OFF, mk.PAIR_ON]


@pytest.fixture(scope="module", autouse=True)
def built():
    from comm_gemm_tile_gb300 import build
    build.build()
    torch.cuda.init()


def _ok(ws=None):
    st, detail = mk.device_status(ws)
    assert st == mk.MK_OK, (mk.status_string(st), detail)


def _ag_check(R, mr, n, k, local, cfg, seed=11):
    w = I.GemmWorkload("t", "ag", R=R, m=mr, n=n, k=k, out="bf16", a_seed=seed, b_seed=seed + 1,
                       integer=True)
    a, b = I.gemm_inputs(w)
    g, c = mk.ag_gemm(dev(a), b[0].cuda(), local_rank=local, cfg=cfg)
    _ok()
    gathered, want = O.ag_gemm([I.bits(x) for x in a], I.bits(b[0]), out="bf16")
    np.testing.assert_array_equal(I.bits(g), gathered)
    np.testing.assert_array_equal(gpu_bits(c), want)


def _rs_check(R, m, n, k, cfg, out="bf16", seed=21):
    w = I.GemmWorkload("t", "rs", R=R, m=m, n=n, k=k, out=out, a_seed=seed, b_seed=seed + 1,
                       integer=True)
    a, b = I.gemm_inputs(w)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    blocks = mk.gemm_rs(dev(a), dev(b), out_dtype=dt, cfg=cfg)
    _ok()
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    np.testing.assert_array_equal(gpu_bits(torch.cat(blocks, 0)), oracle_bits(exact, out))


def _ar_check(R, m, n, k, cfg, seed=31):
    w = I.GemmWorkload("t", "ar", R=R, m=m, n=n, k=k, out="bf16", a_seed=seed, b_seed=seed + 1,
                       integer=True)
    a, b = I.gemm_inputs(w)
    reps = mk.gemm_ar(dev(a), dev(b), cfg=cfg)
    _ok()
    a_bits, b_bits = [I.bits(x) for x in a], [I.bits(x) for x in b]
    if cfg.mode == mk.MODE_GEMM_ONLY:   # the baseline: replica r holds rank r's own product
        for r, part in enumerate(O.rank_partials(a_bits, b_bits)):
            np.testing.assert_array_equal(gpu_bits(reps[r]), oracle_bits(part, "bf16"))
        return
    want = oracle_bits(O.sum_over_ranks(a_bits, b_bits), "bf16")
    for r in reps:
        np.testing.assert_array_equal(gpu_bits(r), want)


@pytest.mark.parametrize("pair", PAIRS)
@pytest.mark.parametrize("R,mr,n,k,local", [
    (1, 300, 256, 64, 0),     # 3 row blocks: the last pair's second half is empty
    (4, 200, 512, 256, 2),    # shards straddle row blocks and pairs
    (4, 384, 264, 520, 1),    # 3 row blocks per shard: pairs straddle shards
    (8, 256, 512, 512, 6),
])
def test_ag_pairs(R, mr, n, k, local, pair):
    _ag_check(R, mr, n, k, local, mk.Config(cta_pair=pair))


@pytest.mark.parametrize("pair", PAIRS)
@pytest.mark.parametrize("R,m,n,k", [
    (4, 520, 520, 200),       # 5 row blocks, ragged n and k
    (2, 384, 264, 136),
    (1, 136, 256, 64),
    (8, 1024, 512, 512),
])
@pytest.mark.parametrize("reduce", [mk.REDUCE_RUNNING_SUM, mk.REDUCE_LAST_ARRIVAL])
def test_rs_pairs(R, m, n, k, reduce, pair):
    _rs_check(R, m, n, k, mk.Config(cta_pair=pair, reduce=reduce))


@pytest.mark.parametrize("pair", PAIRS)
@pytest.mark.parametrize("R,m,n,k,split_k", [
    (8, 128, 1032, 512, 1),   # one row block: every pair's second half is empty
    (8, 128, 1032, 512, 3),
    (4, 200, 512, 264, 1),
])
def test_ar_pairs(R, m, n, k, split_k, pair):
    _ar_check(R, m, n, k, mk.Config(cta_pair=pair, split_k=split_k))


@pytest.mark.parametrize("mode", [mk.MODE_GEMM_ONLY, mk.MODE_UNFUSED])
def test_baseline_modes_with_pairs(mode):
    cfg = mk.Config(mode=mode, cta_pair=mk.PAIR_ON)
    _rs_check(4, 640, 512, 256, cfg)
    _ar_check(2, 384, 264, 136, cfg)
    if mode == mk.MODE_UNFUSED:
        _ag_check(4, 128, 512, 256, 1, cfg)


@pytest.mark.parametrize("max_ctas", [2, 3, 6])
def test_few_pairs(max_ctas):
    # one or a few pairs walk the whole item list; chains wait across rounds
    cfg = mk.Config(cta_pair=mk.PAIR_ON, max_ctas=max_ctas)
    _rs_check(4, 512, 512, 256, cfg, out="f32")
    _ag_check(4, 256, 512, 256, 3, cfg)


def test_pairs_match_single_cta_float():
    R, m, n, k = 4, 512, 776, 1032
    w = I.GemmWorkload("t", "rs", R=R, m=m, n=n, k=k, out="f32", a_seed=41, b_seed=42)
    a, b = I.gemm_inputs(w)
    da, db = dev(a), dev(b)
    x = mk.gemm_rs(da, db, out_dtype=torch.float32, cfg=mk.Config(cta_pair=mk.PAIR_OFF))
    y = mk.gemm_rs(da, db, out_dtype=torch.float32, cfg=mk.Config(cta_pair=mk.PAIR_ON))
    _ok()
    exact = O.sum_over_ranks([I.bits(t) for t in a], [I.bits(t) for t in b])
    for got in (x, y):
        assert norm_err(gpu_values(torch.cat(got, 0)), exact, R * k, absmax(a), absmax(b)) <= TOL["f32"]


def test_pair_abort_on_missing_copy_piece():
    R, mr, n, k = 4, 256, 512, 256
    w = I.GemmWorkload("t", "ag", R=R, m=mr, n=n, k=k, out="bf16", a_seed=1, b_seed=2, integer=True)
    a, b = I.gemm_inputs(w)
    ws = mk.Workspace()
    mk.ag_gemm(dev(a), b[0].cuda(), workspace=ws,
               cfg=mk.Config(inject=1, wait_limit_ns=20_000_000, cta_pair=mk.PAIR_ON))
    st, _ = mk.device_status(ws)
    assert st == mk.MK_ERR_TIMEOUT
    g, c = mk.ag_gemm(dev(a), b[0].cuda(), workspace=ws, cfg=mk.Config(cta_pair=mk.PAIR_ON))
    _ok(ws)
    _, want = O.ag_gemm([I.bits(x) for x in a], I.bits(b[0]), out="bf16")
    np.testing.assert_array_equal(gpu_bits(c), want)


@pytest.mark.parametrize("reduce", [mk.REDUCE_RUNNING_SUM, mk.REDUCE_LAST_ARRIVAL])
def test_pair_abort_on_missing_partial(reduce):
    R, m, n, k = 2, 512, 512, 128
    w = I.GemmWorkload("t", "rs", R=R, m=m, n=n, k=k, out="bf16", a_seed=3, b_seed=4, integer=True)
    a, b = I.gemm_inputs(w)
    ws = mk.Workspace()
    mk.gemm_rs(dev(a), dev(b), workspace=ws,
               cfg=mk.Config(inject=2, wait_limit_ns=20_000_000, cta_pair=mk.PAIR_ON, reduce=reduce))
    st, _ = mk.device_status(ws)
    if reduce == mk.REDUCE_RUNNING_SUM:
        assert st == mk.MK_ERR_TIMEOUT
    blocks = mk.gemm_rs(dev(a), dev(b), workspace=ws, cfg=mk.Config(cta_pair=mk.PAIR_ON))
    _ok(ws)
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    np.testing.assert_array_equal(gpu_bits(torch.cat(blocks, 0)), oracle_bits(exact, "bf16"))


@pytest.mark.parametrize("max_ctas", [2, 4])
@pytest.mark.parametrize("reduce", [mk.REDUCE_RUNNING_SUM, mk.REDUCE_LAST_ARRIVAL])
def test_few_pairs_odd_row_blocks(max_ctas, reduce):
    # 5 row blocks: every pass over the last pair row has an empty half, and a
    # pair goes on to later items after it (the per-buffer publish barrier
    # must keep its own phase across items that publish nothing)
    cfg = mk.Config(cta_pair=mk.PAIR_ON, max_ctas=max_ctas, reduce=reduce)
    _rs_check(4, 640, 520, 256, cfg)
    _ar_check(2, 640, 264, 136, cfg)
