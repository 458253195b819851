"""CUDA path vs the CPU oracle (GPU).

Small shapes span several 128x256 tiles with ragged edges in every dimension
and are compared element by element; integer-valued twins (exact fp32 sums)
must match bit for bit, float inputs within the normalised tolerance.
"""
import hashlib
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import inputs as I
from parity_util import TOL, absmax, dev, gpu_bits, gpu_values, norm_err, oracle_bits

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def built():
    from comm_gemm_tile_gb300 import build
    build.build()
    torch.cuda.init()


def _ok():
    st, detail = mk.device_status()
    assert st == mk.MK_OK, (mk.status_string(st), detail)


# ------------------------------------------------------------------ GEMM + ReduceScatter

def test_rs_tiny_integer_bit_exact_vs_golden():
    w = I.RS_R2_256_INT
    a, b = I.gemm_inputs(w)
    blocks = mk.gemm_rs(dev(a), dev(b), out_dtype=torch.float32)
    _ok()
    gold = json.load(open(os.path.join(HERE, "golden", "oracle_golden.json")))["rs_r2_256_int"]
    for o, blk in enumerate(blocks):
        got = blk.cpu().numpy()
        assert hashlib.sha256(got.tobytes()).hexdigest() == gold["block_sha256_f32_le"][o]
    want = O.gemm_rs([I.bits(x) for x in a], [I.bits(x) for x in b], out="f32")
    for o in range(2):
        np.testing.assert_array_equal(blocks[o].cpu().numpy(), want[o])


RS_SHAPES = [  # R, m, n, k   (ragged rows, cols and K)
    (4, 520, 520, 200),
    (2, 384, 264, 136),
    (8, 1024, 512, 512),
    (1, 136, 256, 64),
]


@pytest.mark.parametrize("R,m,n,k", RS_SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_rs_integer_bit_exact(R, m, n, k, out):
    w = I.GemmWorkload("t", "rs", R=R, m=m, n=n, k=k, out=out, a_seed=31, b_seed=41, integer=True)
    a, b = I.gemm_inputs(w)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    blocks = mk.gemm_rs(dev(a), dev(b), out_dtype=dt)
    _ok()
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    h = m // R
    for o in range(R):
        np.testing.assert_array_equal(gpu_bits(blocks[o]), oracle_bits(exact[o * h:(o + 1) * h], out))


@pytest.mark.parametrize("R,m,n,k", RS_SHAPES)
def test_rs_float_within_tolerance(R, m, n, k):
    w = I.GemmWorkload("t", "rs", R=R, m=m, n=n, k=k, out="bf16", a_seed=51, b_seed=61)
    a, b = I.gemm_inputs(w)
    blocks = mk.gemm_rs(dev(a), dev(b), out_dtype=torch.bfloat16)
    _ok()
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    got = np.concatenate([gpu_values(x) for x in blocks], 0)
    assert norm_err(got, exact, R * k, absmax(a), absmax(b)) <= TOL["bf16"]
    # a sharper diagnostic than the normalised bar: relative error against the exact sum
    assert np.max(np.abs(got - exact) / (np.abs(exact) + 1e-2)) < 0.05


@pytest.mark.parametrize("R,m,n,k", RS_SHAPES[:3])
@pytest.mark.parametrize("n_red", [1, 3, 8])
def test_rs_reduce_role_integer_bit_exact(R, m, n, k, n_red):
    # Staged partials summed by dedicated reduce-role CTAs.
    w = I.GemmWorkload("t", "rs", R=R, m=m, n=n, k=k, out="bf16", a_seed=33, b_seed=43, integer=True)
    a, b = I.gemm_inputs(w)
    blocks = mk.gemm_rs(dev(a), dev(b), cfg=mk.Config(n_reduce_ctas=n_red))
    _ok()
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    np.testing.assert_array_equal(gpu_bits(torch.cat(blocks, 0)), oracle_bits(exact, "bf16"))


def test_rs_reduce_role_matches_running_sum_bits():
    # Both reductions add the partials in rank order 0..R-1: identical float bits.
    R, m, n, k = 4, 520, 520, 200
    w = I.GemmWorkload("t", "rs", R=R, m=m, n=n, k=k, out="f32", a_seed=53, b_seed=63)
    a, b = I.gemm_inputs(w)
    da, db = dev(a), dev(b)
    x = mk.gemm_rs(da, db, out_dtype=torch.float32)
    y = mk.gemm_rs(da, db, out_dtype=torch.float32, cfg=mk.Config(n_reduce_ctas=4))
    z = mk.gemm_rs(da, db, out_dtype=torch.float32, cfg=mk.Config(max_ctas=7))   # cross-CTA chains
    u = mk.gemm_rs(da, db, out_dtype=torch.float32, cfg=mk.Config(reduce=mk.REDUCE_LAST_ARRIVAL))
    v = mk.gemm_rs(da, db, out_dtype=torch.float32,
                   cfg=mk.Config(reduce=mk.REDUCE_LAST_ARRIVAL, max_ctas=5))
    _ok()
    for o in range(R):
        for other in (y, z, u, v):
            assert torch.equal(x[o], other[o])


# ------------------------------------------------------------------ GEMM + AllReduce

AR_SHAPES = [(8, 128, 1032, 512), (4, 200, 512, 264), (2, 64, 256, 64)]


@pytest.mark.parametrize("R,m,n,k", AR_SHAPES)
def test_ar_integer_bit_exact_and_replicas_identical(R, m, n, k):
    w = I.GemmWorkload("t", "ar", R=R, m=m, n=n, k=k, out="bf16", a_seed=71, b_seed=81, integer=True)
    a, b = I.gemm_inputs(w)
    reps = mk.gemm_ar(dev(a), dev(b))
    _ok()
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    want = oracle_bits(exact, "bf16")
    for r in reps:
        np.testing.assert_array_equal(gpu_bits(r), want)


@pytest.mark.parametrize("R,m,n,k", AR_SHAPES)
def test_ar_float(R, m, n, k):
    w = I.GemmWorkload("t", "ar", R=R, m=m, n=n, k=k, out="bf16", a_seed=91, b_seed=101)
    a, b = I.gemm_inputs(w)
    reps = mk.gemm_ar(dev(a), dev(b))
    _ok()
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    r0 = gpu_bits(reps[0])
    for r in reps[1:]:
        np.testing.assert_array_equal(gpu_bits(r), r0)
    assert norm_err(gpu_values(reps[0]), exact, R * k, absmax(a), absmax(b)) <= TOL["bf16"]


@pytest.mark.parametrize("reduce", [mk.REDUCE_RUNNING_SUM, mk.REDUCE_LAST_ARRIVAL])
@pytest.mark.parametrize("split_k", [1, 3])
def test_ar_reductions_integer_bit_exact(reduce, split_k):
    R, m, n, k = 8, 128, 1032, 512
    w = I.GemmWorkload("t", "ar", R=R, m=m, n=n, k=k, out="bf16", a_seed=75, b_seed=85, integer=True)
    a, b = I.gemm_inputs(w)
    reps = mk.gemm_ar(dev(a), dev(b), cfg=mk.Config(reduce=reduce, split_k=split_k))
    _ok()
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    for r in reps:
        np.testing.assert_array_equal(gpu_bits(r), oracle_bits(exact, "bf16"))


def test_ar_equals_rs_blocks():
    R, m, n, k = 4, 512, 512, 256
    w = I.GemmWorkload("t", "rs", R=R, m=m, n=n, k=k, out="bf16", a_seed=5, b_seed=6)
    a, b = I.gemm_inputs(w)
    da, db = dev(a), dev(b)
    blocks = mk.gemm_rs(da, db)
    # Same partial tiles (no split-K) and the same rank-order sum: the same bits.
    reps = mk.gemm_ar(da, db, cfg=mk.Config(split_k=1))
    _ok()
    np.testing.assert_array_equal(gpu_bits(torch.cat(blocks, 0)), gpu_bits(reps[0]))
    # With split-K the order of the fp32 partial sums differs: equal within tolerance.
    reps2 = mk.gemm_ar(da, db, cfg=mk.Config(split_k=2))
    _ok()
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    assert norm_err(gpu_values(reps2[0]), exact, R * k, absmax(a), absmax(b)) <= TOL["bf16"]


# ------------------------------------------------------------------ AllGather + GEMM

AG_SHAPES = [  # R, m_r, n, k, local
    (4, 256, 264, 520, 1),
    (4, 200, 512, 256, 2),   # m_r not a multiple of 128: chunks straddle shards
    (8, 128, 256, 128, 0),
    (1, 300, 256, 64, 0),
]


@pytest.mark.parametrize("R,mr,n,k,local", AG_SHAPES)
def test_ag_integer_bit_exact(R, mr, n, k, local):
    w = I.GemmWorkload("t", "ag", R=R, m=mr, n=n, k=k, out="bf16", a_seed=111, b_seed=121,
                       integer=True)
    a, b = I.gemm_inputs(w)
    g, c = mk.ag_gemm(dev(a), b[0].cuda(), local_rank=local)
    _ok()
    gathered, want = O.ag_gemm([I.bits(x) for x in a], I.bits(b[0]), out="bf16")
    np.testing.assert_array_equal(I.bits(g), gathered)
    np.testing.assert_array_equal(gpu_bits(c), want)


@pytest.mark.parametrize("R,mr,n,k,local", AG_SHAPES)
def test_ag_float(R, mr, n, k, local):
    w = I.GemmWorkload("t", "ag", R=R, m=mr, n=n, k=k, out="f32", a_seed=131, b_seed=141)
    a, b = I.gemm_inputs(w)
    g, c = mk.ag_gemm(dev(a), b[0].cuda(), local_rank=local, out_dtype=torch.float32)
    _ok()
    gathered, exact = O.ag_gemm([I.bits(x) for x in a], I.bits(b[0]), out="f64")
    np.testing.assert_array_equal(I.bits(g), gathered)
    assert norm_err(gpu_values(c), exact, k, absmax(a), absmax(b)) <= TOL["f32"]


@pytest.mark.parametrize("n_copy", [1, 3, 8, 16, 40])
def test_ag_copy_role_sizes(n_copy):
    R, mr, n, k, local = 8, 256, 512, 256, 5
    w = I.GemmWorkload("t", "ag", R=R, m=mr, n=n, k=k, out="bf16", a_seed=171, b_seed=173,
                       integer=True)
    a, b = I.gemm_inputs(w)
    g, c = mk.ag_gemm(dev(a), b[0].cuda(), local_rank=local, cfg=mk.Config(n_copy_ctas=n_copy))
    _ok()
    gathered, want = O.ag_gemm([I.bits(x) for x in a], I.bits(b[0]), out="bf16")
    np.testing.assert_array_equal(I.bits(g), gathered)
    np.testing.assert_array_equal(gpu_bits(c), want)


def test_ag_aliased_local_shard():
    # The caller's local shard already sits inside the gathered buffer: it is not copied.
    R, mr, n, k, local = 4, 256, 256, 256, 3
    w = I.GemmWorkload("t", "ag", R=R, m=mr, n=n, k=k, out="bf16", a_seed=151, b_seed=161,
                       integer=True)
    a, b = I.gemm_inputs(w)
    g = torch.zeros((R * mr, k), dtype=torch.bfloat16, device="cuda")
    g[local * mr:(local + 1) * mr] = a[local].cuda()
    shards = dev(a)
    shards[local] = g[local * mr:(local + 1) * mr]
    g2, c = mk.ag_gemm(shards, b[0].cuda(), local_rank=local, a_gathered=g)
    _ok()
    gathered, want = O.ag_gemm([I.bits(x) for x in a], I.bits(b[0]), out="bf16")
    np.testing.assert_array_equal(I.bits(g2), gathered)
    np.testing.assert_array_equal(gpu_bits(c), want)


# ------------------------------------------------------------------ baselines and repeat calls

@pytest.mark.parametrize("mode", [mk.MODE_GEMM_ONLY, mk.MODE_UNFUSED])
def test_baseline_modes_integer(mode):
    R, m, n, k = 4, 512, 512, 256
    w = I.GemmWorkload("t", "rs", R=R, m=m, n=n, k=k, out="bf16", a_seed=171, b_seed=181,
                       integer=True)
    a, b = I.gemm_inputs(w)
    da, db = dev(a), dev(b)
    cfg = mk.Config(mode=mode)
    blocks = mk.gemm_rs(da, db, cfg=cfg)
    reps = mk.gemm_ar(da, db, cfg=cfg)
    _ok()
    a_bits, b_bits = [I.bits(x) for x in a], [I.bits(x) for x in b]
    exact = O.sum_over_ranks(a_bits, b_bits)
    want = oracle_bits(exact, "bf16")
    np.testing.assert_array_equal(gpu_bits(torch.cat(blocks, 0)), want)
    if mode == mk.MODE_GEMM_ONLY:
        # the AR baseline: replica r holds rank r's own product (no reduction)
        for r, part in enumerate(O.rank_partials(a_bits, b_bits)):
            np.testing.assert_array_equal(gpu_bits(reps[r]), oracle_bits(part, "bf16"))
    else:
        np.testing.assert_array_equal(gpu_bits(reps[-1]), want)
    wa = I.GemmWorkload("t", "ag", R=R, m=128, n=n, k=k, out="bf16", a_seed=191, b_seed=201,
                        integer=True)
    aa, bb = I.gemm_inputs(wa)
    gathered, want = O.ag_gemm([I.bits(x) for x in aa], I.bits(bb[0]), out="bf16")
    g = torch.from_numpy(gathered.view(np.int16)).view(torch.bfloat16).cuda() \
        if mode == mk.MODE_GEMM_ONLY else None
    g2, c = mk.ag_gemm(dev(aa), bb[0].cuda(), a_gathered=g, cfg=cfg)
    _ok()
    np.testing.assert_array_equal(I.bits(g2), gathered)
    np.testing.assert_array_equal(gpu_bits(c), want)


def test_repeated_calls_reuse_workspace():
    R, m, n, k = 2, 256, 512, 128
    ws = mk.Workspace()
    for seed in range(3):
        w = I.GemmWorkload("t", "rs", R=R, m=m, n=n, k=k, out="f32", a_seed=300 + seed,
                           b_seed=400 + seed, integer=True)
        a, b = I.gemm_inputs(w)
        blocks = mk.gemm_rs(dev(a), dev(b), out_dtype=torch.float32, workspace=ws)
        st, _ = mk.device_status(ws)
        assert st == mk.MK_OK
        want = O.gemm_rs([I.bits(x) for x in a], [I.bits(x) for x in b], out="f32")
        for o in range(R):
            np.testing.assert_array_equal(blocks[o].cpu().numpy(), want[o])


def test_empty_and_k_zero():
    a = [torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")] * 2
    b = [torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")] * 2
    out = mk.gemm_rs(a, b)
    assert out[0].shape == (0, 256)
    a = [torch.ones((128, 0), dtype=torch.bfloat16, device="cuda")] * 2
    b = [torch.ones((0, 256), dtype=torch.bfloat16, device="cuda")] * 2
    outs = [torch.full((64, 256), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    mk.gemm_rs(a, b, c_blocks=outs)
    _ok()
    assert all(float(o.abs().max()) == 0.0 for o in outs)


# ------------------------------------------------------------------ bounded waits

def test_missing_copy_flag_times_out_and_context_survives():
    R, mr, n, k = 4, 256, 256, 256
    w = I.GemmWorkload("t", "ag", R=R, m=mr, n=n, k=k, out="bf16", a_seed=1, b_seed=2, integer=True)
    a, b = I.gemm_inputs(w)
    ws = mk.Workspace()
    mk.ag_gemm(dev(a), b[0].cuda(), cfg=mk.Config(inject=1, wait_limit_ns=20_000_000), workspace=ws)
    st, detail = mk.device_status(ws)
    assert st == mk.MK_ERR_TIMEOUT
    # the next call on the same workspace is clean
    g, c = mk.ag_gemm(dev(a), b[0].cuda(), workspace=ws)
    st, _ = mk.device_status(ws)
    assert st == mk.MK_OK
    gathered, _ = O.ag_gemm([I.bits(x) for x in a], I.bits(b[0]))
    np.testing.assert_array_equal(I.bits(g), gathered)


@pytest.mark.parametrize("n_red", [0, 2])
def test_missing_partial_flag_times_out(n_red):
    R, m, n, k = 2, 256, 256, 128
    w = I.GemmWorkload("t", "rs", R=R, m=m, n=n, k=k, out="bf16", a_seed=3, b_seed=4, integer=True)
    a, b = I.gemm_inputs(w)
    ws = mk.Workspace()
    mk.gemm_rs(dev(a), dev(b), cfg=mk.Config(inject=2, wait_limit_ns=20_000_000, n_reduce_ctas=n_red),
               workspace=ws)
    st, _ = mk.device_status(ws)
    assert st == mk.MK_ERR_TIMEOUT
    blocks = mk.gemm_rs(dev(a), dev(b), workspace=ws)
    st, _ = mk.device_status(ws)
    assert st == mk.MK_OK
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    np.testing.assert_array_equal(gpu_bits(torch.cat(blocks, 0)), oracle_bits(exact, "bf16"))


def test_ops_share_one_workspace():
    # RS leaves epoch-tagged flags where AG keeps its chunk counters; AG must not care.
    ws = mk.Workspace()
    w = I.GemmWorkload("t", "rs", R=2, m=256, n=256, k=256, out="bf16", a_seed=21, b_seed=22,
                       integer=True)
    a, b = I.gemm_inputs(w)
    mk.gemm_rs(dev(a), dev(b), workspace=ws)
    wa = I.GemmWorkload("t", "ag", R=4, m=128, n=256, k=256, out="bf16", a_seed=23, b_seed=24,
                        integer=True)
    aa, bb = I.gemm_inputs(wa)
    for cfg in (None, mk.Config(n_copy_ctas=4), None):
        g, c = mk.ag_gemm(dev(aa), bb[0].cuda(), local_rank=1, cfg=cfg, workspace=ws)
        st, detail = mk.device_status(ws)
        assert st == mk.MK_OK, (mk.status_string(st), detail)
        gathered, want = O.ag_gemm([I.bits(x) for x in aa], I.bits(bb[0]), out="bf16")
        np.testing.assert_array_equal(I.bits(g), gathered)
        np.testing.assert_array_equal(gpu_bits(c), want)
    blocks = mk.gemm_rs(dev(a), dev(b), workspace=ws)
    st, _ = mk.device_status(ws)
    assert st == mk.MK_OK
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    np.testing.assert_array_equal(gpu_bits(torch.cat(blocks, 0)), oracle_bits(exact, "bf16"))
