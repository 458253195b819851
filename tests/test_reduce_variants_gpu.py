"""Reduction variants of GEMM + ReduceScatter / AllReduce (GPU): the running
sum forwarded with bf16 on the wire, and the atomic reduction (every partial
added into one fp32 tile per output tile with red.global.add).

bf16 wire: integer-valued inputs keep every rank's partial exact in fp32, so
the result must equal the oracle's bf16-wire running sum bit for bit (the
forwarded sums do round: they exceed bf16's exact range); float inputs stay
within the normalised tolerance of the plain sum.
Atomic: with integer-valued inputs every partial sum is exact in fp32 in any
order, so the result equals the plain definition bit for bit; float inputs
within tolerance.  Shapes cover one and several ranks, ragged n and k, odd
row-block counts with CTA pairs, split-K and repeated calls on one workspace
(the accumulator tiles are zeroed by each call).
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


def _inputs(op, R, m, n, k, integer, seed):
    w = I.GemmWorkload("t", op, R=R, m=m, n=n, k=k, out="bf16", a_seed=seed, b_seed=seed + 1,
                       integer=integer)
    return I.gemm_inputs(w)


def _run(op, a, b, cfg, out_dtype=torch.bfloat16, ws=None):
    if op == "rs":
        res = mk.gemm_rs(dev(a), dev(b), out_dtype=out_dtype, cfg=cfg, workspace=ws)
        return torch.cat(res, 0)
    reps = mk.gemm_ar(dev(a), dev(b), out_dtype=out_dtype, cfg=cfg, workspace=ws)
    for r in reps[1:]:
        assert torch.equal(r, reps[0])          # replicas: the same bits
    return reps[0]


SHAPES = [  # op, R, m, n, k
    ("rs", 1, 136, 256, 64),
    ("rs", 4, 520, 520, 200),     # 5 row blocks (odd with pairs), ragged n and k
    ("rs", 8, 1024, 512, 512),
    ("ar", 8, 128, 1032, 512),
    ("ar", 2, 384, 264, 136),
]


@pytest.mark.parametrize("pair", PAIRS)
@pytest.mark.parametrize("op,R,m,n,k", SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_bf16_wire_integer_bit_exact(op, R, m, n, k, pair, out):
    a, b = _inputs(op, R, m, n, k, True, 101)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    got = _run(op, a, b, mk.Config(cta_pair=pair, wire=mk.WIRE_BF16), dt)
    _ok()
    want = O.running_sum_bf16_wire(O.rank_partials([I.bits(x) for x in a], [I.bits(x) for x in b]), out)
    np.testing.assert_array_equal(gpu_bits(got), want if out == "bf16" else want.view(np.uint32))


@pytest.mark.parametrize("op,R,m,n,k", SHAPES[1:4])
def test_bf16_wire_float_within_tolerance(op, R, m, n, k):
    a, b = _inputs(op, R, m, n, k, False, 111)
    got = _run(op, a, b, mk.Config(wire=mk.WIRE_BF16))
    _ok()
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    assert norm_err(gpu_values(got), exact, R * k, absmax(a), absmax(b)) <= TOL["bf16"]


@pytest.mark.parametrize("pair", PAIRS)
@pytest.mark.parametrize("op,R,m,n,k", SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_atomic_integer_bit_exact(op, R, m, n, k, pair, out):
    a, b = _inputs(op, R, m, n, k, True, 121)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    got = _run(op, a, b, mk.Config(cta_pair=pair, reduce=mk.REDUCE_ATOMIC), dt)
    _ok()
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    np.testing.assert_array_equal(gpu_bits(got), oracle_bits(exact, out))


@pytest.mark.parametrize("op,R,m,n,k", SHAPES[1:4])
def test_atomic_float_within_tolerance(op, R, m, n, k):
    a, b = _inputs(op, R, m, n, k, False, 131)
    got = _run(op, a, b, mk.Config(reduce=mk.REDUCE_ATOMIC), torch.float32)
    _ok()
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    assert norm_err(gpu_values(got), exact, R * k, absmax(a), absmax(b)) <= TOL["f32"]


def test_atomic_split_k_and_repeated_calls():
    # split-K: 3 partials per rank, all added; a second and third call on the same
    # workspace must zero the accumulators again
    a, b = _inputs("rs", 4, 512, 512, 1032, True, 141)
    ws = mk.Workspace()
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    for _ in range(3):
        got = _run("rs", a, b, mk.Config(reduce=mk.REDUCE_ATOMIC, split_k=3), ws=ws)
        _ok(ws)
        np.testing.assert_array_equal(gpu_bits(got), oracle_bits(exact, "bf16"))


def test_variants_agree_with_default_on_integers():
    a, b = _inputs("rs", 8, 1024, 768, 512, True, 151)
    base = _run("rs", a, b, mk.Config(), torch.float32)
    atom = _run("rs", a, b, mk.Config(reduce=mk.REDUCE_ATOMIC), torch.float32)
    last = _run("rs", a, b, mk.Config(reduce=mk.REDUCE_LAST_ARRIVAL), torch.float32)
    _ok()
    assert torch.equal(base, atom) and torch.equal(base, last)


def test_few_ctas_atomic_and_wire():
    # one pair / a few CTAs walk every tile (zero shares of the idle CTAs included)
    for pair, max_ctas in [(mk.PAIR_ON, 2), (mk.PAIR_OFF, 3)]:
        a, b = _inputs("rs", 4, 512, 512, 256, True, 161)
        exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
        got = _run("rs", a, b, mk.Config(reduce=mk.REDUCE_ATOMIC, cta_pair=pair, max_ctas=max_ctas))
        _ok()
        np.testing.assert_array_equal(gpu_bits(got), oracle_bits(exact, "bf16"))
        got = _run("rs", a, b, mk.Config(wire=mk.WIRE_BF16, cta_pair=pair, max_ctas=max_ctas))
        _ok()
        want = O.running_sum_bf16_wire(O.rank_partials([I.bits(x) for x in a], [I.bits(x) for x in b]), "bf16")
        np.testing.assert_array_equal(gpu_bits(got), want)


# Sliced reduction (reduce = 4): every partial staged, then slices summed in
# rank order by all epilogue warps.  The order is the running sum's, so on any
# inputs the result must be the same bits as reduce = 1 (fp32 addition of the
# same values in the same order); with integer inputs it equals the oracle.
@pytest.mark.parametrize("pair", PAIRS)
@pytest.mark.parametrize("op,R,m,n,k", SHAPES)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_sliced_same_bits_as_running_sum(op, R, m, n, k, pair, out):
    a, b = _inputs(op, R, m, n, k, False, 171)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    chain = _run(op, a, b, mk.Config(cta_pair=pair, reduce=mk.REDUCE_RUNNING_SUM), dt)
    sliced = _run(op, a, b, mk.Config(cta_pair=pair, reduce=mk.REDUCE_SLICED), dt)
    _ok()
    assert torch.equal(chain, sliced)


@pytest.mark.parametrize("op,R,m,n,k", SHAPES)
def test_sliced_integer_bit_exact_few_ctas(op, R, m, n, k):
    # three CTAs: every epilogue warp takes several slices after its tiles
    a, b = _inputs(op, R, m, n, k, True, 181)
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    got = _run(op, a, b, mk.Config(reduce=mk.REDUCE_SLICED, cta_pair=mk.PAIR_OFF, max_ctas=3))
    _ok()
    np.testing.assert_array_equal(gpu_bits(got), oracle_bits(exact, "bf16"))


def test_sliced_is_the_small_allreduce_default_and_repeats():
    # the decode-like AR (few output tiles) takes the sliced reduction by default;
    # repeated calls on one workspace (counters zeroed by each call) agree
    a, b = _inputs("ar", 8, 128, 1024, 512, False, 191)
    ws = mk.Workspace()
    base = _run("ar", a, b, mk.Config(reduce=mk.REDUCE_RUNNING_SUM), ws=ws)
    for _ in range(3):
        got = _run("ar", a, b, mk.Config(), ws=ws)
        _ok(ws)
        assert torch.equal(got, base)
