"""Pins for the CPU oracle (CPU only).

Each check ties the oracle to something other than itself: the IEEE
definition of round-to-nearest-even, brute-force loops on tiny inputs, closed
forms, invariants of the collectives, and special cases that reduce to a
library routine (torch's fp32->bf16 cast, numpy's stable argsort).  The cases
are chosen so that a dropped term, a wrong sign or index, a transposed
operand, a wrong gather order or a wrong owner block fails at least one.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle as O
from comm_gemm_tile_gb300 import inputs as I


def bf(x):
    """float values -> bf16 bits via torch (inputs only; exact for small ints)."""
    return I.bits(torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def rand_int_bits(shape, seed, lo=-3, hi=3):
    g = np.random.default_rng(seed)
    return bf(g.integers(lo, hi + 1, size=shape).astype(np.float32))


def brute_matmul(a, b):
    """Pure-Python triple loop on float64 values."""
    m, k = a.shape
    k2, n = b.shape
    assert k == k2
    c = np.zeros((m, n))
    for i in range(m):
        for j in range(n):
            s = 0.0
            for t in range(k):
                s += float(a[i, t]) * float(b[t, j])
            c[i, j] = s
    return c


# ---------------------------------------------------------------- rounding

@pytest.mark.parametrize("x,expect", [
    (1.0, 0x3F80),
    (-1.5, 0xBFC0),
    (1.0 + 2.0 ** -8, 0x3F80),                 # tie -> even (mantissa 0)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),             # tie -> even (mantissa 2)
    (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),    # just above the tie -> up
    (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),    # single rounding (via fp32 would give 0x3F80)
    (-(1.0 + 2.0 ** -8 + 2.0 ** -20), 0xBF81),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (2.0 ** -133, 0x0001),                     # smallest subnormal
    (2.0 ** -134, 0x0000),                     # tie with 0 -> even (0)
    (3 * 2.0 ** -134, 0x0002),                 # 1.5 quanta: tie -> 2
    (2.0 ** -126, 0x0080),                     # smallest normal
    ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),    # largest finite
    ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),    # tie between max and 2^128 -> even -> inf
    (-1e39, 0xFF80),
    (float("inf"), 0x7F80),
    (65536.0 + 256.0, 0x4780),                 # 65792 = 2^16(1+2^-8): tie -> 65536
    (65536.0 + 257.0, 0x4781),
])
def test_bf16_rne_closed_forms(x, expect):
    assert int(O.f64_to_bf16_bits(np.array([x]))[0]) == expect


def test_bf16_rne_nan():
    b = int(O.f64_to_bf16_bits(np.array([np.nan]))[0])
    assert (b & 0x7F80) == 0x7F80 and (b & 0x7F) != 0


def test_bf16_rne_matches_torch_on_fp32_values():
    # For values that are exactly fp32, single RNE to bf16 equals torch's cast.
    g = np.random.default_rng(7)
    x = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (g.standard_normal(2000) * 1e-39).astype(np.float32),    # fp32 subnormals
        g.integers(-70000, 70000, 5000).astype(np.float32),
    ])
    want = I.bits(torch.from_numpy(x).to(torch.bfloat16))
    got = O.f64_to_bf16_bits(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("b,val", [(0x3F80, 1.0), (0xC000, -2.0), (0x0001, 2.0 ** -133),
                                   (0x7F80, np.inf), (0x4049, 3.140625)])
def test_bf16_widen_closed_forms(b, val):
    assert O.bf16_to_f64(np.array([b], np.uint16))[0] == val


def test_bf16_roundtrip_all_finite_patterns():
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = O.bf16_to_f64(allb)
    fin = np.isfinite(v)
    back = O.f64_to_bf16_bits(v[fin])
    # -0.0 and +0.0 keep their sign
    np.testing.assert_array_equal(back, allb[fin])


def test_f32_output_rounding():
    x = np.array([1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24, 0.1])
    got = O.round_out(x, "f32")
    assert got[0] == np.float32(1.0)                      # tie -> even
    assert got[1] == np.float32(1.0 + 2.0 ** -22)         # tie -> even (up)
    assert got.dtype == np.float32


# ---------------------------------------------------------------- AllGather + GEMM

def test_ag_brute_force_tiny():
    R, mr, k, n = 3, 2, 5, 4
    shards = [rand_int_bits((mr, k), 10 + r) for r in range(R)]
    b = rand_int_bits((k, n), 99)
    gathered, c = O.ag_gemm(shards, b, out="f32")
    A = np.concatenate([O.bf16_to_f64(s) for s in shards], 0)
    want = brute_matmul(A, O.bf16_to_f64(b))
    np.testing.assert_array_equal(c, want.astype(np.float32))
    assert gathered.shape == (R * mr, k)


def test_ag_gather_order_closed_form():
    # shard r is all (r+1): block r of C must be (r+1) * column sums of B.
    R, mr, k, n = 4, 3, 6, 5
    shards = [bf(np.full((mr, k), r + 1.0)) for r in range(R)]
    b = rand_int_bits((k, n), 5)
    gathered, c = O.ag_gemm(shards, b, out="f32")
    colsum = O.bf16_to_f64(b).sum(0)
    for r in range(R):
        np.testing.assert_array_equal(c[r * mr:(r + 1) * mr], np.tile((r + 1) * colsum, (mr, 1)))
        np.testing.assert_array_equal(gathered[r * mr:(r + 1) * mr], shards[r])


def test_ag_row_sample_matches_full():
    R, mr, k, n = 2, 8, 16, 8
    shards = [rand_int_bits((mr, k), 20 + r) for r in range(R)]
    b = rand_int_bits((k, n), 30)
    _, full = O.ag_gemm(shards, b)
    rows = np.array([0, 5, 9, 15])
    _, part = O.ag_gemm(shards, b, rows=rows)
    np.testing.assert_array_equal(part, full[rows])


# ---------------------------------------------------------------- GEMM + RS / AR

def test_rs_brute_force_tiny():
    R, m, k, n = 2, 4, 3, 5
    a = [rand_int_bits((m, k), 40 + r) for r in range(R)]
    b = [rand_int_bits((k, n), 50 + r) for r in range(R)]
    blocks = O.gemm_rs(a, b, out="f32")
    want = sum(brute_matmul(O.bf16_to_f64(a[r]), O.bf16_to_f64(b[r])) for r in range(R))
    np.testing.assert_array_equal(np.concatenate(blocks, 0), want.astype(np.float32))
    assert [blk.shape for blk in blocks] == [(2, 5), (2, 5)]


def test_rs_closed_form_constant():
    # A_r = 1, B_r = (r+1): S = k * R(R+1)/2 everywhere.
    R, m, k, n = 4, 8, 7, 3
    a = [bf(np.ones((m, k))) for _ in range(R)]
    b = [bf(np.full((k, n), r + 1.0)) for r in range(R)]
    for blk in O.gemm_rs(a, b, out="f32"):
        assert np.all(blk == k * R * (R + 1) / 2)


def test_rs_owner_blocks_closed_form():
    # Row i of every A_r is (i+1) e_0, row 0 of B_r is r+1: S[i, j] = (i+1) * R(R+1)/2.
    R, m, k, n = 4, 16, 3, 2
    a_np = np.zeros((m, k))
    a_np[:, 0] = np.arange(1, m + 1)
    a = [bf(a_np) for _ in range(R)]
    b = []
    for r in range(R):
        bb = np.zeros((k, n))
        bb[0, :] = r + 1
        b.append(bf(bb))
    blocks = O.gemm_rs(a, b, out="f32")
    h = m // R
    for o, blk in enumerate(blocks):
        rows = np.arange(o * h, (o + 1) * h)
        np.testing.assert_array_equal(blk[:, 0], (rows + 1) * R * (R + 1) / 2)
        assert list(O.owner_rows(m, R, o)) == rows.tolist()


def test_rs_rank_sum_not_product_and_all_terms():
    # Dropping any rank's term changes the result (each rank contributes a distinct power of 2).
    R, m, k, n = 3, 3, 2, 2
    a = [bf(np.full((m, k), 2.0 ** r)) for r in range(R)]
    b = [bf(np.ones((k, n))) for _ in range(R)]
    s = np.concatenate(O.gemm_rs(a, b, out="f32"), 0)
    assert np.all(s == k * (2 ** R - 1))


def test_rs_requires_divisible_m():
    a = [bf(np.ones((5, 2)))] * 2
    b = [bf(np.ones((2, 2)))] * 2
    with pytest.raises(ValueError):
        O.gemm_rs(a, b)


def test_r1_is_plain_gemm_brute_force():
    a = [rand_int_bits((3, 4), 61)]
    b = [rand_int_bits((4, 6), 62)]
    want = brute_matmul(O.bf16_to_f64(a[0]), O.bf16_to_f64(b[0])).astype(np.float32)
    np.testing.assert_array_equal(O.gemm_rs(a, b, "f32")[0], want)
    np.testing.assert_array_equal(O.gemm_ar(a, b, "f32")[0], want)
    np.testing.assert_array_equal(O.ag_gemm(a, b[0], "f32")[1], want)


def test_ar_replicas_equal_rs_blocks_union():
    R, m, k, n = 4, 8, 16, 8
    g = np.random.default_rng(3)
    a = [bf(g.standard_normal((m, k))) for _ in range(R)]
    b = [bf(g.standard_normal((k, n)) * 0.02) for _ in range(R)]
    reps = O.gemm_ar(a, b, "bf16")
    rs = np.concatenate(O.gemm_rs(a, b, "bf16"), 0)
    for rep in reps:
        np.testing.assert_array_equal(rep, reps[0])
    np.testing.assert_array_equal(reps[0], rs)


def test_rs_rank_permutation_invariant_integers():
    R, m, k, n = 3, 6, 5, 4
    a = [rand_int_bits((m, k), 70 + r) for r in range(R)]
    b = [rand_int_bits((k, n), 80 + r) for r in range(R)]
    base = np.concatenate(O.gemm_rs(a, b, "f32"), 0)
    for perm in itertools.permutations(range(R)):
        s = np.concatenate(O.gemm_rs([a[p] for p in perm], [b[p] for p in perm], "f32"), 0)
        np.testing.assert_array_equal(s, base)
    assert np.all(base == np.round(base))


def test_integer_config_sums_are_exact_in_fp32():
    # The tiny bit-exact workload: |S| <= 2*2*256*2 < 2**24, so any fp32 summation order is exact.
    w = I.RS_R2_256_INT
    a, b = I.gemm_inputs(w)
    s = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])
    assert np.abs(s).max() < 2 ** 24
    assert np.all(s == np.round(s))


# ---------------------------------------------------------------- MoE

# ---- the bf16-wire running sum (a reduction variant of GEMM + ReduceScatter / AllReduce)


def test_wire_single_partial_is_plain_rounding():
    rng = np.random.default_rng(5)
    x = rng.normal(size=(4, 9)) * 100
    for out in ("bf16", "f32"):
        np.testing.assert_array_equal(O.running_sum_bf16_wire([x], out), O.round_out(x, out))


def test_wire_hand_worked_example():
    # partials 256, 1, 1 (exact sum 258): s0 = bf16(256) = 256; 256 + 1 = 257 lies halfway
    # between the bf16 neighbours 256 and 258 and rounds to the even mantissa, 256; the last
    # part adds 1 in fp32: 257 (fp32 out), which rounds to 256 in bf16 (halfway again).
    parts = [np.array([[256.0]]), np.array([[1.0]]), np.array([[1.0]])]
    assert float(O.running_sum_bf16_wire(parts, "f32")[0, 0]) == 257.0
    assert O.bf16_to_f64(O.running_sum_bf16_wire(parts, "bf16"))[0, 0] == 256.0
    # with two parts nothing is rounded before the last addition: 256 + 1 + 1 ... = plain sum
    assert float(O.running_sum_bf16_wire([np.array([[256.0]]), np.array([[2.0]])], "f32")[0, 0]) == 258.0
    # the order matters once rounding happens: 1, 1, 256 keeps every bit
    assert float(O.running_sum_bf16_wire(parts[::-1], "f32")[0, 0]) == 258.0


def test_wire_equals_plain_sum_when_every_forward_is_exact():
    # integers whose running sums stay within bf16's exact range (|s| <= 256)
    rng = np.random.default_rng(6)
    parts = [rng.integers(-30, 31, size=(8, 16)).astype(np.float64) for _ in range(8)]
    exact = sum(parts)
    for out in ("bf16", "f32"):
        np.testing.assert_array_equal(O.running_sum_bf16_wire(parts, out), O.round_out(exact, out))


def test_wire_error_within_its_roundings():
    # each forward rounds to bf16 (at most half a bf16 unit, 2^-9 relative) and the last
    # addition to fp32; the result stays within the sum of those half-units of the exact sum
    rng = np.random.default_rng(7)
    parts = [rng.normal(size=(32, 32)) * 50 for _ in range(6)]
    got = O.running_sum_bf16_wire(parts, "f32").astype(np.float64)
    bound = np.zeros_like(got)
    s = np.zeros_like(got)
    for x in parts[:-1]:
        s = s + x
        bound += np.abs(s) * 2.0 ** -8 + 1e-12
    exact = sum(parts)
    bound += np.abs(exact) * 2.0 ** -23 + 1e-12
    assert np.all(np.abs(got - exact) <= bound)
    # and it is not the plain rounding in general (the wire does round)
    assert not np.array_equal(got, O.round_out(exact, "f32"))


def test_rank_partials_sum_to_s():
    rng = np.random.default_rng(8)
    a = [I.bits(torch.from_numpy(rng.normal(size=(6, 10)).astype(np.float32)).bfloat16()) for _ in range(3)]
    b = [I.bits(torch.from_numpy(rng.normal(size=(10, 5)).astype(np.float32)).bfloat16()) for _ in range(3)]
    np.testing.assert_allclose(sum(O.rank_partials(a, b)), O.sum_over_ranks(a, b), rtol=0, atol=1e-12)


def test_rank_partials_brute_force_and_row_sample():
    # each term is its own rank's product (brute force), and a row sample is those rows
    R, m, k, n = 3, 5, 4, 3
    a = [rand_int_bits((m, k), 60 + r) for r in range(R)]
    b = [rand_int_bits((k, n), 70 + r) for r in range(R)]
    parts = O.rank_partials(a, b)
    for r in range(R):
        np.testing.assert_array_equal(parts[r], brute_matmul(O.bf16_to_f64(a[r]), O.bf16_to_f64(b[r])))
    rows = np.array([4, 0, 2])
    for full, part in zip(parts, O.rank_partials(a, b, rows=rows)):
        np.testing.assert_array_equal(part, full[rows])


def test_unrounded_output_is_the_float64_result():
    # out='f64' returns the exact sum itself: a value no fp32 or bf16 holds survives unrounded
    x = np.array([1.0 + 2.0 ** -40, -3.0, 2.0 ** -140])
    np.testing.assert_array_equal(O.round_out(x, "f64"), x)
    shards = [rand_int_bits((2, 3), 80 + r) for r in range(2)]
    b = rand_int_bits((3, 2), 90)
    _, c64 = O.ag_gemm(shards, b, out="f64")
    A = np.concatenate([O.bf16_to_f64(s) for s in shards], 0)
    np.testing.assert_array_equal(c64, brute_matmul(A, O.bf16_to_f64(b)))
    assert c64.dtype == np.float64


# ---- fp8 e4m3 operands


def test_e4m3_all_patterns_match_torch():
    b = np.arange(256, dtype=np.uint8)
    mine = O.e4m3_to_f64(b)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    np.testing.assert_array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])


@pytest.mark.parametrize("byte,val", [(0x38, 1.0), (0xB8, -1.0), (0x7E, 448.0), (0x01, 2.0 ** -9),
                                      (0x08, 2.0 ** -6), (0x07, 7 * 2.0 ** -9), (0x40, 2.0),
                                      (0x3C, 1.5), (0x00, 0.0)])
def test_e4m3_closed_forms(byte, val):
    assert O.e4m3_to_f64(np.array([byte], dtype=np.uint8))[0] == val


def test_e4m3_nan_patterns_only():
    v = O.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    assert set(np.flatnonzero(np.isnan(v)).tolist()) == {0x7F, 0xFF}
    assert np.nanmax(np.abs(v)) == 448.0


def test_fp8_gemm_brute_force_tiny():
    rng = np.random.default_rng(9)
    ok = np.array([x for x in range(256) if (x & 0x7F) != 0x7F], dtype=np.uint8)
    a = [rng.choice(ok, size=(3, 16)) for _ in range(2)]
    bt = rng.choice(ok, size=(5, 16))
    gathered, c = O.ag_gemm_fp8(a, bt, "f32")
    np.testing.assert_array_equal(gathered, np.concatenate(a, 0))
    dec = O.e4m3_to_f64
    for i in range(6):
        for j in range(5):
            row = dec(gathered[i])
            want = sum(row[kk] * dec(bt[j])[kk] for kk in range(16))
            assert c[i, j] == np.float32(want)
    s = O.sum_over_ranks_fp8(a, [bt, bt])
    np.testing.assert_allclose(s, dec(a[0]) @ dec(bt).T + dec(a[1]) @ dec(bt).T, rtol=0, atol=0)


def test_route_matches_stable_argsort():
    g = np.random.default_rng(11)
    lg = np.round(g.standard_normal((500, 16)) * 2) / 2      # many ties
    lg = lg.astype(np.float32)
    want = np.argsort(-lg, axis=1, kind="stable")[:, :3]
    np.testing.assert_array_equal(O.moe_route(lg, 3), want)


@pytest.mark.parametrize("row,k,expect", [
    ([1.0, 3.0, 3.0, 2.0], 2, [1, 2]),
    ([5.0, 5.0, 5.0, 5.0], 2, [0, 1]),
    ([-1.0, -3.0, 7.0, 0.0], 1, [2]),
    ([0.5, -0.5, 0.25, 0.75], 4, [3, 0, 2, 1]),
    ([-np.inf, -np.inf, -1.0], 3, [2, 0, 1]),
])
def test_route_hand_cases(row, k, expect):
    got = O.moe_route(np.array([row], dtype=np.float32), k)
    assert got[0].tolist() == expect


def test_route_rejects_topk_above_E():
    with pytest.raises(ValueError):
        O.moe_route(np.zeros((2, 3), np.float32), 4)


def test_dispatch_hand_worked_example():
    # R=2 ranks, 2 experts each (E=4), T=2 tokens per rank, top-2.
    idx0 = np.array([[3, 0], [1, 2]])      # rank 0: g=0 -> {3,0}, g=1 -> {1,2}
    idx1 = np.array([[0, 1], [2, 3]])      # rank 1: g=2 -> {0,1}, g=3 -> {2,3}
    recv_src, seg = O.moe_dispatch([idx0, idx1], E_loc=2)
    # rank 0 (experts 0,1): e0 <- (g0,slot1)=1, (g2,slot0)=4 ; e1 <- (g1,slot0)=2, (g2,slot1)=5
    assert recv_src[0].tolist() == [1, 4, 2, 5]
    assert seg[0].tolist() == [2, 2]
    # rank 1 (experts 2,3): e2 <- (g1,slot1)=3, (g3,slot0)=6 ; e3 <- (g0,slot0)=0, (g3,slot1)=7
    assert recv_src[1].tolist() == [3, 6, 0, 7]
    assert seg[1].tolist() == [2, 2]
    counts = O.moe_counts([idx0, idx1], 4)
    assert counts.tolist() == [[1, 1, 1, 1], [1, 1, 1, 1]]


def test_dispatch_invariants_random():
    R, E_loc, T, topk = 4, 3, 50, 2
    logits = [I.zipf_logits(T, R * E_loc, 900 + r).numpy() for r in range(R)]
    idx = [O.moe_route(lg, topk) for lg in logits]
    counts = O.moe_counts(idx, R * E_loc)
    recv_src, seg = O.moe_dispatch(idx, E_loc)
    assert counts.sum() == R * T * topk
    allsrc = np.concatenate(recv_src)
    assert sorted(allsrc.tolist()) == list(range(R * T * topk))      # bijection onto (g, slot)
    idx_all = np.concatenate(idx, 0)
    for d in range(R):
        assert seg[d].sum() == len(recv_src[d])
        start = 0
        for l in range(E_loc):
            e = d * E_loc + l
            part = recv_src[d][start:start + seg[d][l]]
            g = part // topk
            assert np.all(np.diff(g) > 0)                               # token order
            assert np.all(idx_all[g, part % topk] == e)                 # right expert
            assert seg[d][l] == counts[:, e].sum()
            start += seg[d][l]


def test_dispatch_single_expert_is_identity():
    T = 17
    idx = [np.zeros((T, 1), np.int64)]
    recv_src, seg = O.moe_dispatch(idx, E_loc=1)
    assert recv_src[0].tolist() == list(range(T)) and seg[0].tolist() == [T]


def test_expert_gemm_scaled_identity_closed_form():
    # W_l = (l+1) * I: each received row comes back scaled by its expert's factor.
    H = N = 8
    seg = np.array([3, 0, 2])
    rx = rand_int_bits((5, H), 123)
    w = np.stack([bf(np.eye(H) * (l + 1)) for l in range(3)], 0)
    y = O.moe_expert_gemm(rx, seg, w, out="f32")
    scale = np.array([1, 1, 1, 3, 3])[:, None]
    np.testing.assert_array_equal(y, (O.bf16_to_f64(rx) * scale).astype(np.float32))


def test_moe_end_to_end_brute_force_tiny():
    R, E_loc, T, H, N, topk = 2, 2, 3, 4, 3, 2
    x = [rand_int_bits((T, H), 200 + r) for r in range(R)]
    logits = [I.zipf_logits(T, R * E_loc, 300 + r).numpy() for r in range(R)]
    w = [np.stack([rand_int_bits((H, N), 400 + 10 * d + l) for l in range(E_loc)], 0)
         for d in range(R)]
    res = O.moe_dispatch_gemm(x, logits, w, E_loc, topk, out="f32")
    xall = np.concatenate([O.bf16_to_f64(v) for v in x], 0)
    idx_all = np.concatenate(res["topk_idx"], 0)
    for d in range(R):
        for j, src in enumerate(res["recv_src"][d]):
            g, slot = divmod(int(src), topk)
            e = int(idx_all[g, slot])
            assert e // E_loc == d
            np.testing.assert_array_equal(res["recv_x"][d][j], np.concatenate(x, 0)[g])
            want = brute_matmul(xall[g:g + 1], O.bf16_to_f64(w[d][e % E_loc]))[0]
            np.testing.assert_array_equal(res["y"][d][j], want.astype(np.float32))


# ---------------------------------------------------------------- MoE combine

def _combine_case(R, E_loc, T, N, H, topk, seed, gates=None):
    """Routing from seeded Zipf logits, integer hidden rows and weights."""
    logits = [I.zipf_logits(T, R * E_loc, seed + r).numpy() for r in range(R)]
    idx = [O.moe_route(lg, topk) for lg in logits]
    counts = O.moe_counts(idx, R * E_loc)
    recv_src, seg = O.moe_dispatch(idx, E_loc)
    h = [rand_int_bits((len(recv_src[d]) + 3, N), seed + 100 + d) for d in range(R)]  # + junk rows
    w2 = [np.stack([rand_int_bits((N, H), seed + 200 + 10 * d + l) for l in range(E_loc)], 0)
          for d in range(R)]
    if gates is None:
        g = np.random.default_rng(seed + 300)
        gates = [g.choice([0.25, 0.5, 0.75, 1.0], size=(T, topk)).astype(np.float32)
                 for _ in range(R)]
    return idx, counts, recv_src, seg, h, w2, gates


def test_combine_brute_force_tiny():
    # Every (token, slot): find its received row by a linear search of recv_src
    # (not the inverse map), multiply by the slot's expert with a triple loop,
    # round to bf16, weight and sum over slots in Python floats.
    R, E_loc, T, N, H, topk = 2, 2, 5, 3, 4, 2
    idx, counts, recv_src, seg, h, w2, gates = _combine_case(R, E_loc, T, N, H, topk, 510)
    res = O.moe_combine(h, recv_src, counts, w2, gates, E_loc, topk, T, out="f32")
    idx_all = np.concatenate(idx, 0)
    for r in range(R):
        for t in range(T):
            g = r * T + t
            acc = np.zeros(H)
            for k in range(topk):
                e = int(idx_all[g, k])
                d, l = divmod(e, E_loc)
                j = [i for i, v in enumerate(recv_src[d].tolist()) if v == g * topk + k]
                assert len(j) == 1
                z = brute_matmul(O.bf16_to_f64(h[d][j[0]:j[0] + 1]), O.bf16_to_f64(w2[d][l]))[0]
                y = O.bf16_to_f64(O.f64_to_bf16_bits(z))
                np.testing.assert_array_equal(res["ret"][r][t, k], O.f64_to_bf16_bits(z))
                acc += float(gates[r][t, k]) * y
            np.testing.assert_array_equal(res["out"][r][t], acc.astype(np.float32))


def test_combine_one_hot_gates_return_the_slot_rows():
    # gates (1, 0) give back slot 0's expert row exactly, (0, 1) slot 1's:
    # catches a swapped slot or a transposed gate matrix.
    R, E_loc, T, N, H, topk = 3, 2, 9, 4, 5, 2
    for hot in range(topk):
        gates = [np.eye(topk, dtype=np.float32)[np.full(T, hot)] for _ in range(R)]
        idx, counts, recv_src, seg, h, w2, _ = _combine_case(R, E_loc, T, N, H, topk, 520)
        res = O.moe_combine(h, recv_src, counts, w2, gates, E_loc, topk, T)
        for r in range(R):
            np.testing.assert_array_equal(res["out"][r], res["ret"][r][:, hot, :])


def test_dispatch_then_combine_with_identity_experts_returns_the_tokens():
    # x -> dispatch -> (expert = identity) -> combine with gates summing to 1
    # in powers of two gives back x exactly.
    R, E_loc, T, H, topk = 2, 3, 11, 6, 2
    x = [rand_int_bits((T, H), 530 + r) for r in range(R)]
    logits = [I.zipf_logits(T, R * E_loc, 540 + r).numpy() for r in range(R)]
    idx = [O.moe_route(lg, topk) for lg in logits]
    counts = O.moe_counts(idx, R * E_loc)
    recv_src, seg = O.moe_dispatch(idx, E_loc)
    recv_x = [O.moe_gather_rows(x, recv_src[d], topk) for d in range(R)]
    eye = [np.stack([bf(np.eye(H))] * E_loc, 0) for _ in range(R)]
    gates = [np.tile(np.array([[0.75, 0.25]], np.float32), (T, 1)) for _ in range(R)]
    res = O.moe_combine(recv_x, recv_src, counts, eye, gates, E_loc, topk, T)
    for r in range(R):
        np.testing.assert_array_equal(res["out"][r], x[r])


def test_combine_is_linear_in_gates_and_single_rounding():
    # out(a*g) == RNE(a * exact(g)) for a power of two a; and a non-dyadic
    # gate is rounded once (not once per slot).
    R, E_loc, T, N, H, topk = 2, 2, 7, 3, 4, 2
    idx, counts, recv_src, seg, h, w2, gates = _combine_case(R, E_loc, T, N, H, topk, 550)
    base = O.moe_combine(h, recv_src, counts, w2, gates, E_loc, topk, T, out="f32")
    dbl = O.moe_combine(h, recv_src, counts, w2, [2 * g for g in gates], E_loc, topk, T, out="f32")
    for r in range(R):
        np.testing.assert_array_equal(dbl["out"][r], 2 * base["out"][r])
    third = [np.full((T, topk), 1.0 / 3.0) for _ in range(R)]
    res = O.moe_combine(h, recv_src, counts, w2, third, E_loc, topk, T, out="f32")
    for r in range(R):
        exact = O.bf16_to_f64(base["ret"][r]).sum(axis=1) / 3.0
        np.testing.assert_array_equal(res["out"][r], exact.astype(np.float32))


def test_combine_seg_from_counts_and_coverage_check():
    counts = np.array([[1, 2, 0, 3], [4, 0, 5, 6]])
    seg = O.moe_seg_from_counts(counts, 2)
    assert [s.tolist() for s in seg] == [[5, 2], [5, 9]]
    with pytest.raises(ValueError):
        O.moe_return_rows([np.zeros((1, 2), np.uint16)], [np.array([0])], topk=2, T=1, R=1)


# ---------------------------------------------------------------- chained MLP (AG+GEMM -> ReLU -> GEMM+RS)

def test_mlp_brute_force_tiny():
    # triple loops: gather in rank order, ReLU, bf16 rounding of H, sum over ranks, owner blocks
    R, m, h, f = 2, 2, 3, 2
    x = [rand_int_bits((m, h), 600 + r) for r in range(R)]
    w1 = [rand_int_bits((h, f), 610 + r) for r in range(R)]
    w2 = [rand_int_bits((f, h), 620 + r) for r in range(R)]
    res = O.mlp_ag_rs(x, w1, w2, out="f32")
    X = np.concatenate([O.bf16_to_f64(v) for v in x], 0)
    S = np.zeros((R * m, h))
    for r in range(R):
        H = brute_matmul(X, O.bf16_to_f64(w1[r]))
        H = np.where(H > 0, H, 0.0)
        Hb = O.bf16_to_f64(O.f64_to_bf16_bits(H))
        np.testing.assert_array_equal(res["hidden"][r], O.f64_to_bf16_bits(H))
        S += brute_matmul(Hb, O.bf16_to_f64(w2[r]))
    for o in range(R):
        np.testing.assert_array_equal(res["blocks"][o], S[o * m:(o + 1) * m].astype(np.float32))


def test_mlp_relu_kills_negative_preactivations():
    # W1 = -I: every pre-activation is -x, so H = ReLU(-x) keeps only the negative inputs
    R, m, h = 2, 3, 4
    x = [rand_int_bits((m, h), 630 + r) for r in range(R)]
    w1 = [bf(-np.eye(h)) for _ in range(R)]
    hid = O.mlp_hidden(x, w1[0])
    X = np.concatenate([O.bf16_to_f64(v) for v in x], 0)
    np.testing.assert_array_equal(O.bf16_to_f64(hid), np.maximum(-X, 0))


def test_mlp_identity_weights_closed_form():
    # W1_r = I on rank 0 only (others zero), W2_0 = I: the layer returns ReLU(x) row blocks
    R, m, h = 3, 2, 5
    x = [rand_int_bits((m, h), 640 + r) for r in range(R)]
    eye, zero = bf(np.eye(h)), bf(np.zeros((h, h)))
    w1 = [eye] + [zero] * (R - 1)
    w2 = [eye] + [zero] * (R - 1)
    res = O.mlp_ag_rs(x, w1, w2, out="f32")
    for o in range(R):
        np.testing.assert_array_equal(res["blocks"][o],
                                      np.maximum(O.bf16_to_f64(x[o]), 0).astype(np.float32))


def test_mlp_row_sample_matches_full_and_rank_blocks_tile():
    R, m, h, f = 4, 3, 6, 5
    x = [rand_int_bits((m, h), 650 + r) for r in range(R)]
    w1 = [rand_int_bits((h, f), 660 + r) for r in range(R)]
    w2 = [rand_int_bits((f, h), 670 + r) for r in range(R)]
    full = O.mlp_ag_rs(x, w1, w2)
    rows = np.array([0, 5, 11])
    part = O.mlp_ag_rs(x, w1, w2, rows=rows)
    np.testing.assert_array_equal(part["rows"], np.concatenate(full["blocks"], 0)[rows])


# ---------------------------------------------------------------- ring attention

def _attn_case(R, heads, s_r, d, seed):
    q = [rand_int_bits((heads, s_r, d), seed + r, -2, 2) for r in range(R)]
    k = [rand_int_bits((heads, s_r, d), seed + 10 + r, -2, 2) for r in range(R)]
    v = [rand_int_bits((heads, s_r, d), seed + 20 + r, -2, 2) for r in range(R)]
    return q, k, v


@pytest.mark.parametrize("causal", [False, True])
def test_ring_attention_brute_force_tiny(causal):
    # per query: Python loops over every key of every rank, softmax by its definition
    import math
    R, heads, s_r, d, scale = 3, 2, 2, 3, 0.25
    q, k, v = _attn_case(R, heads, s_r, d, 700)
    got = O.ring_attention(q, k, v, causal, scale, out="f32")
    for r in range(R):
        for hh in range(heads):
            for i in range(s_r):
                qi = O.bf16_to_f64(q[r][hh, i])
                scores, vals = [], []
                for s_ in range(R):
                    for j in range(s_r):
                        if causal and s_ * s_r + j > r * s_r + i:
                            continue
                        scores.append(scale * float(np.dot(qi, O.bf16_to_f64(k[s_][hh, j]))))
                        vals.append(O.bf16_to_f64(v[s_][hh, j]))
                e = [math.exp(x) for x in scores]
                want = sum(w * vv for w, vv in zip(e, vals)) / sum(e)
                np.testing.assert_allclose(got[r][hh, i], want.astype(np.float32), rtol=1e-6, atol=1e-6)


def test_ring_attention_zero_queries_average_the_values():
    # Q = 0: every score is 0, so each output row is the mean of the visible values
    R, heads, s_r, d = 2, 3, 4, 5
    _, k, v = _attn_case(R, heads, s_r, d, 710)
    q = [bf(np.zeros((heads, s_r, d))) for _ in range(R)]
    vall = np.concatenate([O.bf16_to_f64(x) for x in v], axis=1)
    got = O.ring_attention(q, k, v, False, 1.0, out="f32")
    for r in range(R):
        np.testing.assert_allclose(got[r], np.broadcast_to(vall.mean(axis=1, keepdims=True),
                                                           got[r].shape), rtol=1e-6, atol=1e-6)
    got = O.ring_attention(q, k, v, True, 1.0, out="f32")
    for r in range(R):
        for i in range(s_r):
            n = r * s_r + i + 1
            np.testing.assert_allclose(got[r][:, i], vall[:, :n].mean(axis=1), rtol=1e-6, atol=1e-6)


def test_ring_attention_single_key_and_rank_one_match_softmax_library():
    # one position in all: the output is that value row; R = 1 reduces to
    # scipy's softmax times V
    from scipy.special import softmax
    q, k, v = _attn_case(1, 2, 1, 4, 720)
    np.testing.assert_array_equal(O.ring_attention(q, k, v, True, 0.5)[0], v[0])
    q, k, v = _attn_case(1, 2, 6, 4, 730)
    Q, K, V = (O.bf16_to_f64(x[0]) for x in (q, k, v))
    want = np.einsum("hqk,hkd->hqd", softmax(0.5 * np.einsum("hqd,hkd->hqk", Q, K), axis=2), V)
    np.testing.assert_allclose(O.ring_attention(q, k, v, False, 0.5, out="f32")[0], want.astype(np.float32),
                               rtol=1e-6)


def test_ring_attention_rank_blocks_and_causal_mask_positions():
    # moving rank 1's keys/values away (zero logits cannot do it; use a huge
    # negative score instead) changes only rows that see them: with causal
    # masking, rank 0's queries never see rank 1's keys
    R, heads, s_r, d = 2, 1, 3, 4
    q, k, v = _attn_case(R, heads, s_r, d, 740)
    a = O.ring_attention(q, k, v, True, 0.3, out="f32")
    v2 = [v[0], bf(np.full((heads, s_r, d), 64.0))]
    b = O.ring_attention(q, k, v2, True, 0.3, out="f32")
    np.testing.assert_array_equal(a[0], b[0])          # rank 0 only sees its own block
    assert not np.array_equal(a[1], b[1])
    assert O.ring_order(0, 4) == [0, 3, 2, 1] and O.ring_order(3, 4) == [3, 2, 1, 0]


def test_norm_scale():
    assert O.norm_scale(16, 2.0, 0.5) == 4.0


# ---------------------------------------------------------------- stored oracle outputs

def test_golden_file_matches_oracle():
    import hashlib
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_golden.json")
    gold = json.load(open(path))
    w = I.RS_R2_256_INT
    a, b = I.gemm_inputs(w)
    blocks = O.gemm_rs([I.bits(x) for x in a], [I.bits(x) for x in b], out="f32")
    g = gold["rs_r2_256_int"]
    for o, blk in enumerate(blocks):
        assert hashlib.sha256(blk.tobytes()).hexdigest() == g["block_sha256_f32_le"][o]
    for o, i, j, v in g["samples"]:
        assert blocks[o][i, j] == v
    gm = gold["moe_small_route"]
    R, E_loc, T = 4, 4, 256
    logits = [I.zipf_logits(T, R * E_loc, 7000 + r).numpy() for r in range(R)]
    idx = [O.moe_route(lg, 2) for lg in logits]
    assert O.moe_counts(idx, R * E_loc).tolist() == gm["counts"]
