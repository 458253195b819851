"""CPU oracle for the fused collective + GEMM ops -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or call this module.  The
product path (the CUDA library and its Python binding) never does, and shares
no code with it.

What it computes is the plain definition of each fused op, written out with
numpy in float64:

* bf16 inputs are widened exactly to float64 (a bf16 value has 8 significant
  bits, so every product of two of them is exact in float64 and every sum
  used here carries at most float64 rounding, ~1e-16 relative);
* contractions use ``np.matmul`` on float64 as the one library step;
* the result is rounded ONCE to the output type: round-to-nearest-even to bf16
  (``f64_to_bf16_bits``) or to fp32 (numpy's IEEE cast).

The ops (mKernel write-up, news.chathome.org, "五种融合内核" table):

* AllGather + GEMM (table row "AllGather + GEMM"): each rank holds one row
  shard of A; the gathered A is the shards stacked in rank order and
  C = gather(A) @ B.
* GEMM + ReduceScatter (row "GEMM + ReduceScatter"): S = sum_r A_r @ B_r;
  row block o of S (rows [o*m/R, (o+1)*m/R)) belongs to rank o.
* GEMM + AllReduce (row "GEMM + AllReduce"): S as above, and every rank ends
  with all of S.  One reduction variant has a result of its own:
  ``running_sum_bf16_wire`` (the running sum forwarded in bf16); the atomic
  variant's result is S itself, up to fp32 rounding in an unfixed order.
* MoE Dispatch + GEMM (row "MoE Dispatch + GEMM"): route each token to its
  top-k experts, move each (token, expert) row to the rank that holds the
  expert, then multiply the rows of each expert by that expert's weight.
  The pages leave the gating, tie-breaking and row order open; the readings
  used here are: top-k on the raw logits (largest first, ties to the lower
  expert id), expert e lives on rank e // E_loc, and the rows that rank d
  receives are ordered by (local expert, global token id g = r*T + t).
* Chained MLP (the roadmap's multi-step kernel, built from the rows
  "AllGather + GEMM" and "GEMM + ReduceScatter"): X = gather(X_r); every rank
  r computes H_r = bf16(ReLU(X @ W1_r)) with its column shard W1_r, then
  S = sum_r H_r @ W2_r with its row shard W2_r, and rank o keeps row block o
  of S.  The pages name no activation; ReLU is the reading used (exact, so
  the integer twins stay bit-exact), and H_r is rounded to bf16 as the
  layer's stored activation.
* Ring Attention (row "Ring Attention"): every rank holds one contiguous
  block of the sequence's Q, K and V; the K/V blocks travel around the ring
  and each rank attends its queries to all of them, merging the partial
  softmax results as the blocks arrive.  The result is plain (optionally
  causal) softmax attention over the whole sequence, computed here directly.
* MoE combine, the step after the same row: the expert rows are multiplied
  by each expert's down-projection, the products (rounded to bf16, the
  expert output) return to the token's source rank, and each token's output
  is the gate-weighted sum of its top-k returned rows.  The pages do not
  describe combine; its readings: the gate weights are an input (fp32,
  [T x topk] per source rank), and the weighted sum is exact, rounded once.

Pins: every function here is checked in ``tests/test_oracle.py`` against
brute force on tiny inputs, closed forms, invariants, and special cases that
reduce to a library routine.  Nothing in this file is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# bf16 <-> float64
# ----------------------------------------------------------------------------


def bf16_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of raw bf16 bit patterns (uint16) to float64.

    A bf16 value is the top half of an IEEE binary32 value, so shifting the
    16 bits up by 16 gives that binary32 exactly; binary32 -> binary64 is exact.
    """
    b = np.asarray(b, dtype=np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


_BF16_MIN_QUANTUM_EXP = -133   # bf16 subnormal spacing 2**-133 (2**-126 * 2**-7)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 with round-to-nearest, ties-to-even, once.

    bf16 keeps 8 significant bits.  For |x| in [2**(e-1), 2**e) the spacing of
    bf16 values is 2**(e-8); below the normal range (2**-126) the spacing stays
    2**-133.  Dividing by the spacing, rounding to the nearest integer with
    ties to even (``np.rint``) and scaling back is the textbook definition.
    Results at or beyond 2**128 overflow to +-inf; NaN stays NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(x)
        q = np.maximum(e.astype(np.int64) - 8, _BF16_MIN_QUANTUM_EXP)
        r = np.ldexp(np.rint(np.ldexp(x, -q)), q)
        r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, x), r)
        r = np.where(np.isnan(x), np.nan, r)
        f32 = r.astype(np.float32)            # exact: r has <= 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def round_out(x: np.ndarray, out: str) -> np.ndarray:
    """Round an exact float64 result to the output dtype: 'bf16' -> uint16
    bit patterns, 'f32' -> float32 values.  'f64' leaves the float64 result
    unrounded (the value the float parity bar measures errors against)."""
    if out == "bf16":
        return f64_to_bf16_bits(x)
    if out == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32)
    if out == "f64":
        return np.asarray(x, dtype=np.float64)
    raise ValueError(f"unknown output dtype {out!r}")


# ----------------------------------------------------------------------------
# AllGather + GEMM
# ----------------------------------------------------------------------------


def allgather_rows(a_shards) -> np.ndarray:
    """The gathered A: the row shards stacked in rank order r = 0..R-1
    (a bit copy; the order in which shards travel does not change it)."""
    return np.concatenate([np.asarray(a, dtype=np.uint16) for a in a_shards], axis=0)


def ag_gemm(a_shards, b, out: str = "bf16", rows=None):
    """C = gather_r(A_r) @ B.

    a_shards: R arrays of bf16 bits, each [m_r x k]; b: [k x n] bf16 bits.
    rows: optional index array of gathered rows to compute (row sample).
    Returns (gathered A bits [R*m_r x k], C rounded to `out` [len(rows) x n]).
    """
    gathered = allgather_rows(a_shards)
    a_sel = gathered if rows is None else gathered[np.asarray(rows)]
    c = bf16_to_f64(a_sel) @ bf16_to_f64(b)
    return gathered, round_out(c, out)


# ----------------------------------------------------------------------------
# GEMM + ReduceScatter / GEMM + AllReduce
# ----------------------------------------------------------------------------


def sum_over_ranks(a_list, b_list, rows=None) -> np.ndarray:
    """S = sum_r A_r @ B_r in float64 (rows: optional sample of S's rows)."""
    assert len(a_list) == len(b_list) and len(a_list) >= 1
    s = None
    for a, b in zip(a_list, b_list):
        a_sel = np.asarray(a) if rows is None else np.asarray(a)[np.asarray(rows)]
        p = bf16_to_f64(a_sel) @ bf16_to_f64(b)
        s = p if s is None else s + p
    return s


def owner_rows(m: int, R: int, o: int) -> range:
    """Rows of S owned by rank o after the reduce-scatter: the o-th of R
    contiguous row blocks (m must be a multiple of R)."""
    if m % R:
        raise ValueError("m must be a multiple of R for a row-block reduce-scatter")
    h = m // R
    return range(o * h, (o + 1) * h)


def gemm_rs(a_list, b_list, out: str = "bf16"):
    """GEMM + ReduceScatter: returns R row blocks; block o = rows owner_rows(o) of S."""
    s = sum_over_ranks(a_list, b_list)
    R, m = len(a_list), s.shape[0]
    blocks = []
    for o in range(R):
        rr = owner_rows(m, R, o)
        blocks.append(round_out(s[rr.start:rr.stop], out))
    return blocks


def gemm_ar(a_list, b_list, out: str = "bf16"):
    """GEMM + AllReduce: returns R replicas, each equal to all of S."""
    c = round_out(sum_over_ranks(a_list, b_list), out)
    return [c.copy() for _ in range(len(a_list))]


def rank_partials(a_list, b_list, rows=None) -> list:
    """The terms of S: P_r = A_r @ B_r in float64, one per rank, in rank order
    (table row "GEMM + ReduceScatter": each rank's partial product).
    rows: optional sample of S's rows (every partial restricted to them)."""
    assert len(a_list) == len(b_list) and len(a_list) >= 1
    sel = (lambda a: np.asarray(a)) if rows is None else (lambda a: np.asarray(a)[np.asarray(rows)])
    return [bf16_to_f64(sel(a)) @ bf16_to_f64(np.asarray(b)) for a, b in zip(a_list, b_list)]


def f64_to_f32(x) -> np.ndarray:
    """Round float64 to the nearest fp32 (ties to even) and widen back, exactly."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def running_sum_bf16_wire(partials, out: str = "bf16") -> np.ndarray:
    """S = sum of the partials, reduced as a running sum forwarded from part to
    part with bf16 on the wire (the reduction variant that halves the partial
    traffic of "GEMM + ReduceScatter" / "GEMM + AllReduce").

    The pages fix no dtype for the partials in flight; the reading used for this
    variant: every part holds its own partial in fp32, adds the bf16 sum it
    received in one fp32 addition, and forwards that sum rounded to bf16
    (nearest, ties to even); the last part rounds once to the output dtype:

        s_0 = bf16(f32(P_0)),  s_j = bf16(f32(s_{j-1} + f32(P_j))) for 0 < j < P-1,
        result = round_out(f32(s_{P-2} + f32(P_{P-1})))      (P = 1: round_out(P_0)).
    """
    parts = [np.asarray(x, dtype=np.float64) for x in partials]
    if len(parts) == 1:
        return round_out(parts[0], out)
    s = bf16_to_f64(f64_to_bf16_bits(f64_to_f32(parts[0])))
    for x in parts[1:-1]:
        s = bf16_to_f64(f64_to_bf16_bits(f64_to_f32(s + f64_to_f32(x))))
    return round_out(f64_to_f32(s + f64_to_f32(parts[-1])), out)


# ----------------------------------------------------------------------------
# fp8 operands (the e4m3 variant of AllGather + GEMM, GEMM + ReduceScatter /
# AllReduce).  The write-up names fp8 only as a capability of the GB300 rack
# (first section, "问题：主机驱动通信", point (1)); the format is the OCP 8-bit
# e4m3 encoding: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
# exponent field 0 for subnormals (m/8 * 2^-6), no infinities, and S.1111.111
# the only NaN (largest finite value 448).  Reading used for the operand
# layout: B is given as its transpose B^T [n x k] (both operands K-major).
# ----------------------------------------------------------------------------


def e4m3_to_f64(b) -> np.ndarray:
    """Exact value of raw e4m3 bytes (uint8) as float64."""
    b = np.asarray(b, dtype=np.uint8)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = ((b >> 3) & 0x0F).astype(np.int64)
    m = (b & 0x07).astype(np.float64)
    val = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    val = sign * val
    return np.where((b & 0x7F) == 0x7F, np.nan, val)


def ag_gemm_fp8(a_shards, b_t, out: str = "bf16", rows=None):
    """C = gather_r(A_r) @ B with fp8 operands: a_shards R arrays of e4m3
    bytes [m_r x k], b_t the bytes of B^T [n x k].  Returns (gathered bytes,
    C rounded to `out`)."""
    gathered = np.concatenate([np.asarray(a, dtype=np.uint8) for a in a_shards], axis=0)
    a_sel = gathered if rows is None else gathered[np.asarray(rows)]
    c = e4m3_to_f64(a_sel) @ e4m3_to_f64(b_t).T
    return gathered, round_out(c, out)


def sum_over_ranks_fp8(a_list, bt_list, rows=None) -> np.ndarray:
    """S = sum_r A_r @ B_r in float64, fp8 operands (bt_list: the bytes of B_r^T)."""
    assert len(a_list) == len(bt_list) and len(a_list) >= 1
    s = None
    for a, bt in zip(a_list, bt_list):
        a_sel = np.asarray(a) if rows is None else np.asarray(a)[np.asarray(rows)]
        p = e4m3_to_f64(a_sel) @ e4m3_to_f64(bt).T
        s = p if s is None else s + p
    return s


# ----------------------------------------------------------------------------
# MoE dispatch + grouped GEMM
# ----------------------------------------------------------------------------


def moe_route(logits: np.ndarray, topk: int) -> np.ndarray:
    """Top-k experts of each token: largest logit first, ties to the lower
    expert id.  logits: [T x E] float32 (no NaN).  Returns int32 [T x topk].

    Written as k rounds of "take the best expert not taken yet": each round
    scans the experts in id order and replaces the running best only on a
    strictly larger value, so the lower id wins a tie (a -inf logit is still
    a valid pick when nothing larger is left).
    """
    work = np.asarray(logits, dtype=np.float64)
    T, E = work.shape
    if not 1 <= topk <= E:
        raise ValueError("need 1 <= topk <= E")
    taken = np.zeros((T, E), dtype=bool)
    out = np.empty((T, topk), dtype=np.int32)
    rows = np.arange(T)
    for j in range(topk):
        best_idx = np.full(T, -1, dtype=np.int64)
        best_val = np.zeros(T, dtype=np.float64)
        for e in range(E):
            better = ~taken[:, e] & ((best_idx < 0) | (work[:, e] > best_val))
            best_val = np.where(better, work[:, e], best_val)
            best_idx = np.where(better, e, best_idx)
        out[:, j] = best_idx
        taken[rows, best_idx] = True
    return out


def moe_counts(topk_idx_list, E: int) -> np.ndarray:
    """counts[r][e] = number of (token, slot) pairs of source rank r routed to e."""
    counts = np.zeros((len(topk_idx_list), E), dtype=np.int64)
    for r, idx in enumerate(topk_idx_list):
        for e in np.asarray(idx).reshape(-1):
            counts[r, int(e)] += 1
    return counts


def moe_dispatch(topk_idx_list, E_loc: int):
    """The all-to-all token permutation.

    topk_idx_list: R arrays [T x topk] (expert ids of rank r's tokens).
    Expert e is held by rank e // E_loc.  Rank d receives every (token, slot)
    pair routed to one of its experts, ordered by local expert, then by global
    token id g = r*T + t.  Returns (recv_src, seg) where recv_src[d] is an
    int64 array of g*topk + slot per received row, and seg[d][l] is the number
    of rows of local expert l on rank d.
    """
    R = len(topk_idx_list)
    idx_all = np.concatenate([np.asarray(i) for i in topk_idx_list], axis=0)   # [R*T x topk]
    topk = idx_all.shape[1]
    recv_src, seg = [], []
    for d in range(R):
        src_d, seg_d = [], []
        for l in range(E_loc):
            e = d * E_loc + l
            g, j = np.nonzero(idx_all == e)      # row-major: g ascending
            src_d.append(g.astype(np.int64) * topk + j)
            seg_d.append(len(g))
        recv_src.append(np.concatenate(src_d) if src_d else np.zeros(0, np.int64))
        seg.append(np.asarray(seg_d, dtype=np.int64))
    return recv_src, seg


def moe_gather_rows(x_list, recv_src_d, topk: int) -> np.ndarray:
    """recv_x rows of one destination rank: bit copies of the source token rows."""
    x_all = np.concatenate([np.asarray(x, dtype=np.uint16) for x in x_list], axis=0)
    g = np.asarray(recv_src_d, dtype=np.int64) // topk
    return x_all[g]


def moe_expert_gemm(recv_x_d, seg_d, w_d, out: str = "bf16", rows=None):
    """Grouped GEMM of one destination rank: the rows of local expert l
    (the l-th segment) times W_l.  w_d: [E_loc x H x N] bf16 bits.
    rows: optional sample of received row indices.  Returns rounded [rows x N]."""
    seg_d = np.asarray(seg_d, dtype=np.int64)
    starts = np.concatenate([[0], np.cumsum(seg_d)])
    nrows = int(starts[-1])
    sel = np.arange(nrows) if rows is None else np.asarray(rows, dtype=np.int64)
    N = np.asarray(w_d).shape[2]
    y = np.zeros((len(sel), N), dtype=np.float64)
    expert_of = np.searchsorted(starts, sel, side="right") - 1
    for l in range(len(seg_d)):
        pick = np.nonzero(expert_of == l)[0]
        if len(pick):
            y[pick] = bf16_to_f64(np.asarray(recv_x_d)[sel[pick]]) @ bf16_to_f64(np.asarray(w_d)[l])
    return round_out(y, out)


def moe_dispatch_gemm(x_list, logits_list, w_list, E_loc: int, topk: int, out: str = "bf16"):
    """The whole MoE path for all ranks: route, count, dispatch, grouped GEMM."""
    topk_idx = [moe_route(lg, topk) for lg in logits_list]
    counts = moe_counts(topk_idx, len(x_list) * E_loc)
    recv_src, seg = moe_dispatch(topk_idx, E_loc)
    recv_x = [moe_gather_rows(x_list, recv_src[d], topk) for d in range(len(x_list))]
    y = [moe_expert_gemm(recv_x[d], seg[d], w_list[d], out) for d in range(len(x_list))]
    return dict(topk_idx=topk_idx, counts=counts, recv_src=recv_src, seg=seg, recv_x=recv_x, y=y)


def moe_seg_from_counts(counts, E_loc: int):
    """seg[d][l]: rows that rank d holds for its local expert l, i.e. the
    total over source ranks of counts[:, d*E_loc + l]."""
    counts = np.asarray(counts, dtype=np.int64)
    R = counts.shape[0]
    tot = counts.sum(axis=0)
    return [tot[d * E_loc:(d + 1) * E_loc].copy() for d in range(R)]


def moe_return_rows(y2_list, recv_src_list, topk: int, T: int, R: int):
    """The return all-to-all of MoE combine: row j of destination rank d came
    from (token g, slot k) with recv_src[d][j] = g*topk + k; it goes back to
    source rank r = g // T at ret[r][t, k] (t = g % T).  Returns R arrays
    [T x topk x H] of bf16 bits; every (r, t, k) must be covered exactly once."""
    H = None
    for y in y2_list:
        if np.asarray(y).ndim == 2 and np.asarray(y).shape[0] > 0:
            H = np.asarray(y).shape[1]
    H = 0 if H is None else H
    ret = [np.zeros((T, topk, H), dtype=np.uint16) for _ in range(R)]
    seen = [np.zeros((T, topk), dtype=np.int64) for _ in range(R)]
    for d in range(R):
        src = np.asarray(recv_src_list[d], dtype=np.int64)
        y = np.asarray(y2_list[d], dtype=np.uint16)
        for j, s_ in enumerate(src.tolist()):
            g, k = divmod(s_, topk)
            r, t = divmod(g, T)
            ret[r][t, k] = y[j]
            seen[r][t, k] += 1
    for r in range(R):
        if not np.all(seen[r] == 1):
            raise ValueError("the received rows do not cover every (token, slot) exactly once")
    return ret


def moe_weighted_sum(ret_r, gates_r, out: str = "bf16"):
    """Combine of one source rank: out[t] = sum_k gates[t, k] * ret[t, k], the
    slot rows widened exactly, the sum exact in float64, rounded once."""
    ret64 = bf16_to_f64(np.asarray(ret_r, dtype=np.uint16))            # [T x topk x H]
    g = np.asarray(gates_r, dtype=np.float64)                           # [T x topk]
    return round_out(np.einsum("tk,tkh->th", g, ret64), out)


def moe_combine(h_list, recv_src_list, counts, w2_list, gates_list, E_loc: int, topk: int,
                T: int, out: str = "bf16"):
    """MoE combine, the step after dispatch + up-projection: each destination
    rank multiplies the rows of local expert l by that expert's down-projection
    W2_l (rounded to bf16: the expert output), the rows return to their source
    ranks (slot k of token t), and every token's output is the gate-weighted
    sum of its top-k returned rows.

    h_list[d]: [>= rows_d x N] bf16 bits (the expert hidden rows, in the order
    the dispatch delivered them); recv_src_list[d]: g*topk + k per row;
    counts: [R x E] (source rank x expert) from the dispatch; w2_list[d]:
    [E_loc x N x H] bf16 bits; gates_list[r]: [T x topk] fp32.
    Returns dict(y2=[per d: rows_d x H bits], ret=[per r: T x topk x H bits],
    out=[per r: T x H])."""
    R = len(h_list)
    seg = moe_seg_from_counts(counts, E_loc)
    y2 = []
    for d in range(R):
        n = int(np.sum(seg[d]))
        y2.append(moe_expert_gemm(np.asarray(h_list[d])[:n], seg[d], w2_list[d], "bf16"))
    ret = moe_return_rows(y2, recv_src_list, topk, T, R)
    res = [moe_weighted_sum(ret[r], gates_list[r], out) for r in range(R)]
    return dict(y2=y2, ret=ret, out=res)


def mlp_hidden(x_shards, w1_r, rows=None) -> np.ndarray:
    """Up-projection of one rank in the tensor-parallel MLP: the gathered input
    times the rank's column shard W1_r, ReLU, rounded once to bf16 (bits).
    rows: optional sample of the gathered rows (each hidden row depends only
    on the input row of the same index)."""
    xg = allgather_rows(x_shards)
    if rows is not None:
        xg = xg[np.asarray(rows, dtype=np.int64)]
    h = bf16_to_f64(xg) @ bf16_to_f64(np.asarray(w1_r, dtype=np.uint16))
    return f64_to_bf16_bits(np.maximum(h, 0.0))


def mlp_ag_rs(x_shards, w1_list, w2_list, out: str = "bf16", rows=None):
    """Tensor-parallel MLP over R ranks, the chained AllGather+GEMM -> ReLU ->
    GEMM+ReduceScatter layer: X = gather_r(X_r) (rank order); H_r =
    bf16(ReLU(X @ W1_r)); S = sum_r H_r @ W2_r; rank o receives rows
    [o*m, (o+1)*m) of S (m = rows per shard), rounded once.
    rows: optional sample of S's rows (then hidden holds those rows only and
    the result is dict(gathered, hidden, rows=S rows rounded)).
    Returns dict(gathered=bits, hidden=[H_r bits], blocks=[per rank o])."""
    R = len(x_shards)
    m = np.asarray(x_shards[0]).shape[0]
    gathered = allgather_rows(x_shards)
    hidden = [mlp_hidden(x_shards, w1_list[r], rows) for r in range(R)]
    s = sum(bf16_to_f64(hidden[r]) @ bf16_to_f64(np.asarray(w2_list[r], dtype=np.uint16))
            for r in range(R))
    if rows is not None:   # hidden holds the sampled rows only
        return dict(gathered=gathered, hidden=hidden, rows=round_out(s, out))
    blocks = [round_out(s[o * m:(o + 1) * m], out) for o in range(R)]
    return dict(gathered=gathered, hidden=hidden, blocks=blocks)


def ring_order(r: int, R: int):
    """The KV blocks rank r sees in a ring: its own first, then the block of
    rank r-1, r-2, ... (each step passes every block one rank forward)."""
    return [(r - j) % R for j in range(R)]


def ring_attention(q_list, k_list, v_list, causal: bool, scale: float, out: str = "bf16",
                   q_rows=None):
    """Ring attention over R ranks that each hold a contiguous block of the
    sequence (rank s: positions [s*S_r, (s+1)*S_r)) for every head.
    q_list[r], k_list[r], v_list[r]: [heads x S_r x d] bf16 bits.
    O_r = softmax(scale * Q_r @ K^T + mask) @ V for the whole sequence's K, V
    (mask: -inf where the key position is after the query position when
    causal).  The ring only fixes the order in which the blocks arrive; the
    result is the plain attention, computed here in float64 with the
    row-wise maximum subtracted, rounded once.  Returns R arrays.
    q_rows: optional per-rank arrays of query positions within the rank's
    block (a row sample); then only those rows are returned."""
    R = len(q_list)
    k = np.concatenate([bf16_to_f64(np.asarray(x, dtype=np.uint16)) for x in k_list], axis=1)
    v = np.concatenate([bf16_to_f64(np.asarray(x, dtype=np.uint16)) for x in v_list], axis=1)
    outs = []
    for r in range(R):
        q = bf16_to_f64(np.asarray(q_list[r], dtype=np.uint16))          # [heads x S_r x d]
        s_r = q.shape[1]
        rows = np.arange(s_r) if q_rows is None else np.asarray(q_rows[r], dtype=np.int64)
        q = q[:, rows]
        logits = scale * np.einsum("hqd,hkd->hqk", q, k)
        if causal:
            qpos = r * s_r + rows[:, None]
            kpos = np.arange(k.shape[1])[None, :]
            logits = np.where(kpos <= qpos, logits, -np.inf)
        mx = logits.max(axis=2, keepdims=True)
        w = np.exp(logits - mx)
        w = w / w.sum(axis=2, keepdims=True)
        outs.append(round_out(np.einsum("hqk,hkd->hqd", w, v), out))
    return outs


# ----------------------------------------------------------------------------
# tolerance used for float parity
# ----------------------------------------------------------------------------


def norm_scale(K: int, a_absmax: float, b_absmax: float) -> float:
    """Error normaliser sqrt(K) * max|a| * max|b| (K = contraction length)."""
    return float(np.sqrt(K) * a_absmax * b_absmax)
