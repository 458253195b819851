"""Full-size parity (GPU): the AllGather+GEMM, GEMM+ReduceScatter and
GEMM+AllReduce workloads at their real sizes, run in the default launch
configuration that bench.py times, against the CPU oracle on a seeded row
sample (two rows per 128-row tile plus the first and last row, all columns).
The gathered A is compared in full.  Each workload's integer-valued twin
(values in {-2..2}, exact fp32 sums) must match bit for bit on the sample.
Every expected value comes from an oracle function that tests/test_oracle.py
pins.  Beside the normalised bar, the float bf16 outputs are held to at most
two bf16 ulps from the oracle's rounding of the exact result wherever |exact|
is at least 1/64 of its maximum (check_bf16_ulps); the combined MoE output,
a sum of rows each rounded to bf16 first, to the bound those roundings give.
The same holds for the fp8 AllGather+GEMM of the headline shape and for the
RS reduction variants (bf16 wire against the oracle's bf16-wire schedule,
atomic against the plain sum).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import inputs as I
from parity_util import TOL, absmax, check_bf16_ulps, gpu_bits, gpu_values, norm_err, oracle_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from comm_gemm_tile_gb300 import build
    build.build()
    torch.cuda.init()


def _ok(ws):
    st, detail = mk.device_status(ws)
    assert st == mk.MK_OK, (mk.status_string(st), detail)


@pytest.mark.parametrize("integer", [False, True])
def test_ag_full_size(integer):
    w = I.AG_R8_TP8_UP.integer_twin() if integer else I.AG_R8_TP8_UP
    a, b = I.gemm_inputs(w)
    ws = mk.Workspace()
    g, c = mk.ag_gemm([x.cuda() for x in a], b[0].cuda(), local_rank=w.local_rank, workspace=ws)
    _ok(ws)
    a_bits = [I.bits(x) for x in a]
    assert np.array_equal(I.bits(g), O.allgather_rows(a_bits))
    rows = I.sample_rows(w.R * w.m, seed=7)
    _, exact = O.ag_gemm(a_bits, I.bits(b[0]), out="f64", rows=rows)
    got = c[torch.from_numpy(rows).cuda()]
    if integer:
        np.testing.assert_array_equal(gpu_bits(got), oracle_bits(exact, "bf16"))
    else:
        assert norm_err(gpu_values(got), exact, w.k, absmax(a), absmax(b)) <= TOL["bf16"]
        print("AG full size: max bf16 ulps", check_bf16_ulps(gpu_bits(got), exact))


@pytest.mark.parametrize("integer", [False, True])
def test_rs_full_size(integer):
    w = I.RS_R8_TP8_DOWN.integer_twin() if integer else I.RS_R8_TP8_DOWN
    a, b = I.gemm_inputs(w)
    ws = mk.Workspace()
    blocks = mk.gemm_rs([x.cuda() for x in a], [x.cuda() for x in b], workspace=ws)
    _ok(ws)
    rows = I.sample_rows(w.m, seed=8)
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b], rows=rows)
    h = w.m // w.R
    got = torch.stack([blocks[r // h][r % h] for r in rows.tolist()], 0)
    if integer:
        np.testing.assert_array_equal(gpu_bits(got), oracle_bits(exact, "bf16"))
    else:
        assert norm_err(gpu_values(got), exact, w.R * w.k, absmax(a), absmax(b)) <= TOL["bf16"]
        print("RS full size: max bf16 ulps", check_bf16_ulps(gpu_bits(got), exact))


@pytest.mark.parametrize("integer", [False, True])
def test_ar_full_size(integer):
    w = I.AR_R8_DECODE.integer_twin() if integer else I.AR_R8_DECODE
    a, b = I.gemm_inputs(w)
    ws = mk.Workspace()
    reps = mk.gemm_ar([x.cuda() for x in a], [x.cuda() for x in b], workspace=ws)
    _ok(ws)
    exact = O.sum_over_ranks([I.bits(x) for x in a], [I.bits(x) for x in b])   # all 128 rows
    r0 = gpu_bits(reps[0])
    for r in reps[1:]:
        np.testing.assert_array_equal(gpu_bits(r), r0)
    if integer:
        np.testing.assert_array_equal(r0, oracle_bits(exact, "bf16"))
    else:
        assert norm_err(gpu_values(reps[0]), exact, w.R * w.k, absmax(a), absmax(b)) <= TOL["bf16"]
        print("AR full size: max bf16 ulps", check_bf16_ulps(r0, exact))


@pytest.mark.parametrize("integer", [False, True])
def test_moe_full_size(integer):
    # 8 ranks x 8 experts, 4096 tokens per rank, hidden 4096, up-proj 1536, top-2, Zipf(1.1)
    w = I.MOE_R8_E64.integer_twin() if integer else I.MOE_R8_E64
    x, logits, wexp = I.moe_inputs(w)
    ws = mk.Workspace()
    res = mk.moe_dispatch_gemm([t.cuda() for t in x], [t.cuda() for t in logits],
                               [t.cuda() for t in wexp], E_loc=w.E_loc, topk=w.topk,
                               cap_rows=w.cap, workspace=ws)
    _ok(ws)
    idx = [O.moe_route(l.numpy(), w.topk) for l in logits]
    np.testing.assert_array_equal(res["topk_idx"].cpu().numpy(), np.concatenate(idx, 0))
    np.testing.assert_array_equal(res["counts"].cpu().numpy(), O.moe_counts(idx, w.E))
    recv_src, seg = O.moe_dispatch(idx, w.E_loc)
    rc = res["recv_counts"].cpu().numpy()
    xb = [I.bits(t) for t in x]
    amax, bmax = absmax(x), absmax(wexp)
    for d in range(w.R):
        assert rc[d] == len(recv_src[d])
        np.testing.assert_array_equal(res["recv_src"][d][:rc[d]].cpu().numpy(), recv_src[d])
        if rc[d] == 0:
            continue
        rows = I.sample_rows(int(rc[d]), seed=100 + d)
        sel = torch.from_numpy(rows).cuda()
        rx = O.moe_gather_rows(xb, recv_src[d][rows], w.topk)
        np.testing.assert_array_equal(I.bits(res["recv_x"][d][sel]), rx)
        full_rx = O.moe_gather_rows(xb, recv_src[d], w.topk)
        exact = O.moe_expert_gemm(full_rx, seg[d], I.bits(wexp[d]), out="f64", rows=rows)
        got = res["y"][d][sel]
        if integer:
            np.testing.assert_array_equal(gpu_bits(got), oracle_bits(exact, "bf16"))
        else:
            assert norm_err(gpu_values(got), exact, w.H, amax, bmax) <= TOL["bf16"]
            print(f"MoE full size, rank {d}: max bf16 ulps", check_bf16_ulps(gpu_bits(got), exact))


@pytest.mark.parametrize("integer", [False, True])
def test_moe_combine_full_size(integer):
    # 8 ranks x 8 experts, 4096 tokens per rank, top-2 (Zipf 1.1), down-proj 1536 -> 4096
    w = I.MOE_COMBINE_R8_E64.integer_twin() if integer else I.MOE_COMBINE_R8_E64
    logits, h, w2, gates = I.combine_inputs(w)
    idx = [O.moe_route(l.numpy(), w.topk) for l in logits]
    counts = O.moe_counts(idx, w.E)
    recv_src, seg = O.moe_dispatch(idx, w.E_loc)
    rs_d = []
    for d in range(w.R):
        t = torch.zeros(w.cap, dtype=torch.int32)
        t[:len(recv_src[d])] = torch.from_numpy(recv_src[d].astype(np.int32))
        rs_d.append(t.cuda())
    ws = mk.Workspace()
    res = mk.moe_combine([t.cuda() for t in h], [t.cuda() for t in w2], [g.cuda() for g in gates],
                         rs_d, torch.from_numpy(counts.astype(np.int32)).cuda(), E_loc=w.E_loc,
                         topk=w.topk, cap_rows=w.cap, workspace=ws)
    _ok(ws)
    # where each (token, slot) landed: rank d and row j
    where = np.empty(w.R * w.T * w.topk, dtype=np.int64)
    for d in range(w.R):
        where[recv_src[d]] = d * w.cap + np.arange(len(recv_src[d]))
    seg = O.moe_seg_from_counts(counts, w.E_loc)
    amax, bmax = absmax(h), absmax(w2)
    for r in range(w.R):
        toks = I.sample_rows(w.T, seed=300 + r)
        g = r * w.T + toks
        # the returned rows of the sampled tokens: each slot's expert row from the oracle's
        # grouped GEMM (rounded to bf16, the expert output), gathered per rank
        ret = np.zeros((len(toks), w.topk, w.H), dtype=np.uint16)
        for k in range(w.topk):
            loc = where[g * w.topk + k]
            for d in np.unique(loc // w.cap):
                pick = np.nonzero(loc // w.cap == d)[0]
                hd = I.bits(h[d][:int(np.sum(seg[d]))])
                ret[pick, k] = O.moe_expert_gemm(hd, seg[d], I.bits(w2[d]), out="bf16",
                                                 rows=loc[pick] - d * w.cap)
        gt = gates[r].numpy()[toks]
        sel = torch.from_numpy(toks).cuda()
        got_ret, got_out = res["ret"][r][sel], res["out"][r][sel]
        if integer:
            np.testing.assert_array_equal(gpu_bits(got_ret), ret)
            np.testing.assert_array_equal(gpu_bits(got_out), O.moe_weighted_sum(ret, gt, "bf16"))
        else:
            exact_out = O.moe_weighted_sum(ret, gt, "f64")
            assert norm_err(gpu_values(got_ret).reshape(len(toks), -1),
                            O.bf16_to_f64(ret).reshape(len(toks), -1), w.N, amax, bmax) <= TOL["bf16"]
            assert norm_err(gpu_values(got_out), exact_out, w.N, amax, bmax) <= TOL["bf16"]
            print(f"combine full size, rank {r}: max bf16 ulps of the returned rows",
                  check_bf16_ulps(gpu_bits(got_ret).reshape(len(toks), -1),
                                  O.bf16_to_f64(ret).reshape(len(toks), -1)))
            # The output sums rows that were each rounded to bf16 on their own: a row
            # that sits an ulp or two from the oracle's (checked just above, <= 2^-6 of
            # the row value) shifts the sum by up to that much times its gate, which a
            # cancelling sum does not shrink.  Bound per element: 2^-6 sum_k g_k |row_k|
            # plus one bf16 ulp of the result (<= 2^-7 |exact|).
            cond = np.einsum("tk,tkh->th", np.abs(gt.astype(np.float64)), np.abs(O.bf16_to_f64(ret)))
            err = np.abs(gpu_values(got_out) - exact_out)
            assert np.all(err <= 2.0 ** -6 * cond + 2.0 ** -7 * np.abs(exact_out) + 1e-30)


@pytest.mark.parametrize("integer", [False, True])
def test_ag_fp8_full_size(integer):
    # the headline shape with fp8 e4m3 operands (B as B^T), default launch configuration
    w = I.AG_R8_TP8_UP.integer_twin() if integer else I.AG_R8_TP8_UP
    w = dataclasses.replace(w, b_std=1.0)
    a, bt = I.gemm_inputs_fp8(w)
    ws = mk.Workspace()
    g, c = mk.ag_gemm([x.cuda() for x in a], bt[0].cuda(), local_rank=w.local_rank, workspace=ws)
    _ok(ws)
    a_bytes = [I.fp8_bytes(x) for x in a]
    assert np.array_equal(I.fp8_bytes(g), np.concatenate(a_bytes, 0))
    rows = I.sample_rows(w.R * w.m, seed=17)
    _, exact = O.ag_gemm_fp8(a_bytes, I.fp8_bytes(bt[0]), "f64", rows=rows)
    got = c[torch.from_numpy(rows).cuda()]
    if integer:
        np.testing.assert_array_equal(gpu_bits(got), oracle_bits(exact, "bf16"))
    else:
        amax = max(float(x.float().abs().max()) for x in a)
        assert norm_err(gpu_values(got), exact, w.k, amax, float(bt[0].float().abs().max())) <= TOL["bf16"]


@pytest.mark.parametrize("variant", ["wire", "atomic"])
def test_rs_reduction_variants_full_size(variant):
    # integer twin: the atomic sum is exact in any order; the bf16 wire follows the oracle's schedule
    w = I.RS_R8_TP8_DOWN.integer_twin()
    a, b = I.gemm_inputs(w)
    ws = mk.Workspace()
    cfg = mk.Config(wire=mk.WIRE_BF16) if variant == "wire" else mk.Config(reduce=mk.REDUCE_ATOMIC)
    blocks = mk.gemm_rs([x.cuda() for x in a], [x.cuda() for x in b], workspace=ws, cfg=cfg)
    _ok(ws)
    rows = I.sample_rows(w.m, seed=18)
    h = w.m // w.R
    got = torch.stack([blocks[r // h][r % h] for r in rows.tolist()], 0)
    a_bits, b_bits = [I.bits(x) for x in a], [I.bits(x) for x in b]
    if variant == "atomic":
        want = oracle_bits(O.sum_over_ranks(a_bits, b_bits, rows=rows), "bf16")
    else:
        want = O.running_sum_bf16_wire(O.rank_partials(a_bits, b_bits, rows=rows), "bf16")
    np.testing.assert_array_equal(gpu_bits(got), want)
