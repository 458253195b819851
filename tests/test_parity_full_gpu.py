"""Full-size parity (GPU): the AllGather+GEMM, GEMM+ReduceScatter and
GEMM+AllReduce workloads at their real sizes, run in the default launch
configuration that bench.py times, against the CPU oracle on a seeded row
sample (two rows per 128-row tile plus the first and last row, all columns).
The gathered A is compared in full.  Each workload's integer-valued twin
(values in {-2..2}, exact fp32 sums) must match bit for bit on the sample.
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
from parity_util import TOL, absmax, gpu_bits, gpu_values, norm_err, oracle_bits

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
    exact = O.bf16_to_f64(O.allgather_rows(a_bits)[rows]) @ O.bf16_to_f64(I.bits(b[0]))
    got = c[torch.from_numpy(rows).cuda()]
    if integer:
        np.testing.assert_array_equal(gpu_bits(got), oracle_bits(exact, "bf16"))
    else:
        assert norm_err(gpu_values(got), exact, w.k, absmax(a), absmax(b)) <= TOL["bf16"]


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
        starts = np.concatenate([[0], np.cumsum(seg[d])])
        expert_of = np.searchsorted(starts, rows, side="right") - 1
        exact = np.zeros((len(rows), w.N))
        wb = I.bits(wexp[d])
        for l in np.unique(expert_of):
            pick = np.nonzero(expert_of == l)[0]
            exact[pick] = O.bf16_to_f64(full_rx[rows[pick]]) @ O.bf16_to_f64(wb[l])
        got = res["y"][d][sel]
        if integer:
            np.testing.assert_array_equal(gpu_bits(got), oracle_bits(exact, "bf16"))
        else:
            assert norm_err(gpu_values(got), exact, w.H, amax, bmax) <= TOL["bf16"]


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
    idx_all = np.concatenate(idx, 0)
    amax, bmax = absmax(h), absmax(w2)
    for r in range(w.R):
        toks = I.sample_rows(w.T, seed=300 + r)
        g = r * w.T + toks
        y2 = np.zeros((len(toks), w.topk, w.H))
        for k in range(w.topk):
            e = idx_all[g, k]
            loc = where[g * w.topk + k]
            for ex in np.unique(e):                     # one product per expert used
                pick = np.nonzero(e == ex)[0]
                d, l = divmod(int(ex), w.E_loc)
                rows = loc[pick] - d * w.cap
                hb = O.bf16_to_f64(I.bits(h[d][torch.from_numpy(rows)]))
                y2[pick, k] = O.bf16_to_f64(O.f64_to_bf16_bits(hb @ O.bf16_to_f64(I.bits(w2[d][l]))))
        gt = gates[r].numpy().astype(np.float64)[toks]
        exact_out = np.einsum("tk,tkh->th", gt, y2)
        sel = torch.from_numpy(toks).cuda()
        got_ret, got_out = res["ret"][r][sel], res["out"][r][sel]
        if integer:
            np.testing.assert_array_equal(gpu_bits(got_ret), O.f64_to_bf16_bits(y2))
            np.testing.assert_array_equal(gpu_bits(got_out), oracle_bits(exact_out, "bf16"))
        else:
            assert norm_err(gpu_values(got_ret).reshape(len(toks), -1), y2.reshape(len(toks), -1),
                            w.N, amax, bmax) <= TOL["bf16"]
            assert norm_err(gpu_values(got_out), exact_out, w.N, amax, bmax) <= TOL["bf16"]


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
    exact = O.e4m3_to_f64(np.concatenate(a_bytes, 0)[rows]) @ O.e4m3_to_f64(I.fp8_bytes(bt[0])).T
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
        parts = [O.bf16_to_f64(x[rows]) @ O.bf16_to_f64(y) for x, y in zip(a_bits, b_bits)]
        want = O.running_sum_bf16_wire(parts, "bf16")
    np.testing.assert_array_equal(gpu_bits(got), want)
