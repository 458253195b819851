"""MoE dispatch + grouped GEMM: CUDA path vs the CPU oracle (GPU).

Routing (top-k ids), counts, the dispatch permutation (recv_src, recv_counts)
and the received rows must match bit for bit; the expert outputs y match bit
for bit on integer-valued inputs and within the normalised tolerance on
float inputs.
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
from parity_util import TOL, absmax, gpu_bits, gpu_values, norm_err, oracle_bits

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def built():
    from comm_gemm_tile_gb300 import build
    build.build()
    torch.cuda.init()


def run_both(w, cfg=None):
    x, logits, wexp = I.moe_inputs(w)
    ws = mk.Workspace()
    res = mk.moe_dispatch_gemm([t.cuda() for t in x], [t.cuda() for t in logits],
                               [t.cuda() for t in wexp], E_loc=w.E_loc, topk=w.topk,
                               cap_rows=w.cap, cfg=cfg, workspace=ws)
    st, detail = mk.device_status(ws)
    return x, logits, wexp, res, st, detail


def check_dispatch(w, x, logits, res):
    xb = [I.bits(t) for t in x]
    idx = [O.moe_route(l.numpy(), w.topk) for l in logits]
    np.testing.assert_array_equal(res["topk_idx"].cpu().numpy(), np.concatenate(idx, 0))
    counts = O.moe_counts(idx, w.E)
    np.testing.assert_array_equal(res["counts"].cpu().numpy(), counts)
    recv_src, seg = O.moe_dispatch(idx, w.E_loc)
    rc = res["recv_counts"].cpu().numpy()
    for d in range(w.R):
        assert rc[d] == len(recv_src[d])
        np.testing.assert_array_equal(res["recv_src"][d][:rc[d]].cpu().numpy(), recv_src[d])
        np.testing.assert_array_equal(I.bits(res["recv_x"][d][:rc[d]]),
                                      O.moe_gather_rows(xb, recv_src[d], w.topk))
    return recv_src, seg


SMALL = [  # R, E_loc, T, H, N
    (2, 2, 100, 64, 256),
    (4, 3, 257, 520, 264),
    (8, 8, 64, 128, 512),
    (1, 4, 300, 256, 256),
]


@pytest.mark.parametrize("pair", [mk.PAIR_OFF, mk.PAIR_ON])
@pytest.mark.parametrize("R,E_loc,T,H,N", SMALL)
def test_moe_integer_bit_exact(R, E_loc, T, H, N, pair):
    # pairs: 256-row tiles of each expert's rows, one 128-row half per CTA
    w = I.MoeWorkload("t", R=R, E_loc=E_loc, T=T, H=H, N=N, integer=True, x_seed=31,
                      logit_seed=41, w_seed=51)
    x, logits, wexp, res, st, detail = run_both(w, cfg=mk.Config(cta_pair=pair))
    assert st == mk.MK_OK, (mk.status_string(st), detail)
    recv_src, seg = check_dispatch(w, x, logits, res)
    xb = [I.bits(t) for t in x]
    for d in range(R):
        rx = O.moe_gather_rows(xb, recv_src[d], w.topk)
        want = O.moe_expert_gemm(rx, seg[d], I.bits(wexp[d]), out="bf16")
        np.testing.assert_array_equal(gpu_bits(res["y"][d][:len(recv_src[d])]), want)


@pytest.mark.parametrize("mode", [mk.MODE_FUSED, mk.MODE_UNFUSED])
@pytest.mark.parametrize("R,E_loc,T,topk", [(2, 3, 200, 1), (4, 2, 150, 3), (2, 4, 130, 8), (8, 4, 64, 5)])
def test_moe_topk_bit_exact(R, E_loc, T, topk, mode):
    # the dispatch copy reads a token once and writes the rows of all its slots
    # (the first slot in dispatch order forwards to the others): every top-k
    w = I.MoeWorkload("t", R=R, E_loc=E_loc, T=T, H=136, N=256, topk=topk, integer=True,
                      x_seed=33, logit_seed=43, w_seed=53)
    x, logits, wexp, res, st, detail = run_both(w, cfg=mk.Config(mode=mode))
    assert st == mk.MK_OK, (mk.status_string(st), detail)
    recv_src, seg = check_dispatch(w, x, logits, res)
    xb = [I.bits(t) for t in x]
    for d in range(R):
        rx = O.moe_gather_rows(xb, recv_src[d], w.topk)
        want = O.moe_expert_gemm(rx, seg[d], I.bits(wexp[d]), out="bf16")
        np.testing.assert_array_equal(gpu_bits(res["y"][d][:len(recv_src[d])]), want)


@pytest.mark.parametrize("R,E_loc,T,H,N", SMALL)
def test_moe_float_within_tolerance(R, E_loc, T, H, N):
    w = I.MoeWorkload("t", R=R, E_loc=E_loc, T=T, H=H, N=N, x_seed=61, logit_seed=71, w_seed=81)
    x, logits, wexp, res, st, detail = run_both(w)
    assert st == mk.MK_OK, (mk.status_string(st), detail)
    recv_src, seg = check_dispatch(w, x, logits, res)
    xb = [I.bits(t) for t in x]
    amax = absmax(x)
    bmax = absmax(wexp)
    for d in range(R):
        n = len(recv_src[d])
        if n == 0:
            continue
        rx = O.moe_gather_rows(xb, recv_src[d], w.topk)
        exact = O.moe_expert_gemm(rx, seg[d], I.bits(wexp[d]), out="f64")
        assert norm_err(gpu_values(res["y"][d][:n]), exact, H, amax, bmax) <= TOL["bf16"]


def test_moe_routing_ties_and_golden():
    # logits quantised to create ties (lower expert id wins), and the stored oracle golden
    gold = json.load(open(os.path.join(HERE, "golden", "oracle_golden.json")))["moe_small_route"]
    R, E_loc, T = 4, 4, 256
    x = [torch.zeros((T, 64), dtype=torch.bfloat16) for _ in range(R)]
    logits = [I.zipf_logits(T, R * E_loc, 7000 + r) for r in range(R)]
    wexp = [torch.zeros((E_loc, 64, 256), dtype=torch.bfloat16) for _ in range(R)]
    res = mk.moe_dispatch_gemm([t.cuda() for t in x], [t.cuda() for t in logits],
                               [t.cuda() for t in wexp], E_loc=E_loc, topk=2)
    st, _ = mk.device_status()
    assert st == mk.MK_OK
    sha = hashlib.sha256(res["topk_idx"].cpu().numpy().astype(np.int32).tobytes()).hexdigest()
    assert sha == gold["topk_sha256_i32"]
    assert res["counts"].cpu().numpy().tolist() == gold["counts"]
    rc = res["recv_counts"].cpu().numpy()
    for d in range(R):
        s = res["recv_src"][d][:rc[d]].cpu().numpy().astype(np.int32)
        assert hashlib.sha256(s.tobytes()).hexdigest() == gold["recv_src_sha256_i32"][d]
    # ties
    lg = [torch.from_numpy((np.round(np.random.default_rng(5 + r).standard_normal((T, R * E_loc)) * 1.5)
                            ).astype(np.float32)) for r in range(R)]
    res = mk.moe_dispatch_gemm([t.cuda() for t in x], [t.cuda() for t in lg],
                               [t.cuda() for t in wexp], E_loc=E_loc, topk=3)
    want = np.concatenate([O.moe_route(l.numpy(), 3) for l in lg], 0)
    np.testing.assert_array_equal(res["topk_idx"].cpu().numpy(), want)


@pytest.mark.parametrize("R,E_loc,T,topk", [
    (2, 80, 300, 5),     # experts in three staging blocks, the last one partial
    (4, 64, 129, 8),     # E = 256, the largest expert set; topk = 8
    (16, 16, 200, 2),    # the most ranks
    (3, 7, 1000, 3),     # E = 21 (one partial block), many chunks
    (1, 1, 50, 1),
])
def test_moe_routing_bookkeeping_shapes(R, E_loc, T, topk):
    # routing, counts and the dispatch permutation alone (N = 0: no GEMM launch),
    # on logits with many ties, including -0 against +0 (a tie: lower id wins)
    E = R * E_loc
    lg = []
    for r in range(R):
        v = np.round(np.random.default_rng(90 + r).standard_normal((T, E)) * 1.2).astype(np.float32)
        v[::7, ::3] = -0.0
        lg.append(torch.from_numpy(v))
    x = [torch.zeros((T, 8), dtype=torch.bfloat16).cuda() for _ in range(R)]
    wexp = [torch.zeros((E_loc, 8, 0), dtype=torch.bfloat16).cuda() for _ in range(R)]
    ws = mk.Workspace()
    res = mk.moe_dispatch_gemm(x, [t.cuda() for t in lg], wexp, E_loc=E_loc, topk=topk, workspace=ws)
    st, _ = mk.device_status(ws)
    assert st == mk.MK_OK
    idx = [O.moe_route(t.numpy(), topk) for t in lg]
    np.testing.assert_array_equal(res["topk_idx"].cpu().numpy(), np.concatenate(idx, 0))
    np.testing.assert_array_equal(res["counts"].cpu().numpy(), O.moe_counts(idx, E))
    recv_src, _ = O.moe_dispatch(idx, E_loc)
    rc = res["recv_counts"].cpu().numpy()
    for d in range(R):
        assert rc[d] == len(recv_src[d])
        np.testing.assert_array_equal(res["recv_src"][d][:rc[d]].cpu().numpy(), recv_src[d])


def test_moe_capacity_overflow_reports_and_dispatches_nothing():
    w = I.MoeWorkload("t", R=2, E_loc=2, T=128, H=64, N=256, integer=True, cap_rows=64)
    x, logits, wexp = I.moe_inputs(w)
    ws = mk.Workspace()
    sentinel = [torch.full((64,), -7, dtype=torch.int32, device="cuda") for _ in range(2)]
    res = mk.moe_dispatch_gemm([t.cuda() for t in x], [t.cuda() for t in logits],
                               [t.cuda() for t in wexp], E_loc=2, topk=2, cap_rows=64,
                               out={"recv_src": sentinel}, workspace=ws)
    st, _ = mk.device_status(ws)
    assert st == mk.MK_ERR_CAPACITY
    assert all(int((s == -7).sum()) == 64 for s in res["recv_src"])
    assert int(res["recv_counts"].sum()) == 2 * 128 * 2


def test_moe_single_expert_identity():
    R, T, H, N = 1, 200, 64, 256
    w = I.MoeWorkload("t", R=R, E_loc=1, T=T, H=H, N=N, topk=1, integer=True)
    x, logits, wexp, res, st, _ = run_both(w)
    assert st == mk.MK_OK
    assert res["recv_src"][0][:T].cpu().tolist() == list(range(T))
    want = O.moe_expert_gemm(I.bits(x[0]), [T], I.bits(wexp[0]), out="bf16")
    np.testing.assert_array_equal(gpu_bits(res["y"][0][:T]), want)


@pytest.mark.parametrize("pair", [mk.PAIR_OFF, mk.PAIR_ON])
def test_moe_missing_rows_time_out(pair):
    w = I.MoeWorkload("t", R=2, E_loc=2, T=128, H=64, N=256, integer=True)
    x, logits, wexp, res, st, _ = run_both(w, cfg=mk.Config(inject=1, wait_limit_ns=20_000_000,
                                                             cta_pair=pair))
    assert st == mk.MK_ERR_TIMEOUT
    x, logits, wexp, res, st, _ = run_both(w)
    assert st == mk.MK_OK
    check_dispatch(w, x, logits, res)


def test_moe_baseline_modes_match_fused():
    w = I.MoeWorkload("t", R=4, E_loc=2, T=200, H=256, N=512, integer=True, x_seed=91,
                      logit_seed=92, w_seed=93)
    x, logits, wexp = I.moe_inputs(w)
    args = ([t.cuda() for t in x], [t.cuda() for t in logits], [t.cuda() for t in wexp])
    ws = mk.Workspace()
    fused = mk.moe_dispatch_gemm(*args, E_loc=w.E_loc, topk=2, workspace=ws)
    unf = mk.moe_dispatch_gemm(*args, E_loc=w.E_loc, topk=2, workspace=ws,
                               cfg=mk.Config(mode=mk.MODE_UNFUSED))
    # GEMM only: recv_x is taken as already filled (here: by the fused call)
    out = {"recv_x": fused["recv_x"]}
    gonly = mk.moe_dispatch_gemm(*args, E_loc=w.E_loc, topk=2, workspace=ws, out=out,
                                 cfg=mk.Config(mode=mk.MODE_GEMM_ONLY))
    st, _ = mk.device_status(ws)
    assert st == mk.MK_OK
    rc = fused["recv_counts"].cpu().numpy()
    for d in range(w.R):
        for other in (unf, gonly):
            assert torch.equal(fused["y"][d][:rc[d]], other["y"][d][:rc[d]])
        assert torch.equal(fused["recv_x"][d][:rc[d]], unf["recv_x"][d][:rc[d]])
