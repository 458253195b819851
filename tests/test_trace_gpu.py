"""In-kernel trace of the fused GEMM kernels (GPU).

With mk_config.trace = 1 every work item of an AllGather+GEMM, GEMM+ReduceScatter
or GEMM+AllReduce call writes, per CTA of the pair, five %globaltimer stamps
(producer takes the item, inputs ready, last load issued, accumulator ready,
epilogue done), the SM's clock64 at the first and fourth, and its epoch / CTA /
pair rank; AllGather's copy warps add one record each (start, end, pieces,
bytes).  Checked here: tracing leaves the results bit-identical; the call's
records are the newest epoch, cover every item index from 0 up with the same
pair ranks, and their stamps are ordered; the clock stamps give an SM clock
within the device's range; a second call on the same workspace overwrites them
with a later epoch.
"""
import pytest
import torch

import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import inputs as I
from parity_util import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from comm_gemm_tile_gb300 import build
    build.build()
    torch.cuda.init()


def _call(op, a, b, cfg, ws):
    if op == "ag":
        _, c = mk.ag_gemm(dev(a), dev(b)[0], cfg=cfg, workspace=ws)
        return c
    if op == "rs":
        return torch.cat(mk.gemm_rs(dev(a), dev(b), cfg=cfg, workspace=ws), 0)
    return mk.gemm_ar(dev(a), dev(b), cfg=cfg, workspace=ws)[0]


OPS = {"ag": mk.OP_AG_GEMM, "rs": mk.OP_GEMM_RS, "ar": mk.OP_GEMM_AR}
CASES = [  # op, R, m (rows per shard for AG), n, k, reduce
    ("ag", 4, 256, 1024, 512, 0),
    ("ag", 3, 200, 520, 136, 0),
    ("rs", 4, 1024, 1024, 512, 0),
    ("rs", 4, 520, 520, 200, mk.REDUCE_LAST_ARRIVAL),
    ("rs", 8, 1024, 512, 512, mk.REDUCE_ATOMIC),
    ("ar", 2, 384, 264, 136, 0),
]


def _latest(rec):
    epochs = rec[:, mk.TRACE_ID] >> 32
    e = int(epochs.max())
    sel = (epochs == e) & (rec[:, 0] != 0)
    return e, sel


@pytest.mark.parametrize("pair", [mk.PAIR_OFF, mk.PAIR_ON])
@pytest.mark.parametrize("op,R,m,n,k,reduce", CASES)
def test_trace_records(op, R, m, n, k, reduce, pair):
    # the atomic reduction's fp32 summation order varies between calls: integer-valued
    # inputs keep every partial sum exact, so its results still match bit for bit
    w = I.GemmWorkload("t", op, R=R, m=m, n=n, k=k, out="bf16", a_seed=7, b_seed=8,
                       integer=(reduce == mk.REDUCE_ATOMIC))
    a, b = I.gemm_inputs(w)
    ws0 = mk.Workspace()
    plain = _call(op, a, b, mk.Config(cta_pair=pair, reduce=reduce), ws0)
    st, detail = mk.device_status(ws0)
    assert st == mk.MK_OK, (mk.status_string(st), detail)

    cfg = mk.Config(cta_pair=pair, reduce=reduce, trace=1)
    ws = mk.Workspace()
    got = _call(op, a, b, cfg, ws)
    st, detail = mk.device_status(ws)
    assert st == mk.MK_OK, (mk.status_string(st), detail)
    assert torch.equal(got, plain)

    rec = mk.trace_records(ws, OPS[op], R, m, n, k, cfg)
    assert rec.shape[0] > 0
    e1, sel = _latest(rec)
    idx = torch.nonzero(sel).flatten()
    items = sorted({int(j) // 2 for j in idx})
    assert items == list(range(len(items)))           # items 0 .. n_items-1, none skipped
    ranks = {int(j) % 2 for j in idx}
    assert len(idx) == len(items) * len(ranks)        # every item on the same pair ranks
    r = rec[idx]
    assert rec.shape[1] == mk.TRACE_WORDS
    for a_, b_ in ((mk.TRACE_START, mk.TRACE_INPUTS), (mk.TRACE_INPUTS, mk.TRACE_ISSUED),
                   (mk.TRACE_START, mk.TRACE_READY), (mk.TRACE_READY, mk.TRACE_END)):
        assert bool((r[:, a_] <= r[:, b_]).all()), (a_, b_)
    # the SM clock over an item (clock64 ticks / ns), where the item spans over 2 us
    dt = (r[:, mk.TRACE_READY] - r[:, mk.TRACE_START]).double()
    dc = (r[:, mk.TRACE_CLK_READY] - r[:, mk.TRACE_CLK_START]).double()
    long_ = dt > 2000
    if bool(long_.any()):
        ghz = dc[long_] / dt[long_]
        assert float(ghz.min()) > 0.3 and float(ghz.max()) < 3.5, (float(ghz.min()), float(ghz.max()))
    assert bool(((r[:, mk.TRACE_ID] & 1) == idx % 2).all())     # the pair rank of the slot
    ctas = (r[:, mk.TRACE_ID] >> 1) & 0x7FFFFFFF
    assert int(ctas.max()) < 4 * torch.cuda.get_device_properties(0).multi_processor_count
    # a tile is split over at most R*split_k items; at least one item per 2 tiles
    n_tiles = -(-(m * (R if op == "ag" else 1)) // 128) * -(-n // 256)
    assert len(items) >= n_tiles // 2

    if op == "ag":
        # the copy warps' records: together they moved every row of the gathered A
        cr = mk.trace_copy_records(ws, OPS[op], R, m, n, k, cfg)
        mine = cr[(cr[:, mk.TRACE_ID] >> 32) == e1]
        assert mine.shape[0] > 0
        assert int(mine[:, 3].sum()) == R * m * k * 2
        assert bool((mine[:, 0] <= mine[:, 1]).all()) and bool((mine[:, 2] >= 0).all())
        assert set((mine[:, mk.TRACE_ID] & 0xFFFFFFFF).tolist()) == set(range(mine.shape[0]))

    got2 = _call(op, a, b, cfg, ws)
    assert torch.equal(got2, plain)
    rec2 = mk.trace_records(ws, OPS[op], R, m, n, k, cfg)
    e2, sel2 = _latest(rec2)
    assert e2 > e1 and torch.equal(sel2, sel)


@pytest.mark.parametrize("pair", [mk.PAIR_OFF, mk.PAIR_ON])
def test_moe_trace_records(pair):
    w = I.MoeWorkload("t", R=4, E_loc=3, T=257, H=520, N=264, integer=True, x_seed=31,
                      logit_seed=41, w_seed=51)
    x, logits, wexp = I.moe_inputs(w)
    args = ([t.cuda() for t in x], [t.cuda() for t in logits], [t.cuda() for t in wexp])

    def run(cfg, ws):
        res = mk.moe_dispatch_gemm(*args, E_loc=w.E_loc, topk=w.topk, cap_rows=w.cap, cfg=cfg,
                                   workspace=ws)
        st, detail = mk.device_status(ws)
        assert st == mk.MK_OK, (mk.status_string(st), detail)
        return res

    plain = run(mk.Config(cta_pair=pair), mk.Workspace())
    cfg = mk.Config(cta_pair=pair, trace=1)
    ws = mk.Workspace()
    got = run(cfg, ws)
    rc = got["recv_counts"].cpu()
    assert torch.equal(rc, plain["recv_counts"].cpu())
    for d in range(w.R):
        n = int(rc[d])
        assert torch.equal(got["y"][d][:n], plain["y"][d][:n])
        assert torch.equal(got["recv_x"][d][:n], plain["recv_x"][d][:n])
    rec, crec = mk.moe_trace_records(ws, w.R, w.E_loc, w.topk, w.T, w.H, w.N, w.cap, cfg)
    e, sel = _latest(rec)
    idx = torch.nonzero(sel).flatten()
    items = sorted({int(j) // 2 for j in idx})
    assert items and items == list(range(len(items)))
    r = rec[idx]
    for a_, b_ in ((mk.TRACE_START, mk.TRACE_INPUTS), (mk.TRACE_INPUTS, mk.TRACE_ISSUED),
                   (mk.TRACE_START, mk.TRACE_READY), (mk.TRACE_READY, mk.TRACE_END)):
        assert bool((r[:, a_] <= r[:, b_]).all()), (a_, b_)
    assert crec.shape == (mk.TRACE_COPY_RECORDS, mk.TRACE_WORDS)
    assert not bool(((crec[:, mk.TRACE_ID] >> 32) == e).any())   # the dispatch writes none


@pytest.mark.parametrize("mode", [mk.MODE_FUSED, mk.MODE_GEMM_ONLY])
@pytest.mark.parametrize("pair", [mk.PAIR_OFF, mk.PAIR_ON])
def test_mlp_trace_records(pair, mode):
    # the chained MLP: every up-projection tile and down-projection item of the
    # traced launch leaves ordered stamps; results unchanged by tracing
    w = I.MlpWorkload("t", R=4, m=200, h=264, f_r=520, integer=True)
    x, w1, w2 = I.mlp_inputs(w)
    args = (dev(x), dev(w1), dev(w2))
    ws0 = mk.Workspace()
    xg, hid, y0 = mk.mlp_ag_rs(*args, workspace=ws0)    # fills x_gathered for GEMM-only
    plain = mk.mlp_ag_rs(*args, x_gathered=xg, cfg=mk.Config(cta_pair=pair, mode=mode), workspace=ws0)[2]
    cfg = mk.Config(cta_pair=pair, mode=mode, trace=1)
    ws = mk.Workspace()
    got = mk.mlp_ag_rs(*args, x_gathered=xg, cfg=cfg, workspace=ws)[2]
    st, detail = mk.device_status(ws)
    assert st == mk.MK_OK, (mk.status_string(st), detail)
    for a_, b_ in zip(got, plain):
        assert torch.equal(a_, b_)
    rec, crec = mk.mlp_trace_records(ws, w.R, w.m, w.h, w.f_r, cfg)
    e, sel = _latest(rec)
    idx = torch.nonzero(sel).flatten()
    items = sorted({int(j) // 2 for j in idx})
    assert items and items == list(range(len(items)))
    # up-projection tiles (R ranks x row tiles x column tiles of f_r) come first
    rows = w.R * w.m
    rt = -(-rows // (256 if pair == mk.PAIR_ON else 128))
    n1 = w.R * rt * -(-w.f_r // 256)
    assert len(items) > n1
    r = rec[idx]
    for a_, b_ in ((mk.TRACE_START, mk.TRACE_INPUTS), (mk.TRACE_INPUTS, mk.TRACE_ISSUED),
                   (mk.TRACE_START, mk.TRACE_READY), (mk.TRACE_READY, mk.TRACE_END)):
        assert bool((r[:, a_] <= r[:, b_]).all()), (a_, b_)
    mine = crec[(crec[:, mk.TRACE_ID] >> 32) == e]
    if mode == mk.MODE_FUSED:   # the AllGather copy-in by copy warps moved every gathered row
        assert mine.shape[0] > 0 and int(mine[:, 3].sum()) >= (w.R - 1) * w.m * w.h * 2
    else:
        assert mine.shape[0] == 0
