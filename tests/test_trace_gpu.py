"""In-kernel trace of the fused GEMM kernels (GPU).

With mk_config.trace = 1 every work item of an AllGather+GEMM, GEMM+ReduceScatter
or GEMM+AllReduce call writes, per CTA of the pair, three %globaltimer stamps
(producer start, accumulator ready, epilogue done) and its epoch / CTA / pair
rank.  Checked here: tracing leaves the results bit-identical; the call's
records are the newest epoch, cover every item index from 0 up with the same
pair ranks, and are ordered start <= ready <= end; a second call on the same
workspace overwrites them with a later epoch.
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
    epochs = rec[:, 3] >> 32
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
    assert bool((r[:, 0] <= r[:, 1]).all()) and bool((r[:, 1] <= r[:, 2]).all())
    assert bool(((r[:, 3] & 1) == idx % 2).all())     # the pair rank of the record's slot
    ctas = (r[:, 3] >> 1) & 0x7FFFFFFF
    assert int(ctas.max()) < 4 * torch.cuda.get_device_properties(0).multi_processor_count
    # a tile is split over at most R*split_k items; at least one item per 2 tiles
    n_tiles = -(-(m * (R if op == "ag" else 1)) // 128) * -(-n // 256)
    assert len(items) >= n_tiles // 2

    got2 = _call(op, a, b, cfg, ws)
    assert torch.equal(got2, plain)
    rec2 = mk.trace_records(ws, OPS[op], R, m, n, k, cfg)
    e2, sel2 = _latest(rec2)
    assert e2 > e1 and torch.equal(sel2, sel)
