"""The bounds-checking build (libmk_debug.so, MK_DEBUG_BOUNDS=1) on the small
parity shapes (GPU).

Its device-side index checks (tile coordinates inside the output and the
operands, copy rows inside the shards and the gathered A, MoE slot positions
and received-row sources inside their buffers, ring tiles inside their blocks)
report MK_ERR_INVALID instead of touching memory out of range.  On valid inputs
none of them may fire: every op must run with MK_OK and give the same bits as
the default build (and, on integer-valued inputs, as the oracle).  Shapes are
ragged in every dimension, with CTA pairs on and off.
"""
import numpy as np
import pytest
import torch

import oracle as O
import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import inputs as I
from parity_util import dev, gpu_bits, oracle_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from comm_gemm_tile_gb300 import build
    build.build(debug=True)
    torch.cuda.init()


def _both(fn):
    """fn() with the default library, then with the bounds-checking one; the
    device status of each must be MK_OK.  Returns both results."""
    ws = mk.Workspace()
    a = fn(ws)
    st, detail = mk.device_status(ws)
    assert st == mk.MK_OK, (mk.status_string(st), detail)
    with mk.use_library(mk.LIB_DEBUG_PATH):
        wsd = mk.Workspace()
        b = fn(wsd)
        st, detail = mk.device_status(wsd)
        assert st == mk.MK_OK, ("bounds build", mk.status_string(st), detail)
    return a, b


def _same(x, y):
    if isinstance(x, (list, tuple)):
        for u, v in zip(x, y):
            _same(u, v)
    elif isinstance(x, dict):
        for key in x:
            _same(x[key], y[key])
    else:
        assert torch.equal(x, y)


@pytest.mark.parametrize("pair", [mk.PAIR_OFF, mk.PAIR_ON])
def test_bounds_build_ag_rs_ar(pair):
    cfg = mk.Config(cta_pair=pair)
    w = I.GemmWorkload("t", "ag", R=4, m=200, n=264, k=520, out="bf16", a_seed=401, b_seed=402,
                       integer=True)
    a, b = I.gemm_inputs(w)
    x, y = _both(lambda ws: mk.ag_gemm(dev(a), b[0].cuda(), local_rank=2, cfg=cfg, workspace=ws))
    _same(x, y)
    gathered, want = O.ag_gemm([I.bits(t) for t in a], I.bits(b[0]), out="bf16")
    np.testing.assert_array_equal(I.bits(y[0]), gathered)
    np.testing.assert_array_equal(gpu_bits(y[1]), want)
    for op, fn in (("rs", mk.gemm_rs), ("ar", mk.gemm_ar)):
        w = I.GemmWorkload("t", op, R=4, m=520, n=264, k=136, out="bf16", a_seed=403, b_seed=404,
                           integer=True)
        a, b = I.gemm_inputs(w)
        x, y = _both(lambda ws: fn(dev(a), dev(b), cfg=cfg, workspace=ws))
        _same(x, y)
        exact = O.sum_over_ranks([I.bits(t) for t in a], [I.bits(t) for t in b])
        got = torch.cat(y, 0) if op == "rs" else y[0]
        np.testing.assert_array_equal(gpu_bits(got), oracle_bits(exact, "bf16"))


@pytest.mark.parametrize("reduce", [mk.REDUCE_LAST_ARRIVAL, mk.REDUCE_ATOMIC])
def test_bounds_build_reductions_and_modes(reduce):
    w = I.GemmWorkload("t", "rs", R=4, m=512, n=512, k=256, out="f32", a_seed=405, b_seed=406,
                       integer=True)
    a, b = I.gemm_inputs(w)
    for cfg in (mk.Config(reduce=reduce), mk.Config(mode=mk.MODE_UNFUSED), mk.Config(n_reduce_ctas=3),
                mk.Config(wire=mk.WIRE_BF16)):
        x, y = _both(lambda ws: mk.gemm_rs(dev(a), dev(b), out_dtype=torch.float32, cfg=cfg, workspace=ws))
        _same(x, y)


def test_bounds_build_moe_dispatch_and_combine():
    w = I.MoeWorkload("t", R=4, E_loc=3, T=257, H=264, N=520, integer=True)
    x, logits, wexp = I.moe_inputs(w)

    def disp(ws):
        return mk.moe_dispatch_gemm([t.cuda() for t in x], [t.cuda() for t in logits],
                                    [t.cuda() for t in wexp], E_loc=w.E_loc, topk=w.topk,
                                    cap_rows=w.cap, workspace=ws)
    r0, r1 = _both(disp)
    rc = r1["recv_counts"].cpu().numpy()
    for key in ("topk_idx", "counts", "recv_counts"):
        assert torch.equal(r0[key], r1[key])
    for d in range(w.R):
        n = int(rc[d])
        assert torch.equal(r0["recv_src"][d][:n], r1["recv_src"][d][:n])
        assert torch.equal(r0["recv_x"][d][:n], r1["recv_x"][d][:n])
        assert torch.equal(r0["y"][d][:n], r1["y"][d][:n])
    # combine of the same routing
    wc = I.MoeCombineWorkload("t", R=4, E_loc=3, T=257, H=264, N=136, integer=True)
    lg, h, w2, gates = I.combine_inputs(wc)
    idx = [O.moe_route(t.numpy(), wc.topk) for t in lg]
    counts = O.moe_counts(idx, wc.E)
    recv_src, _ = O.moe_dispatch(idx, wc.E_loc)
    rs_d = []
    for d in range(wc.R):
        t = torch.zeros(wc.cap, dtype=torch.int32)
        t[:len(recv_src[d])] = torch.from_numpy(recv_src[d].astype(np.int32))
        rs_d.append(t.cuda())
    cnt = torch.from_numpy(counts.astype(np.int32)).cuda()
    c0, c1 = _both(lambda ws: mk.moe_combine([t.cuda() for t in h], [t.cuda() for t in w2],
                                             [g.cuda() for g in gates], rs_d, cnt, E_loc=wc.E_loc,
                                             topk=wc.topk, cap_rows=wc.cap, workspace=ws))
    _same(c0["out"], c1["out"])
    _same(c0["ret"], c1["ret"])


def test_bounds_build_mlp_and_ring_attention():
    wm = I.MlpWorkload("t", R=4, m=200, h=264, f_r=136, integer=True)
    x, w1, w2 = I.mlp_inputs(wm)
    m0, m1 = _both(lambda ws: mk.mlp_ag_rs(dev(x), dev(w1), dev(w2), workspace=ws))
    _same(m0, m1)
    for causal in (False, True):
        wa = I.AttnWorkload("t", R=4, heads=2, s_r=200, causal=causal, q_seed=411, k_seed=412, v_seed=413)
        q, k, v = (dev(t) for t in I.attn_inputs(wa))
        a0, a1 = _both(lambda ws: mk.ring_attention(q, k, v, causal=causal, workspace=ws))
        _same(a0, a1)
