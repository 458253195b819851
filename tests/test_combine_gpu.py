"""MoE combine: CUDA path vs the CPU oracle (GPU).

The routing (top-k ids, dispatch order, counts) comes from the oracle and is
fed to the combine as its input.  The returned expert rows and the combined
outputs must match bit for bit on integer-valued inputs with dyadic gates
(every product and sum is exact in fp32), and within the normalised tolerance
on float inputs.  Shapes cover ragged expert segments, column counts that are
not multiples of the 256-column block or of 64, one and several ranks, CTA
pairs on and off, and the two baseline modes.
"""
import numpy as np
import pytest
import torch

import oracle as O
import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import inputs as I
from parity_util import TOL, absmax, gpu_bits, gpu_values, norm_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from comm_gemm_tile_gb300 import build
    build.build()
    torch.cuda.init()


def route(w, logits):
    idx = [O.moe_route(lg.numpy(), w.topk) for lg in logits]
    counts = O.moe_counts(idx, w.E)
    recv_src, seg = O.moe_dispatch(idx, w.E_loc)
    return idx, counts, recv_src, seg


def device_routing(w, counts, recv_src):
    rs = []
    for d in range(w.R):
        t = torch.zeros(w.cap, dtype=torch.int32)
        t[:len(recv_src[d])] = torch.from_numpy(recv_src[d].astype(np.int32))
        rs.append(t.cuda())
    return torch.from_numpy(counts.astype(np.int32)).cuda(), rs


def run(w, cfg=None, inputs=None):
    logits, h, w2, gates = inputs or I.combine_inputs(w)
    idx, counts, recv_src, seg = route(w, logits)
    cnt_d, rs_d = device_routing(w, counts, recv_src)
    ws = mk.Workspace()
    res = mk.moe_combine([t.cuda() for t in h], [t.cuda() for t in w2], [g.cuda() for g in gates],
                         rs_d, cnt_d, E_loc=w.E_loc, topk=w.topk, cap_rows=w.cap, cfg=cfg,
                         workspace=ws)
    st, detail = mk.device_status(ws)
    return (logits, h, w2, gates), (counts, recv_src), res, st, detail


SMALL = [  # R, E_loc, T, N, H
    (2, 2, 100, 64, 256),
    (4, 3, 257, 264, 520),     # H not a multiple of 64 (two-box B loads), ragged last block
    (8, 8, 64, 128, 512),
    (1, 4, 300, 256, 264),
]


@pytest.mark.parametrize("pair", [mk.PAIR_OFF, mk.PAIR_ON])
@pytest.mark.parametrize("R,E_loc,T,N,H", SMALL)
def test_combine_integer_bit_exact(R, E_loc, T, N, H, pair):
    w = I.MoeCombineWorkload("t", R=R, E_loc=E_loc, T=T, N=N, H=H, integer=True, logit_seed=61,
                             h_seed=71, w2_seed=81, gate_seed=91)
    (logits, h, w2, gates), (counts, recv_src), res, st, detail = run(w, mk.Config(cta_pair=pair))
    assert st == mk.MK_OK, (mk.status_string(st), detail)
    want = O.moe_combine([I.bits(t) for t in h], recv_src, counts, [I.bits(t) for t in w2],
                         [g.numpy() for g in gates], w.E_loc, w.topk, w.T)
    for r in range(R):
        np.testing.assert_array_equal(I.bits(res["ret"][r]), want["ret"][r])
        np.testing.assert_array_equal(I.bits(res["out"][r]), want["out"][r])


@pytest.mark.parametrize("topk", [1, 3])
def test_combine_other_topk_bit_exact(topk):
    w = I.MoeCombineWorkload("t", R=4, E_loc=3, T=150, N=128, H=264, topk=topk, integer=True,
                             logit_seed=64, h_seed=74, w2_seed=84, gate_seed=94)
    (logits, h, w2, gates), (counts, recv_src), res, st, detail = run(w)
    assert st == mk.MK_OK, (mk.status_string(st), detail)
    want = O.moe_combine([I.bits(t) for t in h], recv_src, counts, [I.bits(t) for t in w2],
                         [g.numpy() for g in gates], w.E_loc, w.topk, w.T)
    for r in range(w.R):
        np.testing.assert_array_equal(I.bits(res["ret"][r]), want["ret"][r])
        np.testing.assert_array_equal(I.bits(res["out"][r]), want["out"][r])


@pytest.mark.parametrize("R,E_loc,T,N,H", SMALL[:3])
def test_combine_float_within_tolerance(R, E_loc, T, N, H):
    w = I.MoeCombineWorkload("t", R=R, E_loc=E_loc, T=T, N=N, H=H, logit_seed=62, h_seed=72,
                             w2_seed=82, gate_seed=92)
    (logits, h, w2, gates), (counts, recv_src), res, st, detail = run(w)
    assert st == mk.MK_OK, (mk.status_string(st), detail)
    hb, w2b = [I.bits(t) for t in h], [I.bits(t) for t in w2]
    want = O.moe_combine(hb, recv_src, counts, w2b, [g.numpy() for g in gates], w.E_loc, w.topk, w.T)
    amax, bmax = absmax(h), absmax(w2)
    for r in range(R):
        assert norm_err(gpu_values(res["ret"][r]), O.bf16_to_f64(want["ret"][r]), N, amax, bmax) \
            <= TOL["bf16"]
        assert norm_err(gpu_values(res["out"][r]), O.bf16_to_f64(want["out"][r]), N, amax, bmax) \
            <= TOL["bf16"]


def test_combine_baseline_modes_match_fused():
    w = I.MoeCombineWorkload("t", R=4, E_loc=2, T=200, N=256, H=512, logit_seed=63, h_seed=73,
                             w2_seed=83, gate_seed=93)
    inputs = I.combine_inputs(w)
    _, _, fused, st, _ = run(w, None, inputs)
    assert st == mk.MK_OK
    _, _, gonly, st, _ = run(w, mk.Config(mode=mk.MODE_GEMM_ONLY), inputs)
    assert st == mk.MK_OK
    _, _, unf, st, _ = run(w, mk.Config(mode=mk.MODE_UNFUSED), inputs)
    assert st == mk.MK_OK
    for r in range(w.R):
        assert torch.equal(fused["ret"][r], gonly["ret"][r])
        assert torch.equal(fused["ret"][r], unf["ret"][r])
        assert torch.equal(fused["out"][r], unf["out"][r])     # same fp32 FMAs in slot order


def test_combine_capacity_overflow_reports_and_computes_nothing():
    w = I.MoeCombineWorkload("t", R=2, E_loc=2, T=64, N=64, H=256, integer=True, cap_rows=40)
    logits, h, w2, gates = I.combine_inputs(w)
    idx, counts, recv_src, seg = route(w, logits)
    assert max(len(s) for s in recv_src) > 40
    cnt = torch.from_numpy(counts.astype(np.int32)).cuda()
    rs = [torch.zeros(40, dtype=torch.int32, device="cuda") for _ in range(w.R)]
    ret = [torch.full((w.T, 2, w.H), 3.0, dtype=torch.bfloat16, device="cuda") for _ in range(w.R)]
    out = [torch.full((w.T, w.H), 3.0, dtype=torch.bfloat16, device="cuda") for _ in range(w.R)]
    ws = mk.Workspace()
    mk.moe_combine([t[:40].cuda() for t in h], [t.cuda() for t in w2], [g.cuda() for g in gates], rs,
                   cnt, E_loc=2, topk=2, cap_rows=40, out={"ret": ret, "out": out}, workspace=ws)
    st, _ = mk.device_status(ws)
    assert st == mk.MK_ERR_CAPACITY
    assert all(bool((t == 3.0).all()) for t in ret + out)


def test_dispatch_then_combine_with_identity_experts_returns_the_tokens():
    # GPU dispatch (x -> recv_x) feeds the GPU combine with W2 = I (N = H) and
    # gates 0.75 / 0.25: every token comes back bit for bit.
    R, E_loc, T, H, topk = 4, 2, 300, 256, 2
    wd = I.MoeWorkload("t", R=R, E_loc=E_loc, T=T, H=H, N=64, integer=True, x_seed=201,
                       logit_seed=202, w_seed=203)
    x, logits, wexp = I.moe_inputs(wd)
    ws = mk.Workspace()
    disp = mk.moe_dispatch_gemm([t.cuda() for t in x], [t.cuda() for t in logits],
                                [t.cuda() for t in wexp], E_loc=E_loc, topk=topk, workspace=ws)
    eye = [torch.eye(H, dtype=torch.bfloat16).repeat(E_loc, 1, 1).cuda() for _ in range(R)]
    gates = [torch.tensor([[0.75, 0.25]], dtype=torch.float32).repeat(T, 1).cuda() for _ in range(R)]
    res = mk.moe_combine(disp["recv_x"], eye, gates, disp["recv_src"], disp["counts"], E_loc=E_loc,
                         topk=topk, workspace=ws)
    st, _ = mk.device_status(ws)
    assert st == mk.MK_OK
    for r in range(R):
        assert torch.equal(res["out"][r].cpu(), x[r])


def test_combine_repeated_calls_and_empty_contraction():
    w = I.MoeCombineWorkload("t", R=2, E_loc=2, T=130, N=64, H=256, integer=True)
    inputs = I.combine_inputs(w)
    ws = mk.Workspace()
    first = None
    for _ in range(3):       # counters are zeroed per call: repeated calls agree
        _, _, res, st, _ = run(w, None, inputs)
        assert st == mk.MK_OK
        if first is None:
            first = [t.clone() for t in res["out"]]
        for a, b in zip(first, res["out"]):
            assert torch.equal(a, b)
    # N = 0: every returned row and output is zero
    h0 = [torch.zeros((w.cap, 0), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    w20 = [torch.zeros((2, 0, 256), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    g = [t.cuda() for t in inputs[3]]
    idx, counts, recv_src, seg = route(w, inputs[0])
    cnt_d, rs_d = device_routing(w, counts, recv_src)
    res = mk.moe_combine(h0, w20, g, rs_d, cnt_d, E_loc=2, topk=2, workspace=ws)
    st, _ = mk.device_status(ws)
    assert st == mk.MK_OK
    assert all(float(t.float().abs().max()) == 0.0 for t in res["ret"] + res["out"])


def _random_case(seed):
    g = np.random.default_rng(seed)
    R = int(g.integers(1, 17))                      # up to 16 ranks
    E_loc = int(g.integers(1, 256 // R + 1 if R > 1 else 9))
    E_loc = min(E_loc, 256 // R)
    topk = int(g.integers(1, min(8, R * E_loc) + 1))
    T = int(g.integers(1, 200))
    N = 8 * int(g.integers(1, 40))
    H = 8 * int(g.integers(1, 70))
    pair = [mk.PAIR_OFF, mk.PAIR_ON][int(g.integers(0, 2))]
    return R, E_loc, topk, T, N, H, pair


@pytest.mark.parametrize("seed", list(range(8)))
def test_combine_random_shapes_bit_exact(seed):
    # seeded random shapes: up to 16 ranks and 256 experts (the plan kernel's
    # shared-memory tables and warp scans), top-k 1..8, CTA pairs on and off
    R, E_loc, topk, T, N, H, pair = _random_case(9000 + seed)
    w = I.MoeCombineWorkload("t", R=R, E_loc=E_loc, T=T, N=N, H=H, topk=topk, integer=True,
                             logit_seed=300 + seed, h_seed=310 + seed, w2_seed=320 + seed,
                             gate_seed=330 + seed)
    (logits, h, w2, gates), (counts, recv_src), res, st, detail = run(w, mk.Config(cta_pair=pair))
    assert st == mk.MK_OK, (mk.status_string(st), detail, (R, E_loc, topk, T, N, H, pair))
    want = O.moe_combine([I.bits(t) for t in h], recv_src, counts, [I.bits(t) for t in w2],
                         [g.numpy() for g in gates], w.E_loc, w.topk, w.T)
    for r in range(R):
        np.testing.assert_array_equal(I.bits(res["ret"][r]), want["ret"][r])
        np.testing.assert_array_equal(I.bits(res["out"][r]), want["out"][r])
