"""Ring attention: CUDA path vs the CPU oracle (GPU).

The softmax makes float parity the main bar: max |gpu - exact| / max|V|
within ATT_TOL (P is rounded to bf16 for the tensor cores and the output to
bf16, each about 2^-9 relative).  Exact pins: with Q = 0 every score is 0, so
each output row is the mean of the visible values; with integer values and a
power-of-two key count that mean is exact in fp32 and must match bit for bit.
The receive buffers must hold bit copies of the ring's blocks.  Shapes cover
ragged blocks (positions not a multiple of 128), one rank, several heads,
causal and full attention, all three modes, a missing ring piece and receive
buffers that start as NaN (rows past a ragged block must read as zeros).
"""
import numpy as np
import pytest
import torch

import oracle as O
import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import inputs as I
from parity_util import dev, gpu_values

pytestmark = pytest.mark.gpu
ATT_TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from comm_gemm_tile_gb300 import build
    build.build()
    torch.cuda.init()


def _ok(ws=None):
    st, detail = mk.device_status(ws)
    assert st == mk.MK_OK, (mk.status_string(st), detail)


def _err(got, exact, vmax):
    return float(np.max(np.abs(got - exact))) / vmax


SHAPES = [  # R, heads, s_r
    (2, 2, 256),
    (4, 1, 200),     # ragged: the last key and query tiles of every block are partial
    (1, 3, 384),
    (8, 2, 128),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("R,heads,s_r", SHAPES)
def test_ring_attention_float(R, heads, s_r, causal):
    w = I.AttnWorkload("t", R=R, heads=heads, s_r=s_r, causal=causal, q_seed=51, k_seed=61, v_seed=71)
    q, k, v = I.attn_inputs(w)
    ws = mk.Workspace()
    kr = [torch.empty(((R - 1) * heads, s_r, 128), dtype=torch.bfloat16, device="cuda") for _ in range(R)]
    vr = [torch.empty_like(t) for t in kr]
    out = mk.ring_attention(dev(q), dev(k), dev(v), causal=causal, k_recv=kr if R > 1 else None,
                            v_recv=vr if R > 1 else None, workspace=ws)
    _ok(ws)
    exact = O.ring_attention([I.bits(t) for t in q], [I.bits(t) for t in k], [I.bits(t) for t in v],
                             causal, w.scale, out="f32")
    vmax = max(float(t.float().abs().max()) for t in v)
    for r in range(R):
        assert _err(gpu_values(out[r]), exact[r].astype(np.float64), vmax) <= ATT_TOL
    if R > 1:   # the ring's receive buffers: bit copies of the blocks that were needed
        for r in range(R):
            for j in range(1, R):
                s = (r - j) % R
                if causal and s > r:
                    continue
                blk = slice((j - 1) * heads, j * heads)
                assert torch.equal(kr[r][blk].cpu(), k[s]) and torch.equal(vr[r][blk].cpu(), v[s])


@pytest.mark.parametrize("R,heads,s_r", [(2, 2, 256), (4, 1, 128), (1, 2, 512)])
def test_ring_attention_zero_queries_exact_mean(R, heads, s_r):
    w = I.AttnWorkload("t", R=R, heads=heads, s_r=s_r, integer=True, q_seed=52, k_seed=62, v_seed=72)
    _, k, v = I.attn_inputs(w)
    q = [torch.zeros_like(t) for t in k]
    out = mk.ring_attention(dev(q), dev(k), dev(v))
    _ok()
    exact = O.ring_attention([I.bits(t) for t in q], [I.bits(t) for t in k], [I.bits(t) for t in v],
                             False, w.scale)
    for r in range(R):
        np.testing.assert_array_equal(I.bits(out[r]), exact[r])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mode", [mk.MODE_GEMM_ONLY, mk.MODE_UNFUSED])
def test_ring_attention_modes_match_fused(mode, causal):
    w = I.AttnWorkload("t", R=4, heads=2, s_r=256, causal=causal, q_seed=53, k_seed=63, v_seed=73)
    q, k, v = (dev(x) for x in I.attn_inputs(w))
    ws = mk.Workspace()
    a = mk.ring_attention(q, k, v, causal=causal, workspace=ws)
    b = mk.ring_attention(q, k, v, causal=causal, workspace=ws, cfg=mk.Config(mode=mode))
    _ok(ws)
    for r in range(w.R):
        assert torch.equal(a[r], b[r])


@pytest.mark.parametrize("max_ctas", [1, 3])
def test_ring_attention_few_ctas(max_ctas):
    w = I.AttnWorkload("t", R=4, heads=2, s_r=200, causal=True, q_seed=54, k_seed=64, v_seed=74)
    q, k, v = I.attn_inputs(w)
    out = mk.ring_attention(dev(q), dev(k), dev(v), causal=True, cfg=mk.Config(max_ctas=max_ctas))
    _ok()
    exact = O.ring_attention([I.bits(t) for t in q], [I.bits(t) for t in k], [I.bits(t) for t in v],
                             True, w.scale, out="f32")
    vmax = max(float(t.float().abs().max()) for t in v)
    for r in range(w.R):
        assert _err(gpu_values(out[r]), exact[r].astype(np.float64), vmax) <= ATT_TOL


def test_ring_attention_missing_piece_times_out_and_recovers():
    w = I.AttnWorkload("t", R=2, heads=1, s_r=256, q_seed=55, k_seed=65, v_seed=75)
    q, k, v = (dev(x) for x in I.attn_inputs(w))
    ws = mk.Workspace()
    mk.ring_attention(q, k, v, workspace=ws, cfg=mk.Config(inject=1, wait_limit_ns=20_000_000))
    st, _ = mk.device_status(ws)
    assert st == mk.MK_ERR_TIMEOUT
    a = mk.ring_attention(q, k, v, workspace=ws)
    _ok(ws)
    b = mk.ring_attention(q, k, v, workspace=ws, cfg=mk.Config(mode=mk.MODE_GEMM_ONLY))
    _ok(ws)
    for r in range(w.R):
        assert torch.equal(a[r], b[r])


@pytest.mark.parametrize("causal", [False, True])
def test_ring_attention_full_size_row_sample(causal):
    # 8 ranks x 4096 positions (32768 in all), 8 heads of 128: sampled query rows of every rank
    w = I.RING_R8_H8_S4096_CAUSAL if causal else I.RING_R8_H8_S4096
    q, k, v = I.attn_inputs(w)
    ws = mk.Workspace()
    out = mk.ring_attention(dev(q), dev(k), dev(v), causal=causal, workspace=ws)
    _ok(ws)
    rows = [I.sample_rows(w.s_r, seed=40 + r, per_tile=1) for r in range(w.R)]
    exact = O.ring_attention([I.bits(t) for t in q], [I.bits(t) for t in k], [I.bits(t) for t in v],
                             causal, w.scale, out="f32", q_rows=rows)
    vmax = max(float(t.float().abs().max()) for t in v)
    for r in range(w.R):
        got = gpu_values(out[r][:, torch.from_numpy(rows[r]).cuda()])
        assert _err(got, exact[r].astype(np.float64), vmax) <= ATT_TOL


@pytest.mark.parametrize("causal", [False, True])
def test_ring_attention_large_scores(causal):
    # scale 1 instead of 1/sqrt(d): scores with a standard deviation near 11, so the
    # running maximum grows by more than 2^8 within a row (O rescaled) and most
    # exponentials fall far below 2^-100 (the clamped end of the polynomial)
    w = I.AttnWorkload("t", R=2, heads=2, s_r=384, causal=causal, q_seed=56, k_seed=66, v_seed=76)
    q, k, v = I.attn_inputs(w)
    out = mk.ring_attention(dev(q), dev(k), dev(v), causal=causal, scale=1.0)
    _ok()
    exact = O.ring_attention([I.bits(t) for t in q], [I.bits(t) for t in k], [I.bits(t) for t in v],
                             causal, 1.0, out="f32")
    vmax = max(float(t.float().abs().max()) for t in v)
    for r in range(w.R):
        assert _err(gpu_values(out[r]), exact[r].astype(np.float64), vmax) <= ATT_TOL


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mode", [mk.MODE_FUSED, mk.MODE_UNFUSED])
def test_ring_attention_stale_receive_rows_do_not_leak(mode, causal):
    # Ragged blocks (200 positions: the second key tile has 72 keys).  The
    # receive buffers start as NaN, so rows a tile would read past its block
    # (the next block, which may not have arrived) poison P V unless they read
    # as zeros; the result must be the GEMM-only mode's bits, which reads the
    # source blocks directly.
    wa = I.AttnWorkload("t", R=4, heads=2, s_r=200, causal=causal, q_seed=511, k_seed=512, v_seed=513)
    q, k, v = (dev(t) for t in I.attn_inputs(wa))
    want = mk.ring_attention(q, k, v, causal=causal, cfg=mk.Config(mode=mk.MODE_GEMM_ONLY))
    nan = lambda: [torch.full((3 * 2, 200, 128), float("nan"), dtype=torch.bfloat16, device="cuda")  # noqa: E731
                   for _ in range(4)]
    got = mk.ring_attention(q, k, v, causal=causal, k_recv=nan(), v_recv=nan(), cfg=mk.Config(mode=mode))
    _ok()
    for g, w in zip(got, want):
        assert not torch.isnan(g).any()
        assert torch.equal(g, w)
