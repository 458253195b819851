"""fp8 e4m3 operands for AllGather+GEMM, GEMM+ReduceScatter and GEMM+AllReduce
(GPU): tcgen05.mma kind::f8f6f4 with both operands K-major (B given as B^T),
fp32 accumulation, against the CPU oracle's exact fp8 definition.

Integer-valued operands (exact in e4m3) keep every fp32 sum exact, so the
results must match bit for bit, as must the gathered fp8 bytes of AG; normal
operands stay within the normalised fp32 tolerance of the exact product (the
inputs are fp8, the accumulation and the rounding are the kernel's).  Shapes
cover ragged k (a partial last 128-element k-block), ragged n, one and
several ranks, odd row-block counts with CTA pairs, pairs on and off, and the
two baseline modes.
"""
import numpy as np
import pytest
import torch

import oracle as O
import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import inputs as I
from parity_util import TOL, gpu_bits, gpu_values, norm_err, oracle_bits

pytestmark = pytest.mark.gpu
PAIRS = [mk.PAIR_OFF, mk.PAIR_ON]


@pytest.fixture(scope="module", autouse=True)
def built():
    from comm_gemm_tile_gb300 import build
    build.build()
    torch.cuda.init()


def _ok(ws=None):
    st, detail = mk.device_status(ws)
    assert st == mk.MK_OK, (mk.status_string(st), detail)


def _w(op, R, m, n, k, integer, seed, std=1.0):
    return I.GemmWorkload("t", op, R=R, m=m, n=n, k=k, out="bf16", a_std=std, b_std=std,
                          a_seed=seed, b_seed=seed + 1, integer=integer)


def _cuda(ts):
    return [t.cuda() for t in ts]


@pytest.mark.parametrize("pair", PAIRS)
@pytest.mark.parametrize("R,mr,n,k,local", [
    (1, 300, 256, 128, 0),     # 3 row blocks
    (4, 256, 512, 528, 2),     # ragged k: 4 k-blocks of 128 and one of 16
    (8, 256, 264, 256, 5),     # ragged n
    (4, 200, 512, 384, 1),     # shards straddle row blocks
])
def test_ag_fp8_integer_bit_exact(R, mr, n, k, local, pair):
    a, b = I.gemm_inputs_fp8(_w("ag", R, mr, n, k, True, 201))
    g, c = mk.ag_gemm(_cuda(a), b[0].cuda(), local_rank=local, cfg=mk.Config(cta_pair=pair))
    _ok()
    assert g.dtype == mk.FP8
    gathered, want = O.ag_gemm_fp8([I.fp8_bytes(x) for x in a], I.fp8_bytes(b[0]), "bf16")
    np.testing.assert_array_equal(I.fp8_bytes(g), gathered)
    np.testing.assert_array_equal(gpu_bits(c), want)


@pytest.mark.parametrize("R,mr,n,k", [(4, 256, 512, 512), (2, 384, 264, 1024)])
def test_ag_fp8_float_within_tolerance(R, mr, n, k):
    a, b = I.gemm_inputs_fp8(_w("ag", R, mr, n, k, False, 211))
    _, c = mk.ag_gemm(_cuda(a), b[0].cuda(), out_dtype=torch.float32)
    _ok()
    _, exact = O.ag_gemm_fp8([I.fp8_bytes(x) for x in a], I.fp8_bytes(b[0]), "f64")
    amax = max(float(x.float().abs().max()) for x in a)
    bmax = float(b[0].float().abs().max())
    assert norm_err(gpu_values(c), exact, k, amax, bmax) <= TOL["f32"]


@pytest.mark.parametrize("mode", [mk.MODE_GEMM_ONLY, mk.MODE_UNFUSED])
def test_ag_fp8_baseline_modes(mode):
    a, b = I.gemm_inputs_fp8(_w("ag", 4, 256, 512, 256, True, 221))
    da = _cuda(a)
    if mode == mk.MODE_GEMM_ONLY:   # the GEMM reads a gathered A that is already filled
        gathered = torch.cat([t.view(torch.uint8) for t in da], 0).view(mk.FP8)
        _, c = mk.ag_gemm(da, b[0].cuda(), a_gathered=gathered, cfg=mk.Config(mode=mode))
    else:
        _, c = mk.ag_gemm(da, b[0].cuda(), cfg=mk.Config(mode=mode))
    _ok()
    _, want = O.ag_gemm_fp8([I.fp8_bytes(x) for x in a], I.fp8_bytes(b[0]), "bf16")
    np.testing.assert_array_equal(gpu_bits(c), want)


@pytest.mark.parametrize("pair", PAIRS)
@pytest.mark.parametrize("op,R,m,n,k", [
    ("rs", 4, 520, 520, 256),     # 5 row blocks, ragged n
    ("rs", 8, 1024, 512, 512),
    ("rs", 1, 136, 256, 144),      # one rank, ragged k
    ("ar", 8, 128, 1032, 512),
    ("ar", 2, 384, 264, 160),
])
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_rs_ar_fp8_integer_bit_exact(op, R, m, n, k, pair, out):
    a, b = I.gemm_inputs_fp8(_w(op, R, m, n, k, True, 231))
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    cfg = mk.Config(cta_pair=pair)
    if op == "rs":
        got = torch.cat(mk.gemm_rs(_cuda(a), _cuda(b), out_dtype=dt, cfg=cfg), 0)
    else:
        reps = mk.gemm_ar(_cuda(a), _cuda(b), out_dtype=dt, cfg=cfg)
        for r in reps[1:]:
            assert torch.equal(r, reps[0])
        got = reps[0]
    _ok()
    exact = O.sum_over_ranks_fp8([I.fp8_bytes(x) for x in a], [I.fp8_bytes(x) for x in b])
    np.testing.assert_array_equal(gpu_bits(got), oracle_bits(exact, out))


def test_rs_fp8_float_within_tolerance_and_reduction_variants():
    R, m, n, k = 4, 512, 512, 512
    a, b = I.gemm_inputs_fp8(_w("rs", R, m, n, k, False, 241))
    exact = O.sum_over_ranks_fp8([I.fp8_bytes(x) for x in a], [I.fp8_bytes(x) for x in b])
    amax = max(float(x.float().abs().max()) for x in a)
    bmax = max(float(x.float().abs().max()) for x in b)
    for cfg in (mk.Config(), mk.Config(reduce=mk.REDUCE_ATOMIC), mk.Config(wire=mk.WIRE_BF16)):
        got = torch.cat(mk.gemm_rs(_cuda(a), _cuda(b), out_dtype=torch.float32, cfg=cfg), 0)
        _ok()
        tol = TOL["f32"] if cfg.wire == 0 else TOL["bf16"]
        assert norm_err(gpu_values(got), exact, R * k, amax, bmax) <= tol


def test_fp8_rejected_by_ops_without_it():
    x = [torch.zeros((64, 256), dtype=mk.FP8, device="cuda") for _ in range(2)]
    with pytest.raises(mk.MkError):
        mk.ring_attention([torch.zeros((1, 128, 128), dtype=torch.bfloat16, device="cuda")] * 2,
                          [torch.zeros((1, 128, 128), dtype=torch.bfloat16, device="cuda")] * 2,
                          [torch.zeros((1, 128, 128), dtype=torch.bfloat16, device="cuda")] * 2,
                          cfg=mk.Config(operand=mk.OPERAND_FP8))
    del x


def test_ag_fp8_copy_role_ctas_and_missing_piece():
    a, b = I.gemm_inputs_fp8(_w("ag", 4, 256, 512, 256, True, 251))
    _, want = O.ag_gemm_fp8([I.fp8_bytes(x) for x in a], I.fp8_bytes(b[0]), "bf16")
    # copy-role CTAs (bulk copies of fp8 rows) instead of the compute CTAs' copy warps
    _, c = mk.ag_gemm(_cuda(a), b[0].cuda(), cfg=mk.Config(n_copy_ctas=8))
    _ok()
    np.testing.assert_array_equal(gpu_bits(c), want)
    # a copy piece that never signals: the bounded waits report a timeout, and the next
    # call on the same workspace is correct
    ws = mk.Workspace()
    mk.ag_gemm(_cuda(a), b[0].cuda(), workspace=ws, cfg=mk.Config(inject=1, wait_limit_ns=20_000_000))
    st, _ = mk.device_status(ws)
    assert st == mk.MK_ERR_TIMEOUT
    _, c = mk.ag_gemm(_cuda(a), b[0].cuda(), workspace=ws)
    _ok(ws)
    np.testing.assert_array_equal(gpu_bits(c), want)
