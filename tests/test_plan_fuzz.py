"""Host planning of the AG / RS / AR, MoE and ring-attention workspaces (CPU, no
launch): for random shapes and configs the workspace sizes are non-zero exactly when
the arguments are valid, and the trace region sits after the untraced layout."""
import ctypes

import pytest

import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import build as mkbuild

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")


@pytest.fixture(scope="module")
def L():
    mkbuild.build()
    return mk.lib()


def valid(op, R, m, n, k, c):
    if not (1 <= R <= mk.MAX_RANKS) or min(m, n, k) < 0 or n % 8 or k % 8:
        return False
    if not (0 <= c.mode <= 2) or not (0 <= c.reduce <= 4) or not (0 <= c.wire <= 1):
        return False
    if not (0 <= c.operand <= 1) or c.trace not in (0, 1):
        return False
    if c.operand == 1 and k % 16:
        return False
    M = m * R if op == mk.OP_AG_GEMM else m
    if max(M, n, k) >= 1 << 31:
        return False
    if op == mk.OP_GEMM_RS and m % R:
        return False
    return True


dims = st.one_of(st.integers(0, 4096), st.sampled_from([8, 16, 128, 136, 1 << 31, -8]))


@hyp.settings(max_examples=400, deadline=None)
@hyp.given(op=st.sampled_from([mk.OP_AG_GEMM, mk.OP_GEMM_RS, mk.OP_GEMM_AR]),
           R=st.integers(-1, 18), m=dims, n=dims, k=dims,
           mode=st.integers(-1, 3), reduce=st.integers(-1, 5), wire=st.integers(-1, 2),
           operand=st.integers(-1, 2), trace=st.integers(-1, 2), split_k=st.integers(0, 9),
           n_reduce=st.sampled_from([0, 0, 4]))
def test_workspace_size_matches_validity(L, op, R, m, n, k, mode, reduce, wire, operand, trace,
                                         split_k, n_reduce):
    c = mk.Config(mode=mode, reduce=reduce, wire=wire, operand=operand, trace=trace,
                  split_k=split_k, n_reduce_ctas=n_reduce)
    size = L.mk_workspace_size(op, R, m, n, k, ctypes.byref(c.c()))
    assert (size > 0) == valid(op, R, m, n, k, c)
    if size and trace == 1:
        base = L.mk_workspace_size(op, R, m, n, k, ctypes.byref(mk.Config(
            mode=mode, reduce=reduce, wire=wire, operand=operand, split_k=split_k,
            n_reduce_ctas=n_reduce).c()))
        off = ctypes.c_size_t(0)
        n_rec = L.mk_trace_entries(op, R, m, n, k, ctypes.byref(c.c()), ctypes.byref(off))
        assert n_rec > 0 and off.value >= base and off.value % 256 == 0
        assert size == off.value + (n_rec + mk.TRACE_COPY_RECORDS) * 64


def moe_valid(R, E_loc, topk, T, H, N, cap, trace):
    if not (1 <= R <= mk.MAX_RANKS) or E_loc < 1:
        return False
    E = R * E_loc
    if E > 256 or not (1 <= topk <= 8) or topk > E:
        return False
    if min(T, H, N, cap) < 0 or H % 8 or N % 8 or trace not in (0, 1):
        return False
    rows = R * T * topk
    if rows >= 1 << 31 or cap >= 1 << 31 or H >= 1 << 31 or N >= 1 << 31 or cap * H >= 1 << 40:
        return False
    n_nblk = -(-N // 256)
    return (rows // 128 + E) * n_nblk < 1 << 30


@hyp.settings(max_examples=400, deadline=None)
@hyp.given(R=st.integers(-1, 18), E_loc=st.integers(-1, 40), topk=st.integers(-1, 10),
           T=st.one_of(st.integers(0, 5000), st.sampled_from([-1, 1 << 28])),
           H=st.one_of(st.integers(0, 9000), st.sampled_from([-8, 1 << 31])),
           N=st.one_of(st.integers(0, 9000), st.sampled_from([-8, 1 << 31])),
           cap=st.one_of(st.integers(0, 1 << 20), st.sampled_from([-1, 1 << 31, 1 << 33])),
           trace=st.integers(-1, 2))
def test_moe_workspace_size_matches_validity(L, R, E_loc, topk, T, H, N, cap, trace):
    c = mk.Config(trace=trace)
    size = L.mk_moe_workspace_size(R, E_loc, topk, T, H, N, cap, ctypes.byref(c.c()))
    assert (size > 0) == moe_valid(R, E_loc, topk, T, H, N, cap, trace)
    if size and trace == 1:
        off = ctypes.c_size_t(0)
        n_rec = L.mk_moe_trace_entries(R, E_loc, topk, T, H, N, cap, ctypes.byref(c.c()),
                                       ctypes.byref(off))
        base = L.mk_moe_workspace_size(R, E_loc, topk, T, H, N, cap, None)
        assert n_rec > 0 and off.value >= base
        assert size >= off.value + (n_rec + mk.TRACE_COPY_RECORDS) * 64


@hyp.settings(max_examples=300, deadline=None)
@hyp.given(R=st.integers(-1, 10), heads=st.integers(-1, 70), s_r=st.one_of(
               st.integers(-1, 70000), st.sampled_from([1 << 20, 1 << 24])),
           d=st.sampled_from([64, 128, 127, 256]), causal=st.integers(0, 1))
def test_attention_workspace_size_matches_validity(L, R, heads, s_r, d, causal):
    size = L.mk_ring_attention_workspace_size(R, heads, s_r, d, causal, None)
    ok = 1 <= R <= 8 and heads >= 1 and s_r >= 0 and d == 128 and heads * s_r < (1 << 31) // 128
    assert (size > 0) == ok
