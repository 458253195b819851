"""The C-ABI library: it loads, exports every entry point declared in
include/mk.h, and rejects bad arguments before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import build as mkbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    mkbuild.build()
    return mk.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mk.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mk_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_bounds_build_exports_the_same_symbols():
    # libmk_debug.so: the same sources with MK_DEBUG_BOUNDS=1 (device-side index checks)
    mkbuild.build(debug=True)
    D = mk.load_library(mk.LIB_DEBUG_PATH)
    for n in declared_functions():
        assert hasattr(D, n), n
    assert D.mk_version() == 1


def test_version_and_status_strings(L):
    assert L.mk_version() == 1
    assert "timed out" in mk.status_string(mk.MK_ERR_TIMEOUT)
    assert "capacity" in mk.status_string(mk.MK_ERR_CAPACITY)
    assert mk.status_string(99) == "unknown status"


def test_workspace_sizes(L):
    # RS, 8 ranks, 8192x8192 output, default (running sum per tile): 2048 fp32 tiles of 128x256.
    sz = mk.workspace_size(mk.OP_GEMM_RS, 8, 8192, 8192, 3584)
    assert 2048 * 128 * 256 * 4 <= sz < 2048 * 128 * 256 * 4 + (1 << 20)
    # staged partials for reduce-role CTAs: 8 fp32 partial tiles per output tile.
    sz = mk.workspace_size(mk.OP_GEMM_RS, 8, 8192, 8192, 3584, mk.Config(n_reduce_ctas=8))
    assert 2048 * 8 * 128 * 256 * 4 <= sz < 2048 * 8 * 128 * 256 * 4 + (1 << 20)
    sz = mk.workspace_size(mk.OP_GEMM_RS, 8, 8192, 8192, 3584, mk.Config(mode=mk.MODE_UNFUSED))
    assert 2048 * 8 * 128 * 256 * 4 <= sz
    # atomic reduction: one fp32 tile per output tile, like the running sum
    sz = mk.workspace_size(mk.OP_GEMM_RS, 8, 8192, 8192, 3584, mk.Config(reduce=mk.REDUCE_ATOMIC))
    assert 2048 * 128 * 256 * 4 <= sz < 2048 * 128 * 256 * 4 + (1 << 20)
    # bf16 wire: the same staging (half of each tile used)
    assert mk.workspace_size(mk.OP_GEMM_RS, 8, 8192, 8192, 3584, mk.Config(wire=mk.WIRE_BF16)) > 0
    # sliced reduction: every partial staged (8 fp32 partial tiles per output tile)
    sz = mk.workspace_size(mk.OP_GEMM_RS, 8, 8192, 8192, 3584, mk.Config(reduce=mk.REDUCE_SLICED))
    assert 2048 * 8 * 128 * 256 * 4 <= sz < 2048 * 8 * 128 * 256 * 4 + (1 << 20)
    # AR defaults: the decode shape (32 output tiles x 8 partials <= 2048) reduces by
    # slices (all partials staged); a large AR keeps one running-sum tile per output tile
    sz = mk.workspace_size(mk.OP_GEMM_AR, 8, 128, 8192, 3584)
    assert 32 * 8 * 128 * 256 * 4 <= sz < 32 * 8 * 128 * 256 * 4 + (1 << 20)
    assert sz == mk.workspace_size(mk.OP_GEMM_AR, 8, 128, 8192, 3584, mk.Config(reduce=mk.REDUCE_SLICED))
    sz = mk.workspace_size(mk.OP_GEMM_AR, 8, 8192, 8192, 3584)
    assert 2048 * 128 * 256 * 4 <= sz < 2048 * 128 * 256 * 4 + (1 << 20)
    # the running sum chosen explicitly, or with the bf16 wire: one tile per output tile
    for cfg in (mk.Config(reduce=mk.REDUCE_RUNNING_SUM), mk.Config(wire=mk.WIRE_BF16)):
        sz = mk.workspace_size(mk.OP_GEMM_AR, 8, 128, 8192, 3584, cfg)
        assert 32 * 128 * 256 * 4 <= sz < 32 * 128 * 256 * 4 + (1 << 20)
    # out-of-range reduce / wire -> 0
    assert mk.workspace_size(mk.OP_GEMM_RS, 8, 8192, 8192, 3584, mk.Config(reduce=5)) == 0
    assert mk.workspace_size(mk.OP_GEMM_RS, 8, 8192, 8192, 3584, mk.Config(wire=2)) == 0
    # fp8 operands: k must be a multiple of 16 (rows of whole 16-byte units)
    assert mk.workspace_size(mk.OP_AG_GEMM, 8, 1024, 3584, 8192, mk.Config(operand=mk.OPERAND_FP8)) > 0
    assert mk.workspace_size(mk.OP_GEMM_RS, 2, 256, 256, 24, mk.Config(operand=mk.OPERAND_FP8)) == 0
    assert mk.workspace_size(mk.OP_GEMM_RS, 2, 256, 256, 24) > 0
    assert mk.workspace_size(mk.OP_GEMM_RS, 2, 256, 256, 64, mk.Config(operand=2)) == 0
    # GEMM-only mode needs no staging.
    assert mk.workspace_size(mk.OP_GEMM_RS, 8, 8192, 8192, 3584,
                             mk.Config(mode=mk.MODE_GEMM_ONLY)) < (1 << 20)
    # AG: up to 16 sub-chunk flags per 128-row chunk of the gathered A (64 chunks).
    assert 256 + 64 * 16 * 4 <= mk.workspace_size(mk.OP_AG_GEMM, 8, 1024, 3584, 8192) < 8192
    # bad shapes -> 0
    assert mk.workspace_size(mk.OP_GEMM_RS, 8, 8190, 64, 64) == 0     # m % R
    assert mk.workspace_size(mk.OP_GEMM_RS, 2, 256, 260, 64) == 0     # n % 8
    assert mk.workspace_size(mk.OP_GEMM_RS, 2, 256, 256, 60) == 0     # k % 8
    assert mk.workspace_size(mk.OP_GEMM_RS, 0, 256, 256, 64) == 0     # R
    assert mk.workspace_size(mk.OP_GEMM_RS, 17, 17 * 16, 256, 64) == 0
    # AR split-K keeps at most 16 partials per tile
    assert mk.workspace_size(mk.OP_GEMM_AR, 8, 128, 8192, 3584) <= 32 * 16 * 128 * 256 * 4 + (1 << 20)


def test_combine_workspace_sizes(L):
    # 8 ranks x 8 experts, T=4096, top-2, N=1536 -> H=4096 (16 column blocks)
    sz = mk.moe_combine_workspace_size(8, 8, 2, 4096, 1536, 4096, 65536)
    cnt = 8 * 4096 * 16 * 4
    tiles = (8 * 4096 * 2 // 128 + 64) * 16 * 5 * 4
    assert cnt + tiles <= sz < cnt + tiles + (1 << 16)
    assert mk.moe_combine_workspace_size(8, 8, 2, 4096, 1532, 4096, 65536) == 0   # N % 8
    assert mk.moe_combine_workspace_size(8, 8, 2, 4096, 1536, 4100, 65536) == 0   # H % 8
    assert mk.moe_combine_workspace_size(8, 8, 9, 4096, 1536, 4096, 65536) == 0   # topk > 8
    assert mk.moe_combine_workspace_size(16, 17, 2, 64, 64, 64, 64) == 0          # E > 256


def test_combine_argument_validation_without_launch(L):
    V = ctypes.c_void_p
    good = 0x10000
    ws = V(good)
    arr = (ctypes.c_void_p * 2)(good, good)
    args = (arr, arr, arr, arr, V(good), 2, 2, 2, 64, 64, 256, 256, arr, arr, ws, 1 << 20, None, None)
    # NULL pointer arrays, misaligned rows, small workspace, bad topk
    assert L.mk_moe_combine(None, *args[1:]) == mk.MK_ERR_INVALID
    a = list(args); a[0] = _null_ptrs(2)
    assert L.mk_moe_combine(*a) == mk.MK_ERR_INVALID
    a = list(args); a[12] = (ctypes.c_void_p * 2)(good, good + 2)
    assert L.mk_moe_combine(*a) == mk.MK_ERR_INVALID
    a = list(args); a[15] = 16
    assert L.mk_moe_combine(*a) == mk.MK_ERR_INVALID
    a = list(args); a[7] = 0
    assert L.mk_moe_combine(*a) == mk.MK_ERR_INVALID
    cfg = mk.Config(mode=7).c()
    a = list(args); a[16] = ctypes.pointer(cfg)
    assert L.mk_moe_combine(*a) == mk.MK_ERR_INVALID


def _null_ptrs(n):
    return (ctypes.c_void_p * n)()


def test_argument_validation_without_launch(L):
    V = ctypes.c_void_p
    good = 0x10000
    ws = V(good)
    arr = (ctypes.c_void_p * 2)(good, good)
    # NULL shard array
    assert L.mk_ag_gemm(None, V(good), V(good), V(good), 0, 2, 0, 128, 256, 64, ws, 1 << 20,
                        None, None) == mk.MK_ERR_INVALID
    # NULL entry inside the array
    assert L.mk_ag_gemm(_null_ptrs(2), V(good), V(good), V(good), 0, 2, 0, 128, 256, 64, ws,
                        1 << 20, None, None) == mk.MK_ERR_INVALID
    # local rank out of range
    assert L.mk_ag_gemm(arr, V(good), V(good), V(good), 0, 2, 2, 128, 256, 64, ws, 1 << 20, None,
                        None) == mk.MK_ERR_INVALID
    # misaligned pointer
    bad = (ctypes.c_void_p * 2)(good, good + 8)
    assert L.mk_ag_gemm(bad, V(good), V(good), V(good), 0, 2, 0, 128, 256, 64, ws, 1 << 20, None,
                        None) == mk.MK_ERR_INVALID
    # workspace too small
    assert L.mk_ag_gemm(arr, V(good), V(good), V(good), 0, 2, 0, 128, 256, 64, ws, 16, None,
                        None) == mk.MK_ERR_INVALID
    # bad dtype
    assert L.mk_ag_gemm(arr, V(good), V(good), V(good), 7, 2, 0, 128, 256, 64, ws, 1 << 20, None,
                        None) == mk.MK_ERR_INVALID
    # RS: m not a multiple of R
    assert L.mk_gemm_rs(arr, arr, arr, 0, 2, 255, 256, 64, ws, 1 << 30, None, None) == \
        mk.MK_ERR_INVALID
    # RS/AR: k not a multiple of 8, R too large
    assert L.mk_gemm_ar(arr, arr, arr, 0, 2, 128, 256, 60, ws, 1 << 30, None, None) == \
        mk.MK_ERR_INVALID
    assert L.mk_gemm_ar(arr, arr, arr, 0, 17, 128, 256, 64, ws, 1 << 30, None, None) == \
        mk.MK_ERR_INVALID
    # NULL workspace / status read
    assert L.mk_gemm_rs(arr, arr, arr, 0, 2, 256, 256, 64, None, 0, None, None) == \
        mk.MK_ERR_INVALID
    assert L.mk_get_device_status(None, None, None) == mk.MK_ERR_INVALID


def test_trace_layout(L):
    off = ctypes.c_size_t(7)
    cfg_off = mk.Config()
    cfg_on = mk.Config(trace=1)
    assert L.mk_trace_entries(mk.OP_GEMM_RS, 8, 8192, 8192, 3584, ctypes.byref(cfg_off.c()),
                              ctypes.byref(off)) == 0 and off.value == 0
    n = L.mk_trace_entries(mk.OP_GEMM_RS, 8, 8192, 8192, 3584, ctypes.byref(cfg_on.c()), ctypes.byref(off))
    # two records (8 x u64) per (tile, partial): 2048 tiles x 8 ranks
    assert n == 2048 * 8 * 2 and off.value % 256 == 0
    base = mk.workspace_size(mk.OP_GEMM_RS, 8, 8192, 8192, 3584)
    assert off.value >= base
    assert mk.workspace_size(mk.OP_GEMM_RS, 8, 8192, 8192, 3584, cfg_on) == \
        off.value + (n + mk.TRACE_COPY_RECORDS) * 64
    n = L.mk_trace_entries(mk.OP_AG_GEMM, 8, 1024, 3584, 8192, ctypes.byref(cfg_on.c()), ctypes.byref(off))
    assert n == 64 * 14 * 2
    assert mk.workspace_size(mk.OP_GEMM_RS, 8, 8192, 8192, 3584, mk.Config(trace=2)) == 0
    # the chained MLP: two records per up-projection tile (64 row tiles x 8 ranks x 14
    # column tiles) and per down-projection (tile, rank) part (64 x 32 tiles x 8 ranks)
    n = L.mk_mlp_trace_entries(8, 1024, 8192, 3584, ctypes.byref(cfg_on.c()), ctypes.byref(off))
    assert n == 2 * (64 * 8 * 14 + 64 * 32 * 8) and off.value % 256 == 0
    assert off.value >= mk.mlp_workspace_size(8, 1024, 8192, 3584)
    assert mk.mlp_workspace_size(8, 1024, 8192, 3584, mk.Config(trace=1)) == \
        off.value + (n + mk.TRACE_COPY_RECORDS) * 64
    assert L.mk_mlp_trace_entries(8, 1024, 8192, 3584, ctypes.byref(cfg_off.c()), ctypes.byref(off)) == 0
    assert mk.mlp_workspace_size(8, 1024, 8192, 3584, mk.Config(trace=1, mode=mk.MODE_UNFUSED)) == 0


def test_moe_trace_layout(L):
    off = ctypes.c_size_t(7)
    args = (8, 8, 2, 4096, 4096, 1536, 65536)
    assert L.mk_moe_trace_entries(*args, ctypes.byref(mk.Config().c()), ctypes.byref(off)) == 0
    assert off.value == 0
    on = mk.Config(trace=1)
    n = L.mk_moe_trace_entries(*args, ctypes.byref(on.c()), ctypes.byref(off))
    # two records per tile-table entry: (65536 / 128 + 64) row tiles x 6 column tiles
    assert n == 2 * (65536 // 128 + 64) * 6
    assert off.value >= mk.moe_workspace_size(*args) and off.value % 256 == 0
    assert mk.moe_workspace_size(*args, cfg=on) >= off.value + (n + mk.TRACE_COPY_RECORDS) * 64
    assert mk.moe_workspace_size(*args, cfg=mk.Config(trace=2)) == 0


def test_trace_copy_record_count_matches_header():
    hdr = open(os.path.join(ROOT, "include", "mk.h")).read()
    assert int(re.search(r"#define MK_TRACE_COPY_RECORDS (\d+)", hdr).group(1)) == mk.TRACE_COPY_RECORDS


def test_mlp_rejects_the_reduction_variants(L):
    # the chained MLP reduces by the fp32 running sum only
    assert mk.mlp_workspace_size(8, 1024, 8192, 3584) > 0
    assert mk.mlp_workspace_size(8, 1024, 8192, 3584, mk.Config(reduce=mk.REDUCE_ATOMIC)) == 0
    assert mk.mlp_workspace_size(8, 1024, 8192, 3584, mk.Config(wire=mk.WIRE_BF16)) == 0
    assert mk.mlp_workspace_size(8, 1024, 8192, 3584, mk.Config(reduce=mk.REDUCE_LAST_ARRIVAL)) == 0


def test_config_struct_layout():
    assert ctypes.sizeof(mk._Cfg) == 56
    assert mk._Cfg.wait_limit_ns.offset == 24 and mk._Cfg.inject.offset == 32
    assert mk._Cfg.reduce.offset == 36 and mk._Cfg.cta_pair.offset == 40
    assert mk._Cfg.wire.offset == 44 and mk._Cfg.operand.offset == 48 and mk._Cfg.trace.offset == 52
