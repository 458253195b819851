"""mk_ag_gemm_noalloc: AllGather + GEMM without a caller-supplied workspace.

Some callers cannot allocate device memory (a plug-in inside an application
that owns every GPU byte through its own pool, or a path that must not
allocate after start-up).  For them the library keeps the kernel's small
scratch in a fixed array of its own.  These tests call that entry point
through the C ABI and check it against the ordinary mk_ag_gemm (bit for bit:
the same kernel) and the oracle, twice in a row, since every call reuses the
same array, and once more after a call that timed out and left its error
words in that array.  This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import inputs as I
import oracle as O
from parity_util import TOL, absmax, dev, gpu_values, norm_err

NOALLOC_SCRATCH_BYTES = 65536


def _noalloc(L, shards, b, g, c, local, status_dev=None, cfg=None, stream=None):
    arr = (ctypes.c_void_p * len(shards))(*[s.data_ptr() for s in shards])
    m_r, k = shards[0].shape
    n = b.shape[1]
    dt = mk.MK_BF16 if c.dtype == torch.bfloat16 else mk.MK_F32
    st = torch.cuda.current_stream().cuda_stream if stream is None else stream
    return L.mk_ag_gemm_noalloc(arr, b.data_ptr(), g.data_ptr(), c.data_ptr(), dt, len(shards),
                                local, m_r, n, k,
                                None if status_dev is None else status_dev.data_ptr(),
                                None if cfg is None else ctypes.byref(cfg.c()), st)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    from comm_gemm_tile_gb300 import build
    build.build()
    L = mk.lib()
    ptrs = (ctypes.c_void_p * 2)(0x10000, 0x10000)
    # 2 x 70000 gathered rows need about 1100 chunks of flags: more than the array holds
    assert mk.workspace_size(mk.OP_AG_GEMM, 2, 70000, 8, 8) > NOALLOC_SCRATCH_BYTES
    assert L.mk_ag_gemm_noalloc(ptrs, 0x10000, 0x10000, 0x10000, mk.MK_BF16, 2, 0, 70000, 8, 8,
                                None, None, None) == mk.MK_ERR_INVALID


def test_noalloc_rejects_trace():
    # a trace would be written into the library's own array, out of the caller's reach
    from comm_gemm_tile_gb300 import build
    build.build()
    L = mk.lib()
    ptrs = (ctypes.c_void_p * 2)(0x10000, 0x10000)
    cfg = mk.Config(trace=1).c()
    assert L.mk_ag_gemm_noalloc(ptrs, 0x10000, 0x10000, 0x10000, mk.MK_BF16, 2, 0, 128, 64, 64,
                                None, ctypes.byref(cfg), None) == mk.MK_ERR_INVALID


def _run(L, w, local, dtype, status):
    """One mk_ag_gemm (caller workspace) and two back-to-back mk_ag_gemm_noalloc
    calls on the same inputs; both no-alloc results must equal the workspace
    call's bit for bit (the same kernel and launch configuration)."""
    a, b = I.gemm_inputs(w)
    shards, bd = dev(a), b[0].cuda()
    g_ref, c_ref = mk.ag_gemm(shards, bd, local_rank=local, out_dtype=dtype)
    st_ref, _ = mk.device_status()
    assert st_ref == mk.MK_OK
    for _ in range(2):   # the second call finds the first call's contents in the shared array
        g = torch.zeros_like(g_ref)
        c = torch.zeros_like(c_ref)
        status.fill_(-1)
        assert _noalloc(L, shards, bd, g, c, local, status_dev=status) == mk.MK_OK
        torch.cuda.synchronize()
        assert int(status.item()) == mk.MK_OK
        assert torch.equal(g, g_ref)                       # the gathered A is a bit copy
        assert torch.equal(c, c_ref)
    return a, b, g, c


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    from comm_gemm_tile_gb300 import build
    build.build()
    L = mk.lib()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    cases = [  # (R, m_r, n, k, local, out dtype, seed): several tiles, ragged n and k
        (4, 256, 264, 520, 1, torch.bfloat16, 11),
        (8, 128, 512, 256, 6, torch.float32, 12),
    ]
    for R, mr, n, k, local, dtype, seed in cases:
        out = "bf16" if dtype == torch.bfloat16 else "f32"
        w = I.GemmWorkload("noalloc", "ag", R=R, m=mr, n=n, k=k, out=out, a_seed=seed, b_seed=seed + 100)
        a, b, g, c = _run(L, w, local, dtype, status)
        _, exact = O.ag_gemm([I.bits(x) for x in a], I.bits(b[0]), out="f64")
        assert norm_err(gpu_values(c), exact, k, absmax(a), absmax(b)) <= TOL[out]


@pytest.mark.gpu
def test_noalloc_integer_twin_bit_exact_and_recovers_after_timeout():
    from comm_gemm_tile_gb300 import build
    build.build()
    L = mk.lib()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    w = I.GemmWorkload("noalloc_int", "ag", R=4, m=256, n=520, k=264, out="bf16", a_seed=13,
                       b_seed=113, integer=True)
    a, b, g, c = _run(L, w, 2, torch.bfloat16, status)
    a_bits, b_bits = [I.bits(x) for x in a], I.bits(b[0])
    gathered, want = O.ag_gemm(a_bits, b_bits, out="bf16")
    np.testing.assert_array_equal(I.bits(g), gathered)
    np.testing.assert_array_equal(I.bits(c), want)
    # a call whose copy-in drops one ready signal times out (20 ms) and leaves its status,
    # detail and abort words in the shared array; the next call clears them and is exact
    shards, bd = dev(a), b[0].cuda()
    status.fill_(-1)
    assert _noalloc(L, shards, bd, torch.zeros_like(g), torch.zeros_like(c), 2, status_dev=status,
                    cfg=mk.Config(inject=1, wait_limit_ns=20_000_000)) == mk.MK_OK
    torch.cuda.synchronize()
    assert int(status.item()) == mk.MK_ERR_TIMEOUT
    g2, c2 = torch.zeros_like(g), torch.zeros_like(c)
    status.fill_(-1)
    assert _noalloc(L, shards, bd, g2, c2, 2, status_dev=status) == mk.MK_OK
    torch.cuda.synchronize()
    assert int(status.item()) == mk.MK_OK
    np.testing.assert_array_equal(I.bits(g2), gathered)
    np.testing.assert_array_equal(I.bits(c2), want)
