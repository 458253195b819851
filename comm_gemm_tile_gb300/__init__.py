"""Python binding of libmk.so: tile-pipelined fused collective + GEMM on one GB300.

Argument marshalling only.  Every step of every op runs in the CUDA library
(include/mk.h); PyTorch provides device memory and streams.  If the library is
missing the calls raise -- there is no fallback path.

The R virtual ranks of an op are R separate device buffers on one GPU.
"""
from __future__ import annotations

import ctypes
import math
import dataclasses
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmk.so")

MK_OK, MK_ERR_INVALID, MK_ERR_UNSUPPORTED, MK_ERR_CUDA, MK_ERR_TIMEOUT, MK_ERR_CAPACITY = range(6)
MK_BF16, MK_F32 = 0, 1
OP_AG_GEMM, OP_GEMM_RS, OP_GEMM_AR, OP_MOE = 0, 1, 2, 3
MODE_FUSED, MODE_GEMM_ONLY, MODE_UNFUSED = 0, 1, 2
REDUCE_AUTO, REDUCE_RUNNING_SUM, REDUCE_LAST_ARRIVAL, REDUCE_ATOMIC, REDUCE_SLICED = 0, 1, 2, 3, 4
WIRE_F32, WIRE_BF16 = 0, 1
OPERAND_BF16, OPERAND_FP8 = 0, 1
FP8 = torch.float8_e4m3fn
# columns of trace_records()
(TRACE_START, TRACE_INPUTS, TRACE_ISSUED, TRACE_READY, TRACE_END, TRACE_CLK_START,
 TRACE_CLK_READY, TRACE_ID) = range(8)
TRACE_WORDS = 8
TRACE_COPY_RECORDS = 1024


def _with_operand(cfg, t):
    """The config for operands of t's dtype: fp8 e4m3 tensors set operand = 1."""
    if t.dtype != FP8:
        return cfg
    c = dataclasses.replace(cfg) if cfg is not None else Config()
    c.operand = OPERAND_FP8
    return c
PAIR_AUTO, PAIR_OFF, PAIR_ON = 0, 1, 2
MAX_RANKS = 16


class MkError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class _Cfg(ctypes.Structure):
    _fields_ = [("n_copy_ctas", ctypes.c_int), ("n_reduce_ctas", ctypes.c_int),
                ("max_ctas", ctypes.c_int), ("group_m", ctypes.c_int), ("split_k", ctypes.c_int),
                ("mode", ctypes.c_int), ("wait_limit_ns", ctypes.c_longlong),
                ("inject", ctypes.c_int), ("reduce", ctypes.c_int), ("cta_pair", ctypes.c_int),
                ("wire", ctypes.c_int), ("operand", ctypes.c_int), ("trace", ctypes.c_int)]


@dataclasses.dataclass
class Config:
    """Tuning / test knobs (mk_config); 0 means the library's own choice."""
    n_copy_ctas: int = 0
    n_reduce_ctas: int = 0
    max_ctas: int = 0
    group_m: int = 0
    split_k: int = 0
    mode: int = MODE_FUSED
    wait_limit_ns: int = 0
    inject: int = 0
    reduce: int = 0
    cta_pair: int = 0
    wire: int = 0
    operand: int = 0
    trace: int = 0

    def c(self) -> _Cfg:
        return _Cfg(self.n_copy_ctas, self.n_reduce_ctas, self.max_ctas, self.group_m,
                    self.split_k, self.mode, self.wait_limit_ns, self.inject, self.reduce,
                    self.cta_pair, self.wire, self.operand, self.trace)


_lib = None
_lib_lock = threading.Lock()


LIB_DEBUG_PATH = os.path.join(_HERE, "libmk_debug.so")


def lib() -> ctypes.CDLL:
    """Load libmk.so (built in-tree by build.py).  Raises if it is missing."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        _lib = load_library(LIB_PATH)
        return _lib


class use_library:
    """Context manager: every op of this module calls the given library (for
    example the bounds-checking LIB_DEBUG_PATH) instead of libmk.so."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.prev = lib()
        with _lib_lock:
            _lib = load_library(self.path)
        return _lib

    def __exit__(self, *exc):
        global _lib
        with _lib_lock:
            _lib = self.prev
        return False


def load_library(path: str) -> ctypes.CDLL:
    """Open a build of the library and declare its C ABI."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run comm_gemm_tile_gb300/build.py "
                           "(or __graft_entry__.build())")
    L = ctypes.CDLL(path)
    vp, sz, ll, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_longlong, ctypes.c_int
    P = ctypes.POINTER
    L.mk_version.restype = i
    L.mk_device_sm_count.restype = i
    L.mk_status_string.restype = ctypes.c_char_p
    L.mk_status_string.argtypes = [i]
    L.mk_workspace_size.restype = sz
    L.mk_workspace_size.argtypes = [i, i, ll, ll, ll, P(_Cfg)]
    L.mk_trace_entries.restype = sz
    L.mk_trace_entries.argtypes = [i, i, ll, ll, ll, P(_Cfg), P(sz)]
    L.mk_moe_trace_entries.restype = sz
    L.mk_moe_trace_entries.argtypes = [i, i, i, ll, ll, ll, ll, P(_Cfg), P(sz)]
    L.mk_mlp_trace_entries.restype = sz
    L.mk_mlp_trace_entries.argtypes = [i, ll, ll, ll, P(_Cfg), P(sz)]
    L.mk_moe_workspace_size.restype = sz
    L.mk_moe_workspace_size.argtypes = [i, i, i, ll, ll, ll, ll, P(_Cfg)]
    L.mk_get_device_status.restype = i
    L.mk_get_device_status.argtypes = [vp, vp, P(ll)]
    L.mk_ag_gemm.restype = i
    L.mk_ag_gemm.argtypes = [P(vp), vp, vp, vp, i, i, i, ll, ll, ll, vp, sz, P(_Cfg), vp]
    for name in ("mk_gemm_rs", "mk_gemm_ar"):
        f = getattr(L, name)
        f.restype = i
        f.argtypes = [P(vp), P(vp), P(vp), i, i, ll, ll, ll, vp, sz, P(_Cfg), vp]
    L.mk_ag_gemm_noalloc.restype = i
    L.mk_ag_gemm_noalloc.argtypes = [P(vp), vp, vp, vp, i, i, i, ll, ll, ll, vp, P(_Cfg), vp]
    L.mk_moe_combine_workspace_size.restype = sz
    L.mk_moe_combine_workspace_size.argtypes = [i, i, i, ll, ll, ll, ll, P(_Cfg)]
    L.mk_moe_combine.restype = i
    L.mk_moe_combine.argtypes = [P(vp), P(vp), P(vp), P(vp), vp, i, i, i, ll, ll, ll, ll,
                                 P(vp), P(vp), vp, sz, P(_Cfg), vp]
    L.mk_mlp_workspace_size.restype = sz
    L.mk_mlp_workspace_size.argtypes = [i, ll, ll, ll, P(_Cfg)]
    L.mk_mlp_ag_rs.restype = i
    L.mk_mlp_ag_rs.argtypes = [P(vp), P(vp), P(vp), i, ll, ll, ll, vp, P(vp), P(vp), vp, sz,
                               P(_Cfg), vp]
    L.mk_ring_attention_workspace_size.restype = sz
    L.mk_ring_attention_workspace_size.argtypes = [i, i, ll, i, i, P(_Cfg)]
    L.mk_ring_attention.restype = i
    L.mk_ring_attention.argtypes = [P(vp), P(vp), P(vp), i, i, ll, i, i, ctypes.c_float, P(vp),
                                    P(vp), P(vp), vp, sz, P(_Cfg), vp]
    L.mk_moe_dispatch_gemm.restype = i
    L.mk_moe_dispatch_gemm.argtypes = [P(vp), P(vp), P(vp), i, i, i, ll, ll, ll, ll, vp, vp,
                                       P(vp), vp, P(vp), P(vp), vp, sz, P(_Cfg), vp]
    return L


def status_string(s: int) -> str:
    return lib().mk_status_string(int(s)).decode()


def _ptrs(ts) -> ctypes.Array:
    arr = (ctypes.c_void_p * len(ts))()
    for j, t in enumerate(ts):
        arr[j] = t.data_ptr() if isinstance(t, torch.Tensor) else t
    return arr


def _cfgp(cfg: Config | None):
    return ctypes.byref(cfg.c()) if cfg is not None else None


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dt(dtype) -> int:
    if dtype == torch.bfloat16:
        return MK_BF16
    if dtype == torch.float32:
        return MK_F32
    raise ValueError(f"unsupported output dtype {dtype}")


def _check(st: int, what: str):
    if st != MK_OK:
        raise MkError(st, what)


# ------------------------------------------------------------------ workspaces

class Workspace:
    """A device workspace, zero-filled once at (re)allocation as the library requires."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = None

    def get(self, nbytes: int) -> torch.Tensor:
        nbytes = max(int(nbytes), 256)
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws: dict = {}


def _ws(workspace, device) -> Workspace:
    if workspace is not None:
        return workspace
    key = torch.device(device).index if torch.device(device).index is not None else \
        torch.cuda.current_device()
    if key not in _default_ws:
        _default_ws[key] = Workspace(torch.device("cuda", key))
    return _default_ws[key]


def workspace_size(op: int, R: int, m: int, n: int, k: int, cfg: Config | None = None) -> int:
    return int(lib().mk_workspace_size(op, R, m, n, k, _cfgp(cfg)))


def device_status(workspace: Workspace | None = None, stream=None, device=None):
    """Synchronise the stream and read-and-clear the workspace's device status.
    Returns (status, detail)."""
    ws = _ws(workspace, device or "cuda")
    detail = ctypes.c_longlong(0)
    st = lib().mk_get_device_status(ctypes.c_void_p(ws.get(256).data_ptr()),
                                    ctypes.c_void_p(_stream(stream, ws.device)), ctypes.byref(detail))
    return int(st), int(detail.value)


# ------------------------------------------------------------------ ops

def ag_gemm(a_shards, b, *, local_rank: int = 0, out_dtype=torch.bfloat16, a_gathered=None,
            c=None, cfg: Config | None = None, workspace: Workspace | None = None, stream=None):
    """AllGather + GEMM: returns (a_gathered = [A_0; ...; A_{R-1}], c = a_gathered @ b).
    With fp8 e4m3 operands b is B^T ([n x k]) and c = a_gathered @ b.T."""
    R = len(a_shards)
    m_r, k = a_shards[0].shape
    cfg = _with_operand(cfg, a_shards[0])
    n = b.shape[0] if a_shards[0].dtype == FP8 else b.shape[1]
    dev = b.device
    if a_gathered is None:
        a_gathered = torch.empty((R * m_r, k), dtype=a_shards[0].dtype, device=dev)
    if c is None:
        c = torch.empty((R * m_r, n), dtype=out_dtype, device=dev)
    ws = _ws(workspace, dev)
    nb = workspace_size(OP_AG_GEMM, R, m_r, n, k, cfg)
    if nb == 0:
        raise MkError(MK_ERR_INVALID, "mk_workspace_size(AG)")
    buf = ws.get(nb)
    st = lib().mk_ag_gemm(_ptrs(a_shards), b.data_ptr(), a_gathered.data_ptr(), c.data_ptr(),
                          _dt(c.dtype), R, local_rank, m_r, n, k, buf.data_ptr(), buf.numel(),
                          _cfgp(cfg), _stream(stream, dev))
    _check(st, "mk_ag_gemm")
    return a_gathered, c


def _rs_ar(fn, op, a, b, outs, R, m, n, k, cfg, workspace, stream, what):
    dev = a[0].device
    ws = _ws(workspace, dev)
    nb = workspace_size(op, R, m, n, k, cfg)
    if nb == 0:
        raise MkError(MK_ERR_INVALID, f"mk_workspace_size({what})")
    buf = ws.get(nb)
    st = fn(_ptrs(a), _ptrs(b), _ptrs(outs), _dt(outs[0].dtype), R, m, n, k, buf.data_ptr(),
            buf.numel(), _cfgp(cfg), _stream(stream, dev))
    _check(st, what)
    return outs


def gemm_rs(a, b, *, out_dtype=torch.bfloat16, c_blocks=None, cfg: Config | None = None,
            workspace: Workspace | None = None, stream=None):
    """GEMM + ReduceScatter: S = sum_r a[r] @ b[r]; returns R row blocks of S.
    With fp8 e4m3 operands b[r] is B_r^T ([n x k]) and S = sum_r a[r] @ b[r].T."""
    R = len(a)
    m, k = a[0].shape
    cfg = _with_operand(cfg, a[0])
    n = b[0].shape[0] if a[0].dtype == FP8 else b[0].shape[1]
    if c_blocks is None:
        c_blocks = [torch.empty((m // R, n), dtype=out_dtype, device=a[0].device) for _ in range(R)]
    return _rs_ar(lib().mk_gemm_rs, OP_GEMM_RS, a, b, c_blocks, R, m, n, k, cfg, workspace, stream,
                  "mk_gemm_rs")


def gemm_ar(a, b, *, out_dtype=torch.bfloat16, c_replicas=None, cfg: Config | None = None,
            workspace: Workspace | None = None, stream=None):
    """GEMM + AllReduce: S = sum_r a[r] @ b[r]; returns R identical replicas of S.
    With fp8 e4m3 operands b[r] is B_r^T ([n x k]) and S = sum_r a[r] @ b[r].T."""
    R = len(a)
    m, k = a[0].shape
    cfg = _with_operand(cfg, a[0])
    n = b[0].shape[0] if a[0].dtype == FP8 else b[0].shape[1]
    if c_replicas is None:
        c_replicas = [torch.empty((m, n), dtype=out_dtype, device=a[0].device) for _ in range(R)]
    return _rs_ar(lib().mk_gemm_ar, OP_GEMM_AR, a, b, c_replicas, R, m, n, k, cfg, workspace,
                  stream, "mk_gemm_ar")


def trace_records(workspace: Workspace, op: int, R, m, n, k, cfg: Config):
    """The in-kernel trace of the last AG / RS / AR call made on `workspace` with
    cfg.trace = 1 and these arguments (m = rows per shard for AG, as for
    workspace_size): an int64 tensor [records x 8], record 2*i + c for work item i
    on the CTA of pair rank c.  Columns (TRACE_* below): ns stamps when the
    producer takes the item, its inputs are ready, its last load is issued, the
    accumulator is ready, the epilogue is done; the SM's clock64 at the first and
    fourth stamps; epoch << 32 | CTA << 1 | pair rank.  Records the call did not
    write keep older contents (another epoch) or zeros."""
    off = ctypes.c_size_t(0)
    n_rec = int(lib().mk_trace_entries(op, R, m, n, k, _cfgp(cfg), ctypes.byref(off)))
    if n_rec == 0:
        return torch.zeros((0, TRACE_WORDS), dtype=torch.int64)
    nb = n_rec * TRACE_WORDS * 8
    buf = workspace.get(int(off.value) + nb)
    raw = buf[int(off.value):int(off.value) + nb]
    return raw.view(torch.int64).view(n_rec, TRACE_WORDS).cpu()


def trace_copy_records(workspace: Workspace, op: int, R, m, n, k, cfg: Config):
    """The copy-warp records that follow the item records: int64 [TRACE_COPY_RECORDS x 8],
    record w for copy worker w: start ns, end ns, pieces, bytes, 0, 0, 0,
    epoch << 32 | w.  Only an AllGather copy-in by copy warps writes them."""
    off = ctypes.c_size_t(0)
    n_rec = int(lib().mk_trace_entries(op, R, m, n, k, _cfgp(cfg), ctypes.byref(off)))
    if n_rec == 0:
        return torch.zeros((0, TRACE_WORDS), dtype=torch.int64)
    o = int(off.value) + n_rec * TRACE_WORDS * 8
    nb = TRACE_COPY_RECORDS * TRACE_WORDS * 8
    buf = workspace.get(o + nb)
    return buf[o:o + nb].view(torch.int64).view(TRACE_COPY_RECORDS, TRACE_WORDS).cpu()


def moe_trace_records(workspace: Workspace, R, E_loc, topk, T, H, N, cap_rows, cfg: Config):
    """The in-kernel trace of the last MoE dispatch + grouped GEMM call made on
    `workspace` with cfg.trace = 1 and these arguments (cap_rows as the call used it):
    (item records [2 x tile-table entries x 8], the reserved copy-warp records), int64,
    with the words of trace_records.  The dispatch copy writes no copy-warp records."""
    off = ctypes.c_size_t(0)
    n_rec = int(lib().mk_moe_trace_entries(R, E_loc, topk, T, H, N, cap_rows, _cfgp(cfg),
                                           ctypes.byref(off)))
    if n_rec == 0:
        z = torch.zeros((0, TRACE_WORDS), dtype=torch.int64)
        return z, z
    o = int(off.value)
    nb = (n_rec + TRACE_COPY_RECORDS) * TRACE_WORDS * 8
    raw = workspace.get(o + nb)[o:o + nb].view(torch.int64).view(-1, TRACE_WORDS).cpu()
    return raw[:n_rec], raw[n_rec:]


def mlp_trace_records(workspace: Workspace, R, m, h, f_r, cfg: Config):
    """The in-kernel trace of the last chained MLP call made on `workspace` with
    cfg.trace = 1 and these arguments: (item records, copy-warp records), int64 with
    the words of trace_records; item i < R * row tiles * f_r column tiles is an
    up-projection tile, the rest are down-projection items."""
    off = ctypes.c_size_t(0)
    n_rec = int(lib().mk_mlp_trace_entries(R, m, h, f_r, _cfgp(cfg), ctypes.byref(off)))
    if n_rec == 0:
        z = torch.zeros((0, TRACE_WORDS), dtype=torch.int64)
        return z, z
    o = int(off.value)
    nb = (n_rec + TRACE_COPY_RECORDS) * TRACE_WORDS * 8
    raw = workspace.get(o + nb)[o:o + nb].view(torch.int64).view(-1, TRACE_WORDS).cpu()
    return raw[:n_rec], raw[n_rec:]


def moe_workspace_size(R, E_loc, topk, T, H, N, cap_rows, cfg: Config | None = None) -> int:
    return int(lib().mk_moe_workspace_size(R, E_loc, topk, T, H, N, cap_rows, _cfgp(cfg)))


def moe_dispatch_gemm(x, logits, w, *, E_loc: int, topk: int = 2, cap_rows: int | None = None,
                      out=None, cfg: Config | None = None, workspace: Workspace | None = None,
                      stream=None):
    """MoE dispatch + grouped GEMM over R virtual ranks.

    x[r]: [T x H] bf16 tokens; logits[r]: [T x E] fp32 (E = R*E_loc); w[d]: [E_loc x H x N] bf16.
    Returns a dict with topk_idx [R*T x topk], counts [R x E], recv_src[d] [cap],
    recv_counts [R] (int32) and recv_x[d] [cap x H], y[d] [cap x N] (bf16); rows of rank d
    past recv_counts[d] are left as they were.  `out` may pass preallocated buffers.
    """
    R = len(x)
    T, H = x[0].shape
    N = w[0].shape[2]
    E = R * E_loc
    cap = cap_rows if cap_rows is not None else R * T * topk
    dev = x[0].device
    o = dict(out or {})
    i32 = torch.int32
    o.setdefault("topk_idx", torch.empty((R * T, topk), dtype=i32, device=dev))
    o.setdefault("counts", torch.empty((R, E), dtype=i32, device=dev))
    o.setdefault("recv_counts", torch.empty((R,), dtype=i32, device=dev))
    o.setdefault("recv_src", [torch.empty((cap,), dtype=i32, device=dev) for _ in range(R)])
    o.setdefault("recv_x", [torch.empty((cap, H), dtype=torch.bfloat16, device=dev) for _ in range(R)])
    o.setdefault("y", [torch.empty((cap, N), dtype=torch.bfloat16, device=dev) for _ in range(R)])
    ws = _ws(workspace, dev)
    nb = moe_workspace_size(R, E_loc, topk, T, H, N, cap, cfg)
    if nb == 0:
        raise MkError(MK_ERR_INVALID, "mk_moe_workspace_size")
    buf = ws.get(nb)
    st = lib().mk_moe_dispatch_gemm(_ptrs(x), _ptrs(logits), _ptrs(w), R, E_loc, topk, T, H, N, cap,
                                    o["topk_idx"].data_ptr(), o["counts"].data_ptr(),
                                    _ptrs(o["recv_src"]), o["recv_counts"].data_ptr(),
                                    _ptrs(o["recv_x"]), _ptrs(o["y"]), buf.data_ptr(), buf.numel(),
                                    _cfgp(cfg), _stream(stream, dev))
    _check(st, "mk_moe_dispatch_gemm")
    return o


def moe_combine_workspace_size(R, E_loc, topk, T, N, H, cap_rows, cfg: Config | None = None) -> int:
    return int(lib().mk_moe_combine_workspace_size(R, E_loc, topk, T, N, H, cap_rows, _cfgp(cfg)))


def moe_combine(h, w2, gates, recv_src, counts, *, E_loc: int, topk: int = 2,
                cap_rows: int | None = None, out=None, cfg: Config | None = None,
                workspace: Workspace | None = None, stream=None):
    """MoE combine over R virtual ranks: down-projection of every expert's rows,
    return of the rows to their source ranks, gate-weighted sum over the top-k.

    h[d]: [cap x N] bf16 expert hidden rows in dispatch order; w2[d]: [E_loc x N x H] bf16;
    gates[r]: [T x topk] fp32; recv_src[d]: [cap] int32 and counts: [R x E] int32 from the
    dispatch.  Returns a dict with ret[r] [T x topk x H] (the returned expert rows) and
    out[r] [T x H] (bf16).  `out` may pass preallocated buffers.
    """
    R = len(h)
    cap = cap_rows if cap_rows is not None else h[0].shape[0]
    N = h[0].shape[1]
    H = w2[0].shape[2]
    T = gates[0].shape[0]
    dev = h[0].device
    o = dict(out or {})
    o.setdefault("ret", [torch.empty((T, topk, H), dtype=torch.bfloat16, device=dev) for _ in range(R)])
    o.setdefault("out", [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(R)])
    ws = _ws(workspace, dev)
    nb = moe_combine_workspace_size(R, E_loc, topk, T, N, H, cap, cfg)
    if nb == 0:
        raise MkError(MK_ERR_INVALID, "mk_moe_combine_workspace_size")
    buf = ws.get(nb)
    st = lib().mk_moe_combine(_ptrs(h), _ptrs(w2), _ptrs(gates), _ptrs(recv_src), counts.data_ptr(),
                              R, E_loc, topk, T, N, H, cap, _ptrs(o["ret"]), _ptrs(o["out"]),
                              buf.data_ptr(), buf.numel(), _cfgp(cfg), _stream(stream, dev))
    _check(st, "mk_moe_combine")
    return o


def mlp_workspace_size(R, m, h, f_r, cfg: Config | None = None) -> int:
    return int(lib().mk_mlp_workspace_size(R, m, h, f_r, _cfgp(cfg)))


def mlp_ag_rs(x_shards, w1, w2, *, x_gathered=None, hid=None, y_blocks=None,
              cfg: Config | None = None, workspace: Workspace | None = None, stream=None):
    """Chained tensor-parallel MLP over R virtual ranks: AllGather + GEMM (w1[r]) ->
    ReLU -> GEMM (w2[r]) + ReduceScatter.  x_shards[r]: [m x h]; w1[r]: [h x f_r];
    w2[r]: [f_r x h] (bf16).  Returns (x_gathered [R*m x h], hid [R x [R*m x f_r]],
    y_blocks [R x [m x h]])."""
    R = len(x_shards)
    m, h = x_shards[0].shape
    f_r = w1[0].shape[1]
    dev = x_shards[0].device
    bf = torch.bfloat16
    if x_gathered is None:
        x_gathered = torch.empty((R * m, h), dtype=bf, device=dev)
    if hid is None:
        hid = [torch.empty((R * m, f_r), dtype=bf, device=dev) for _ in range(R)]
    if y_blocks is None:
        y_blocks = [torch.empty((m, h), dtype=bf, device=dev) for _ in range(R)]
    ws = _ws(workspace, dev)
    nb = mlp_workspace_size(R, m, h, f_r, cfg)
    if nb == 0:
        raise MkError(MK_ERR_INVALID, "mk_mlp_workspace_size")
    buf = ws.get(nb)
    st = lib().mk_mlp_ag_rs(_ptrs(x_shards), _ptrs(w1), _ptrs(w2), R, m, h, f_r, x_gathered.data_ptr(),
                            _ptrs(hid), _ptrs(y_blocks), buf.data_ptr(), buf.numel(), _cfgp(cfg),
                            _stream(stream, dev))
    _check(st, "mk_mlp_ag_rs")
    return x_gathered, hid, y_blocks


def ring_attention(q, k, v, *, causal: bool = False, scale: float | None = None, out=None,
                   k_recv=None, v_recv=None, cfg: Config | None = None,
                   workspace: Workspace | None = None, stream=None):
    """Ring attention over R virtual ranks.  q[r], k[r], v[r]: [heads x s_r x d] bf16
    (d = 128), rank r holding positions [r*s_r, (r+1)*s_r).  Returns out[r] (same shape)
    = softmax(scale * Q_r K^T (+ causal mask)) V over the whole sequence."""
    R = len(q)
    heads, s_r, d = q[0].shape
    dev = q[0].device
    bf = torch.bfloat16
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = [torch.empty((heads, s_r, d), dtype=bf, device=dev) for _ in range(R)]
    mode = cfg.mode if cfg is not None else MODE_FUSED
    if R > 1 and mode != MODE_GEMM_ONLY:
        if k_recv is None:
            k_recv = [torch.empty(((R - 1) * heads, s_r, d), dtype=bf, device=dev) for _ in range(R)]
        if v_recv is None:
            v_recv = [torch.empty(((R - 1) * heads, s_r, d), dtype=bf, device=dev) for _ in range(R)]
    kr = _ptrs(k_recv) if k_recv is not None else None
    vr = _ptrs(v_recv) if v_recv is not None else None
    ws = _ws(workspace, dev)
    nb = int(lib().mk_ring_attention_workspace_size(R, heads, s_r, d, int(causal), _cfgp(cfg)))
    if nb == 0:
        raise MkError(MK_ERR_INVALID, "mk_ring_attention_workspace_size")
    buf = ws.get(nb)
    st = lib().mk_ring_attention(_ptrs(q), _ptrs(k), _ptrs(v), R, heads, s_r, d, int(causal),
                                 float(scale), kr, vr, _ptrs(out), buf.data_ptr(), buf.numel(),
                                 _cfgp(cfg), _stream(stream, dev))
    _check(st, "mk_ring_attention")
    return out


__all__ = ["Config", "MkError", "Workspace", "ag_gemm", "gemm_rs", "gemm_ar", "device_status",
           "workspace_size", "lib", "status_string", "MODE_FUSED", "MODE_GEMM_ONLY",
           "MODE_UNFUSED", "moe_dispatch_gemm", "moe_workspace_size", "moe_combine",
           "moe_combine_workspace_size", "mlp_ag_rs", "mlp_workspace_size", "ring_attention"]
