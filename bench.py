"""Benchmark of the fused collective + GEMM library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mk|reference]

Default workload: AllGather+GEMM with 8 virtual ranks, A shards 1024x8192
bf16 gathered to 8192x8192, B 8192x3584 (TP=8 MLP up-projection), bf16 out.
One step = one fused call (one persistent kernel launch) over one input set;
three input sets (each larger than L2 together with its outputs) are used in
rotation, so no step reads what the previous one left in L2.

Prints one JSON line (rank 0).  Besides the fused throughput it reports the
two baselines the same library provides -- the GEMM alone on pre-gathered A
(no data movement) and the unfused copy-then-GEMM sequence -- and the exposed
time (fused - GEMM only).  GEMM+ReduceScatter (8 ranks, 8192x3584 @
3584x8192 per rank) and GEMM+AllReduce (8 ranks, 128x3584 @ 3584x8192) are
measured the same way and reported under "other_configs".

--impl reference times the CPU oracle (the only other implementation of these
ops that exists here) on host cores, on a bounded row sample per step.
With N > 1 each rank runs an independent replica of the workload on its own
GPU (no collective between GPUs); throughput is the sum over ranks of the
units processed divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from comm_gemm_tile_gb300 import inputs as I  # noqa: E402

METRIC = "fused AG+GEMM TFLOP/s on 1 GB300 (AllGather+GEMM, 8 virtual ranks, 8192x8192x3584 bf16)"
UNIT = "TFLOP/s"
N_SETS = 3


# ------------------------------------------------------------------ environment helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_seed_offset(rank: int) -> int:
    """Seed offset of a replica: every rank draws an independent problem."""
    return 100000 * rank


def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The slowest rank's time (all ranks get the same value)."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, t_max_ms: float) -> float:
    """Units processed by all ranks per second, over the slowest rank's time."""
    return world * units_per_rank / (t_max_ms * 1e-3)


# The sources of mk_fused_kernel and of the host code that plans its launches.
FUSED_KERNEL_SOURCES = ("mk_api.cu", "mk_fused.cu", "mk_internal.h", "mk_ptx.cuh")


ATTN_KERNEL_SOURCES = ("mk_attn.cu", "mk_internal.h", "mk_ptx.cuh")


def kernel_source_sha256(files=FUSED_KERNEL_SOURCES) -> str:
    """Hash of a kernel's sources, to tell whether recorded ncu counters still apply."""
    import hashlib
    root = os.path.join(ROOT, "comm_gemm_tile_gb300", "csrc")
    h = hashlib.sha256()
    for f in files:
        h.update(f.encode())
        h.update(open(os.path.join(root, f), "rb").read())
    return h.hexdigest()


def recorded_traffic(workload: str, key: str = "fused_dram_bytes", kernel: str = "mk_fused_kernel"):
    """DRAM bytes per launch from the committed ncu record of `kernel`
    (mk_fused_kernel or mk_ring_attn_kernel), or None when the kernel sources
    changed since it was taken."""
    files = FUSED_KERNEL_SOURCES if kernel == "mk_fused_kernel" else ATTN_KERNEL_SOURCES
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")))
        if rec.get("source_sha256") != kernel_source_sha256(files):
            return None
        return rec[workload][key]
    except Exception:
        return None


def peaks():
    """(bf16 burst TFLOP/s, bf16 sustained TFLOP/s, HBM GB/s, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            float(d["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 25):
        self.idx = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dev_normal(shape, std, seed, device):
    """Seeded N(0, std^2) samples drawn on the device, packed to bf16."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def time_loop(fn, steps, warmup, stream, dist=None):
    """Device time (ms) of `steps` calls of fn, after `warmup` untimed calls."""
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1)


def traced_sm_mhz(mk, sets, ws, stream, pair, w):
    """Median SM clock (MHz) over the work items of one traced fused AG call: the
    in-kernel trace's clock64 ticks over %globaltimer ns between an item's start and
    its accumulator-ready stamp (items longer than 2 us)."""
    cfg = mk.Config(cta_pair=pair, trace=1)
    tws = mk.Workspace(ws.device)
    shards, b, g, c = sets[0]
    mk.ag_gemm(shards, b, a_gathered=g, c=c, cfg=cfg, workspace=tws, stream=stream)
    torch.cuda.synchronize()
    rec = mk.trace_records(tws, mk.OP_AG_GEMM, w.R, w.m, w.n, w.k, cfg)
    ep = rec[:, mk.TRACE_ID] >> 32
    sel = (ep == ep.max()) & (rec[:, mk.TRACE_START] != 0)
    dt = (rec[sel, mk.TRACE_READY] - rec[sel, mk.TRACE_START]).double()
    dc = (rec[sel, mk.TRACE_CLK_READY] - rec[sel, mk.TRACE_CLK_START]).double()
    ok = dt > 2000
    if not bool(ok.any()):
        return None
    return float((dc[ok] / dt[ok]).median()) * 1e3


def time_interleaved(fns: dict, steps: int, warmup: int, stream, dist=None, rounds: int = 5):
    """Device time (ms per call) of each named mode, the modes timed in turn in `rounds`
    blocks of about steps / rounds calls each, so that every mode sees the same clock
    and power state (a mode timed in one long loop after another runs hotter or cooler).
    Each block starts after one untimed call of its own mode, so that it does not pay for
    the caches the previous mode left dirty.  Call index i runs on over the blocks of a
    mode, rotating its input sets."""
    block = max(1, steps // rounds)
    for fn in fns.values():
        for i in range(warmup):
            fn(i)
    total = {name: 0.0 for name in fns}
    done = {name: 0 for name in fns}
    for _ in range(rounds):
        for name, fn in fns.items():
            i0 = done[name]
            total[name] += time_loop(lambda i, fn=fn, i0=i0: fn(i0 + i), block, 1, stream, dist)
            done[name] += block
    return {name: total[name] / done[name] for name in fns}


# ------------------------------------------------------------------ CPU oracle timing

def oracle_sample_rate(shards_bits, b_bits, target_s: float):
    """Time the oracle's AG+GEMM on a row sample sized to ~target_s seconds.
    Returns (TFLOP/s, rows, seconds)."""
    import oracle as O
    K = b_bits.shape[0]
    N = b_bits.shape[1]
    M = sum(s.shape[0] for s in shards_bits)
    rows = 16
    while True:
        sel = np.linspace(0, M - 1, rows).astype(np.int64)
        t0 = time.perf_counter()
        O.ag_gemm(shards_bits, b_bits, rows=sel)
        t = time.perf_counter() - t0
        if t >= target_s * 0.5 or rows >= M:
            break
        rows = int(min(M, max(rows * 2, rows * target_s / max(t, 1e-3) * 0.9)))
    return 2.0 * rows * N * K / t / 1e12, rows, t


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return int(max(d.get("num_threads", 1) for d in info))
    except Exception:
        pass
    return os.cpu_count() or 1


def _timed_rows(run, n_total: int, target_s: float):
    """Run the oracle on a growing evenly spaced row sample until one run takes
    about target_s seconds (or covers every row).  Returns (rows, seconds)."""
    rows = min(8, n_total)
    while True:
        sel = np.linspace(0, n_total - 1, rows).astype(np.int64)
        t0 = time.perf_counter()
        run(sel)
        t = time.perf_counter() - t0
        if t >= target_s * 0.5 or rows >= n_total:
            return rows, t
        rows = int(min(n_total, max(rows * 2, rows * target_s / max(t, 1e-3) * 0.9)))


def cpu_gemm_baseline(a_dev, b_dev, w, target_s: float = 4.0):
    """The oracle's S = sum_r A_r @ B_r (GEMM+ReduceScatter / GEMM+AllReduce) on a
    row sample of the workload, on the host cores: TFLOP/s of the sampled rows."""
    import oracle as O
    a_bits = [I.bits(x) for x in a_dev]
    b_bits = [I.bits(x) for x in b_dev]
    rows, t = _timed_rows(lambda sel: O.sum_over_ranks(a_bits, b_bits, rows=sel), w.m, target_s)
    rate = 2.0 * rows * w.n * w.k * w.R / t / 1e12
    return {"value": rate, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"{rows} of {w.m} rows of S (all {w.n} columns, {w.R} ranks x K={w.k}), "
                      f"fp64 numpy, {t:.1f} s"}


def cpu_moe_baseline(x_dev, lg_dev, we_dev, w, target_s: float = 4.0):
    """The oracle's MoE path on the host cores: routing, counts and the dispatch
    permutation for every token, then the gather and grouped GEMM of an evenly
    spaced sample of each destination rank's received rows.  TFLOP/s of the
    sampled rows' GEMM over the whole time."""
    import oracle as O
    x_bits = [I.bits(t) for t in x_dev]
    w_bits = [I.bits(t) for t in we_dev]
    logits = [t.cpu().numpy() for t in lg_dev]
    t0 = time.perf_counter()
    idx = [O.moe_route(lg, w.topk) for lg in logits]
    O.moe_counts(idx, w.E)
    recv_src, seg = O.moe_dispatch(idx, w.E_loc)
    t_route = time.perf_counter() - t0
    total = sum(len(s) for s in recv_src)

    def run(sel_frac):
        n = 0
        for d in range(w.R):
            nd = len(recv_src[d])
            if nd == 0:
                continue
            sel = np.unique((sel_frac * (nd - 1)).astype(np.int64))
            rx = O.moe_gather_rows(x_bits, recv_src[d][sel], w.topk)
            # the gathered rows are the sample: expert of each from the segment bounds
            starts = np.concatenate([[0], np.cumsum(seg[d])])
            ex = np.searchsorted(starts, sel, side="right") - 1
            for l in np.unique(ex):
                pick = np.nonzero(ex == l)[0]
                O.moe_expert_gemm(rx[pick], [len(pick)], w_bits[d][l:l + 1])
            n += len(sel)
        run.rows = n

    per = 8
    while True:
        frac = np.linspace(0.0, 1.0, per)
        t1 = time.perf_counter()
        run(frac)
        t = time.perf_counter() - t1
        if t >= target_s * 0.5 or per >= total:
            break
        per = int(min(total, max(per * 2, per * target_s / max(t, 1e-3) * 0.9)))
    rate = 2.0 * run.rows * w.H * w.N / (t + t_route) / 1e12
    return {"value": rate, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"routing + dispatch of all {total} rows ({t_route:.1f} s), then gather + "
                      f"expert GEMM of {run.rows} received rows ({t:.1f} s), fp64 numpy"}


# ------------------------------------------------------------------ the reference (oracle) arm

def run_reference(args):
    _, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle as O
    w = I.AG_R8_TP8_UP
    shards = [I.bits(I.normal_bf16((w.m, w.k), 1.0, w.a_seed + r)) for r in range(w.R)]
    bmat = I.bits(I.normal_bf16((w.k, w.n), w.b_std, w.b_seed))
    per_step = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    _, rows, _ = oracle_sample_rate(shards, bmat, per_step)
    M = w.R * w.m
    sel = np.linspace(0, M - 1, rows).astype(np.int64)
    for _ in range(args.warmup):
        O.ag_gemm(shards, bmat, rows=sel)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.ag_gemm(shards, bmat, rows=sel)
    dt = time.perf_counter() - t0
    val = 2.0 * rows * w.n * w.k * args.steps / dt / 1e12
    cores = blas_threads()
    sample = f"{rows} of {M} output rows per step (all {w.n} columns, K={w.k}), fp64 numpy"
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "R": w.R, "m_r": w.m, "k": w.k,
                                        "n": w.n, "sample": sample},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ the library arm

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--other-steps", type=int, default=30)
    ap.add_argument("--no-other", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--n-copy", type=int, default=0)
    ap.add_argument("--cta-pair", type=int, default=0, choices=[0, 1, 2],
                    help="GEMM tiles: 0 library default, 1 one CTA per tile, 2 CTA pairs")
    ap.add_argument("--only", choices=["rs", "ar", "moe", "combine", "mlp", "ring", "ring_small", "ag_fp8"],
                    default=None,
                    help="time only this secondary workload (profiling aid) and print its entry")
    ap.add_argument("--profile", choices=list(PROFILE_WORKLOADS), default=None,
                    help="profiling aid: make the workload's inputs and run --calls untimed fused calls "
                         "back to back (for an ncu capture of one of them); prints the device status")
    ap.add_argument("--energy", choices=list(PROFILE_WORKLOADS), default=None,
                    help="energy per call (NVML counter) of the workload's fused, GEMM-only and unfused "
                         "modes")
    ap.add_argument("--energy-secs", type=float, default=3.0)
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--scale", choices=["full", "small"], default="full",
                    help="--profile: the bench workload, or a reduced case (inputs still larger than L2)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.profile:
        return run_profile(args)
    if args.energy:
        return run_energy(args)
    if args.only:
        return run_only(args)

    world, rank, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist  # noqa: F811
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    stream = torch.cuda.current_stream(device)

    import comm_gemm_tile_gb300 as mk
    from comm_gemm_tile_gb300 import build as mkbuild
    mkbuild.build()
    mk.lib()
    bf16_peak, _, hbm_peak, peak_src = peaks()

    w = I.AG_R8_TP8_UP
    seed_off = replica_seed_offset(rank)   # replicas: an independent problem per rank
    M = w.R * w.m
    flops = 2.0 * M * w.n * w.k
    sets = []
    for s in range(N_SETS):
        shards = [dev_normal((w.m, w.k), 1.0, w.a_seed + r + 1000 * s + seed_off, device)
                  for r in range(w.R)]
        b = dev_normal((w.k, w.n), w.b_std, w.b_seed + 1000 * s + seed_off, device)
        g = torch.empty((M, w.k), dtype=torch.bfloat16, device=device)
        c = torch.empty((M, w.n), dtype=torch.bfloat16, device=device)
        sets.append((shards, b, g, c))
    wsp = mk.Workspace(device)
    cfg_f = mk.Config(n_copy_ctas=args.n_copy, cta_pair=args.cta_pair)

    def step_fused(i):
        shards, b, g, c = sets[i % N_SETS]
        mk.ag_gemm(shards, b, a_gathered=g, c=c, cfg=cfg_f, workspace=wsp, stream=stream)

    # guard for the timed configuration: device status and the gathered bits
    step_fused(0)
    st, detail = mk.device_status(wsp, stream)
    if st != mk.MK_OK:
        raise SystemExit(f"fused AG+GEMM reported {mk.status_string(st)} ({detail})")
    if not torch.equal(sets[0][2], torch.cat(sets[0][0], 0)):
        raise SystemExit("gathered A differs from the shards")

    with ClockSampler(local) as clk:
        t_fused = time_loop(step_fused, args.steps, args.warmup, stream, dist)
    st, detail = mk.device_status(wsp, stream)
    if st != mk.MK_OK:
        raise SystemExit(f"fused AG+GEMM reported {mk.status_string(st)} ({detail})")
    # the SM clock inside the kernel (the sampler's 200 ms readings show the clock
    # target): one traced call right after the timed loop, SM cycles over ns per item
    traced_mhz = traced_sm_mhz(mk, sets, wsp, stream, args.cta_pair, w)

    cfg_g = mk.Config(mode=mk.MODE_GEMM_ONLY, cta_pair=args.cta_pair)
    cfg_u = mk.Config(mode=mk.MODE_UNFUSED, cta_pair=args.cta_pair)

    def step_gemm(i):
        shards, b, g, c = sets[i % N_SETS]
        mk.ag_gemm(shards, b, a_gathered=g, c=c, cfg=cfg_g, workspace=wsp, stream=stream)

    def step_unfused(i):
        shards, b, g, c = sets[i % N_SETS]
        mk.ag_gemm(shards, b, a_gathered=g, c=c, cfg=cfg_u, workspace=wsp, stream=stream)

    base_steps = max(10, min(args.steps, 200))

    def tmax(x):
        return max_over_ranks(x, dist, device)

    # fused against GEMM-only and unfused: interleaved blocks under the same clocks
    cmp_ms = time_interleaved({"fused": step_fused, "gemm_only": step_gemm,
                               "unfused": step_unfused}, base_steps, 5, stream, dist)
    t_cmp = tmax(cmp_ms["fused"])
    t_gemm = tmax(cmp_ms["gemm_only"])
    t_unf = tmax(cmp_ms["unfused"])
    t_fused_max = tmax(t_fused)
    ms = t_fused_max / args.steps
    value = whole_job_rate(flops * args.steps, world, t_fused_max) / 1e12
    achieved = flops / (t_fused / args.steps * 1e-3) / 1e12

    # ---- end to end: pinned host inputs -> device -> fused call -> host result, every
    # step.  The steps are pipelined over the N_SETS device slots the way a serving loop
    # runs: step i's host->device copies go on a copy stream (after the call that last
    # read that slot), the call on the compute stream after them, and the read-back of
    # its result on a third stream, so copies of one step overlap the call of another.
    hshards = [x.cpu().pin_memory() for x in sets[0][0]]
    hb = sets[0][1].cpu().pin_memory()
    hcs = [torch.empty((M, w.n), dtype=torch.bfloat16).pin_memory() for _ in range(N_SETS)]
    h2d = sum(x.numel() * 2 for x in hshards) + hb.numel() * 2
    d2h = hcs[0].numel() * 2
    # (one host->device stream: spreading the copies over 2, 4 or 9 streams measured the same,
    # ~188 GB/s, which bounds this loop)
    s_in = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)
    ev_in = [torch.cuda.Event() for _ in range(N_SETS)]
    ev_k = [torch.cuda.Event() for _ in range(N_SETS)]
    ev_out = [torch.cuda.Event() for _ in range(N_SETS)]

    def step_e2e(i):
        j = i % N_SETS
        shards, b, g, c = sets[j]
        s_in.wait_event(ev_k[j])                  # the call that last read this slot is done
        with torch.cuda.stream(s_in):
            for d, h in zip(shards, hshards):
                d.copy_(h, non_blocking=True)
            b.copy_(hb, non_blocking=True)
        ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_out[j])              # this slot's previous result has been read back
        mk.ag_gemm(shards, b, a_gathered=g, c=c, cfg=cfg_f, workspace=wsp, stream=stream)
        ev_k[j].record(stream)
        s_out.wait_event(ev_k[j])
        with torch.cuda.stream(s_out):
            hcs[j].copy_(c, non_blocking=True)
        ev_out[j].record(s_out)

    def e2e_loop(steps, warmup):
        for i in range(warmup):
            step_e2e(i)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        s_in.wait_event(e0)
        s_out.wait_event(e0)
        for i in range(steps):
            step_e2e(i)
        for j in range(N_SETS):                   # every copy of the timed steps before e1
            stream.wait_event(ev_out[j])
        e1.record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        return e0.elapsed_time(e1)

    t_e2e = tmax(e2e_loop(args.e2e_steps, 3))
    # guard (untimed): the read-back result is the device result of the same inputs
    if not torch.equal(hcs[0], sets[0][3].cpu()):
        raise SystemExit("e2e read-back differs from the device result")
    e2e_val = whole_job_rate(flops * args.e2e_steps, world, t_e2e) / 1e12
    st, detail = mk.device_status(wsp, stream)
    if st != mk.MK_OK:
        raise SystemExit(f"e2e AG+GEMM reported {mk.status_string(st)} ({detail})")

    other = {}
    if not args.no_other:
        other = bench_other(mk, device, stream, dist, args.other_steps, seed_off, tmax,
                            bf16_peak, hbm_peak, pair=args.cta_pair,
                            cpu=(rank == 0 and not args.no_cpu))

    cpu = None
    if rank == 0 and not args.no_cpu:
        rate, rows, secs = oracle_sample_rate([I.bits(x) for x in hshards], I.bits(hb), 10.0)
        cpu = {"value": rate, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": f"{rows} of {M} output rows (all {w.n} columns, K={w.k}), fp64 numpy, "
                         f"{secs:.1f} s"}

    clocks = clk.summary()
    clocks["traced_sm_mhz"] = traced_mhz
    set_mb = ((w.R * w.m * w.k + w.k * w.n) * 2 + (M * w.k + M * w.n) * 2) / 1e6
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "R": w.R, "m_r": w.m, "k": w.k, "n": w.n,
                       "local_rank": 0, "out": "bf16", "parallelism": f"replicas{world}",
                       "l2": f"{N_SETS} input sets in rotation, each {set_mb:.0f} MB with "
                             f"outputs (> L2)"},
            "pct_of_peak": 100.0 * (flops / (ms * 1e-3) / 1e12) / bf16_peak,
            # exposed: fused minus GEMM-only, both from the interleaved comparison
            "exposed_ms": t_cmp - t_gemm,
            "fused_ms_interleaved": t_cmp,
            "gemm_only_ms": t_gemm,
            "unfused_ms": t_unf,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16_peak,
                         "unit": "TFLOP/s", "frac": achieved / bf16_peak,
                         "traffic": recorded_traffic(w.name),
                         "peak_source": f"{peak_src} bf16 burst"},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "other_configs": other,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


PROFILE_WORKLOADS = ("ag", "rs", "ar", "moe", "combine", "mlp", "ring")


def profile_call(mk, name, small, device, ws):
    """One workload's inputs and a call(cfg=None) that runs it once (fused by
    default; a Config picks GEMM-only or unfused).  small: the reduced case,
    inputs still larger than L2."""
    if name in ("ag", "rs", "ar"):
        w = {"ag": I.AG_R8_TP8_UP, "rs": I.RS_R8_TP8_DOWN, "ar": I.AR_R8_DECODE}[name]
        if small and name != "ar":
            w = I.GemmWorkload(w.name + "_small", w.op, R=w.R, m=w.m // 4, n=w.n, k=w.k, out=w.out,
                               a_seed=w.a_seed, b_seed=w.b_seed, b_std=w.b_std)
        if name == "ag":
            a = [dev_normal((w.m, w.k), 1.0, w.a_seed + r, device) for r in range(w.R)]
            b = dev_normal((w.k, w.n), w.b_std, w.b_seed, device)
            g = torch.empty((w.R * w.m, w.k), dtype=torch.bfloat16, device=device)
            c = torch.empty((w.R * w.m, w.n), dtype=torch.bfloat16, device=device)
            return lambda cfg=None: mk.ag_gemm(a, b, a_gathered=g, c=c, cfg=cfg, workspace=ws)
        a = [dev_normal((w.m, w.k), 1.0, w.a_seed + r, device) for r in range(w.R)]
        b = [dev_normal((w.k, w.n), w.b_std, w.b_seed + r, device) for r in range(w.R)]
        rows = w.m // w.R if name == "rs" else w.m
        o = [torch.empty((rows, w.n), dtype=torch.bfloat16, device=device) for _ in range(w.R)]
        fn = mk.gemm_rs if name == "rs" else mk.gemm_ar
        key = "c_blocks" if name == "rs" else "c_replicas"
        return lambda cfg=None: fn(a, b, cfg=cfg, workspace=ws, **{key: o})
    if name in ("moe", "combine"):
        wd = I.MOE_R8_E64
        T = wd.T // 4 if small else wd.T
        x = [dev_normal((T, wd.H), 1.0, wd.x_seed + r, device) for r in range(wd.R)]
        lg = [I.zipf_logits(T, wd.E, wd.logit_seed + r).to(device) for r in range(wd.R)]
        we = [dev_normal((wd.E_loc, wd.H, wd.N), 0.02, wd.w_seed + d, device) for d in range(wd.R)]
        cap = 2 * T * wd.R
        disp = mk.moe_dispatch_gemm(x, lg, we, E_loc=wd.E_loc, topk=wd.topk, cap_rows=cap, workspace=ws)
        if name == "moe":
            return lambda cfg=None: mk.moe_dispatch_gemm(x, lg, we, E_loc=wd.E_loc, topk=wd.topk,
                                                         cap_rows=cap, out=disp, cfg=cfg, workspace=ws)
        w = I.MOE_COMBINE_R8_E64
        h = [dev_normal((cap, w.N), 1.0, w.h_seed + d, device) for d in range(w.R)]
        w2 = [dev_normal((w.E_loc, w.N, w.H), 0.02, w.w2_seed + d, device) for d in range(w.R)]
        gates = [torch.full((T, w.topk), 0.5, device=device) for _ in range(w.R)]
        del x, we
        outs = mk.moe_combine(h, w2, gates, disp["recv_src"], disp["counts"], E_loc=w.E_loc,
                              topk=w.topk, cap_rows=cap, workspace=ws)
        return lambda cfg=None: mk.moe_combine(h, w2, gates, disp["recv_src"], disp["counts"],
                                               E_loc=w.E_loc, topk=w.topk, cap_rows=cap, out=outs,
                                               cfg=cfg, workspace=ws)
    if name == "mlp":
        w = I.MLP_R8_TP8
        m = w.m // 4 if small else w.m
        x = [dev_normal((m, w.h), 1.0, w.x_seed + r, device) for r in range(w.R)]
        w1 = [dev_normal((w.h, w.f_r), w.w_std, w.w1_seed + r, device) for r in range(w.R)]
        w2 = [dev_normal((w.f_r, w.h), w.w_std, w.w2_seed + r, device) for r in range(w.R)]
        xg, hid, y = mk.mlp_ag_rs(x, w1, w2, workspace=ws)
        return lambda cfg=None: mk.mlp_ag_rs(x, w1, w2, x_gathered=xg, hid=hid, y_blocks=y, cfg=cfg,
                                             workspace=ws)
    w = I.RING_R8_H8_S4096
    s_r = w.s_r // 4 if small else w.s_r
    shape = (w.heads, s_r, w.d)
    q, k, v = ([dev_normal(shape, 1.0, seed + r, device) for r in range(w.R)]
               for seed in (w.q_seed, w.k_seed, w.v_seed))
    out = [torch.empty(shape, dtype=torch.bfloat16, device=device) for _ in range(w.R)]
    return lambda cfg=None: mk.ring_attention(q, k, v, out=out, cfg=cfg, workspace=ws)


class Nvml:
    """Read-only NVML queries through NVIDIA's management library,
    libnvidia-ml (no Python bindings needed): the total-energy counter (mJ),
    the SM clock and the enforced power limit of the GPU that CUDA device
    `idx` is."""

    def __init__(self, idx: int = 0):
        import ctypes
        self.ct = ctypes
        self.nv = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        cnt = ctypes.c_uint()
        self.nv.nvmlDeviceGetCount_v2(ctypes.byref(cnt))
        self.h = ctypes.c_void_p()
        pick = 0
        if cnt.value > 1:
            want = str(getattr(torch.cuda.get_device_properties(idx), "uuid", ""))
            buf = ctypes.create_string_buffer(96)
            pick = -1
            for i in range(cnt.value):
                self.nv.nvmlDeviceGetHandleByIndex_v2(i, ctypes.byref(self.h))
                self.nv.nvmlDeviceGetUUID(self.h, buf, 96)
                if want and want in buf.value.decode():
                    pick = i
                    break
            if pick < 0:
                raise RuntimeError("cannot match the CUDA device to an NVML device")
        if self.nv.nvmlDeviceGetHandleByIndex_v2(pick, ctypes.byref(self.h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByIndex failed")

    def _u(self, fn, *args, ull=False):
        v = self.ct.c_ulonglong() if ull else self.ct.c_uint()
        if fn(self.h, *args, self.ct.byref(v)) != 0:
            raise RuntimeError(f"{fn.__name__} failed")
        return v.value

    def energy_mj(self) -> int:
        return self._u(self.nv.nvmlDeviceGetTotalEnergyConsumption, ull=True)

    def sm_mhz(self) -> int:
        return self._u(self.nv.nvmlDeviceGetClockInfo, 1)   # NVML_CLOCK_SM

    def power_limit_w(self) -> float:
        return self._u(self.nv.nvmlDeviceGetEnforcedPowerLimit) / 1000.0


def run_energy(args):
    """Energy per call of one workload in its fused, GEMM-only and unfused
    modes: NVML's total-energy counter read around ~3 s of back-to-back calls
    per mode, modes interleaved over three rounds, medians reported.  Under
    the power limit the fused call's extra time over GEMM-only follows its
    extra energy: exposed time ~ extra energy / power."""
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    import comm_gemm_tile_gb300 as mk
    from comm_gemm_tile_gb300 import build as mkbuild
    mkbuild.build()
    nv = Nvml(0)
    ws = mk.Workspace(device)
    call = profile_call(mk, args.energy, args.scale == "small", device, ws)
    modes = {"fused": None, "gemm_only": mk.Config(mode=mk.MODE_GEMM_ONLY),
             "unfused": mk.Config(mode=mk.MODE_UNFUSED)}
    res: dict = {m: [] for m in modes}
    for _ in range(3):
        for m, cfg in modes.items():
            for _ in range(5):
                call(cfg)
            torch.cuda.synchronize()
            t = time.time()
            n = 0
            while time.time() - t < 0.3:
                call(cfg)
                n += 1
            torch.cuda.synchronize()
            n = max(10, int(args.energy_secs / ((time.time() - t) / n)))
            clk = []
            e0, t0 = nv.energy_mj(), time.time()
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record()
            last = t0
            for _ in range(n):
                call(cfg)
                if time.time() - last > 0.05:
                    clk.append(nv.sm_mhz())
                    last = time.time()
            ev1.record()
            torch.cuda.synchronize()
            e1, t1 = nv.energy_mj(), time.time()
            res[m].append({"us": ev0.elapsed_time(ev1) / n * 1e3, "mj": (e1 - e0) / n,
                           "w": (e1 - e0) / (t1 - t0) / 1e3,
                           "sm_mhz": statistics.median(clk) if clk else None})
    st, detail = mk.device_status(ws)
    med = {m: {k: statistics.median(r[k] for r in v) if v[0][k] is not None else None
               for k in ("us", "mj", "w", "sm_mhz")} for m, v in res.items()}
    de = med["fused"]["mj"] - med["gemm_only"]["mj"]
    print(json.dumps({"energy": args.energy, "scale": args.scale, "power_limit_w": nv.power_limit_w(),
                      "modes": med, "exposed_us": med["fused"]["us"] - med["gemm_only"]["us"],
                      "extra_energy_mj": de,
                      "extra_energy_us_at_fused_power": de / med["fused"]["w"] * 1e3,
                      "status": mk.status_string(st), "detail": detail}), flush=True)
    return 0 if st == mk.MK_OK else 1


def run_profile(args):
    """Untimed fused calls of one workload (profiling aid: ncu captures one of
    them).  --scale small shrinks the row / token / position counts, keeping the
    inputs larger than L2, so that multi-pass captures stay small."""
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    import comm_gemm_tile_gb300 as mk
    from comm_gemm_tile_gb300 import build as mkbuild
    mkbuild.build()
    ws = mk.Workspace(device)
    name = args.profile
    call = profile_call(mk, name, args.scale == "small", device, ws)
    for _ in range(args.calls):
        call()
    torch.cuda.synchronize()
    st, detail = mk.device_status(ws)
    print(json.dumps({"profile": name, "scale": args.scale, "calls": args.calls,
                      "status": mk.status_string(st), "detail": detail}), flush=True)
    return 0 if st == mk.MK_OK else 1


def run_only(args):
    """Time one secondary workload alone (fused / GEMM-only / unfused) and print it."""
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(device)
    import comm_gemm_tile_gb300 as mk
    from comm_gemm_tile_gb300 import build as mkbuild
    mkbuild.build()
    bf16_peak, _, hbm_peak, _ = peaks()
    if args.only == "moe":
        res = bench_moe(mk, device, stream, None, args.other_steps, 0, lambda x: x, bf16_peak, hbm_peak)
    elif args.only == "ring_small":
        # profiling aid: three calls of a mid-size ring attention (4 ranks x 2048, 4 heads), K/V in place
        shape = (4, 2048, 128)
        q, k, v = ([dev_normal(shape, 1.0, seed + r, device) for r in range(4)] for seed in (1, 11, 21))
        for _ in range(3):
            mk.ring_attention(q, k, v, cfg=mk.Config(mode=mk.MODE_GEMM_ONLY))
        torch.cuda.synchronize()
        res = {"status": mk.status_string(mk.device_status()[0])}
    elif args.only == "ring":
        res = {"full": bench_ring(mk, device, stream, None, args.other_steps, 0, lambda x: x, bf16_peak,
                                  hbm_peak),
               "causal": bench_ring(mk, device, stream, None, args.other_steps, 0, lambda x: x, bf16_peak,
                                    hbm_peak, causal=True)}
    elif args.only == "mlp":
        res = bench_mlp(mk, device, stream, None, args.other_steps, 0, lambda x: x, bf16_peak, hbm_peak)
    elif args.only == "ag_fp8":
        res = bench_ag_fp8(mk, device, stream, None, args.other_steps, 0, lambda x: x, bf16_peak, hbm_peak)
    elif args.only == "combine":
        res = bench_moe_combine(mk, device, stream, None, args.other_steps, 0, lambda x: x, bf16_peak,
                                hbm_peak)
    else:
        w = I.RS_R8_TP8_DOWN if args.only == "rs" else I.AR_R8_DECODE
        res = bench_other(mk, device, stream, None, args.other_steps, 0, lambda x: x, bf16_peak,
                          hbm_peak, only=[w], with_moe=False, pair=args.cta_pair)[w.name]
    print(json.dumps({"only": args.only, **res}), flush=True)
    return 0


def bench_other(mk, device, stream, dist, steps, seed_off, tmax, bf16_peak, hbm_peak,
                only=None, with_moe=True, pair=0, cpu=False):
    """Fused / GEMM-only / unfused timings of the RS and AR workloads (and, with
    cpu=True, the CPU oracle on a row sample of each)."""
    out = {}
    for w in (only or (I.RS_R8_TP8_DOWN, I.AR_R8_DECODE)):
        nsets = 2 if w.op == "rs" else 3
        sets = []
        for s in range(nsets):
            a = [dev_normal((w.m, w.k), 1.0, w.a_seed + r + 1000 * s + seed_off, device)
                 for r in range(w.R)]
            b = [dev_normal((w.k, w.n), w.b_std, w.b_seed + r + 1000 * s + seed_off, device)
                 for r in range(w.R)]
            rows = w.m // w.R if w.op == "rs" else w.m
            o = [torch.empty((rows, w.n), dtype=torch.bfloat16, device=device) for _ in range(w.R)]
            sets.append((a, b, o))
        ws = mk.Workspace(device)
        fn = mk.gemm_rs if w.op == "rs" else mk.gemm_ar
        key = "c_blocks" if w.op == "rs" else "c_replicas"
        steps_fns = {}
        for name, cfg in (("fused", mk.Config(cta_pair=pair)),
                          ("gemm_only", mk.Config(mode=mk.MODE_GEMM_ONLY, cta_pair=pair)),
                          ("unfused", mk.Config(mode=mk.MODE_UNFUSED, cta_pair=pair)),
                          # the reduction variants: bf16 running sum, atomic fp32 tiles
                          ("wire_bf16", mk.Config(wire=mk.WIRE_BF16, cta_pair=pair)),
                          ("atomic", mk.Config(reduce=mk.REDUCE_ATOMIC, cta_pair=pair))):
            def step(i, cfg=cfg):
                a, b, o = sets[i % nsets]
                fn(a, b, cfg=cfg, workspace=ws, stream=stream, **{key: o})
            steps_fns[name] = step
        n = steps if w.op == "rs" else steps * 10
        res = {name: tmax(t) for name, t in
               time_interleaved(steps_fns, n, 3, stream, dist).items()}
        st, _ = mk.device_status(ws, stream)
        flops = w.flops()
        fused_tf = flops / (res["fused"] * 1e-3) / 1e12
        entry = {"fused_ms": res["fused"], "gemm_only_ms": res["gemm_only"],
                 "unfused_ms": res["unfused"], "exposed_ms": res["fused"] - res["gemm_only"],
                 "fused_tflops": fused_tf, "pct_of_peak": 100 * fused_tf / bf16_peak,
                 "wire_bf16_ms": res["wire_bf16"], "atomic_ms": res["atomic"],
                 "status": mk.status_string(st)}
        if w.op == "ar":
            # algorithmic bytes: every B_r and A_r read once, the fp32 running sum forwarded
            # R-1 times (written and read back), and the R bf16 replicas written
            hbm_bytes = (w.R * (w.k * w.n * 2 + w.m * w.k * 2) + (w.R - 1) * 2 * w.m * w.n * 4
                         + w.R * w.m * w.n * 2)
            entry["bound"] = "hbm"
            entry["algorithmic_bytes"] = hbm_bytes
            entry["hbm_gbs"] = hbm_bytes / (res["fused"] * 1e-3) / 1e9
            entry["hbm_frac"] = entry["hbm_gbs"] / hbm_peak
            entry["roofline_frac"] = entry["hbm_frac"]
        else:
            entry["bound"] = "tensor"
            entry["roofline_frac"] = fused_tf / bf16_peak
        entry["traffic"] = recorded_traffic(w.name)
        if cpu:
            entry["cpu_baseline"] = cpu_gemm_baseline(sets[0][0], sets[0][1], w)
        out[w.name] = entry
        del sets, ws
        torch.cuda.empty_cache()
    if with_moe:
        out[I.MOE_R8_E64.name] = bench_moe(mk, device, stream, dist, steps, seed_off, tmax,
                                           bf16_peak, hbm_peak, cpu=cpu)
        torch.cuda.empty_cache()
        out[I.MOE_COMBINE_R8_E64.name] = bench_moe_combine(mk, device, stream, dist, steps, seed_off,
                                                           tmax, bf16_peak, hbm_peak)
        torch.cuda.empty_cache()
        out[I.MLP_R8_TP8.name] = bench_mlp(mk, device, stream, dist, max(3, steps // 3), seed_off, tmax,
                                           bf16_peak, hbm_peak)
        torch.cuda.empty_cache()
        out[I.AG_R8_TP8_UP.name + "_fp8"] = bench_ag_fp8(mk, device, stream, dist, steps, seed_off, tmax,
                                                         bf16_peak, hbm_peak)
        torch.cuda.empty_cache()
        for causal in (False, True):
            wr = I.RING_R8_H8_S4096_CAUSAL if causal else I.RING_R8_H8_S4096
            out[wr.name] = bench_ring(mk, device, stream, dist, max(3, steps // 3), seed_off, tmax,
                                      bf16_peak, hbm_peak, causal=causal)
            torch.cuda.empty_cache()
    return out


def bench_moe(mk, device, stream, dist, steps, seed_off, tmax, bf16_peak, hbm_peak, cpu=False):
    """MoE dispatch + grouped GEMM: fused, GEMM-only and unfused timings."""
    w = I.MOE_R8_E64
    sets = []
    for s in range(2):
        x = [dev_normal((w.T, w.H), 1.0, w.x_seed + r + 1000 * s + seed_off, device) for r in range(w.R)]
        lg = [I.zipf_logits(w.T, w.E, w.logit_seed + r + 1000 * s + seed_off).to(device)
              for r in range(w.R)]
        we = [dev_normal((w.E_loc, w.H, w.N), 0.02, w.w_seed + d + 1000 * s + seed_off, device)
              for d in range(w.R)]
        sets.append((x, lg, we))
    ws = mk.Workspace(device)
    outs = mk.moe_dispatch_gemm(*sets[0], E_loc=w.E_loc, topk=w.topk, workspace=ws, stream=stream)
    fns = {}
    for name, cfg in (("fused", None), ("gemm_only", mk.Config(mode=mk.MODE_GEMM_ONLY)),
                      ("unfused", mk.Config(mode=mk.MODE_UNFUSED))):
        def step(i, cfg=cfg):
            x, lg, we = sets[i % 2]
            mk.moe_dispatch_gemm(x, lg, we, E_loc=w.E_loc, topk=w.topk, out=outs, cfg=cfg,
                                 workspace=ws, stream=stream)
        fns[name] = step
    res = {name: tmax(t) for name, t in time_interleaved(fns, steps, 3, stream, dist).items()}
    st, _ = mk.device_status(ws, stream)
    flops = w.flops()
    rows = w.R * w.T * w.topk
    hbm_bytes = (rows * w.H * 2 * 2            # dispatch: read token rows, write recv_x
                 + rows * w.H * 2              # grouped GEMM reads recv_x
                 + w.R * w.E_loc * w.H * w.N * 2   # expert weights
                 + rows * w.N * 2              # y
                 + w.R * w.T * w.E * 4)        # logits
    fused_tf = flops / (res["fused"] * 1e-3) / 1e12
    t_tensor = flops / (bf16_peak * 1e12)
    t_hbm = hbm_bytes / (hbm_peak * 1e9)
    entry = {"fused_ms": res["fused"], "gemm_only_ms": res["gemm_only"], "unfused_ms": res["unfused"],
             "exposed_ms": res["fused"] - res["gemm_only"], "fused_tflops": fused_tf,
             "pct_of_peak": 100 * fused_tf / bf16_peak, "algorithmic_bytes": hbm_bytes,
             "roofline_ms": 1e3 * max(t_tensor, t_hbm),
             "roofline_frac": 1e3 * max(t_tensor, t_hbm) / res["fused"],
             "traffic": recorded_traffic(w.name),
             "status": mk.status_string(st)}
    if cpu:
        entry["cpu_baseline"] = cpu_moe_baseline(*sets[0], w)
    return entry


def bench_moe_combine(mk, device, stream, dist, steps, seed_off, tmax, bf16_peak, hbm_peak):
    """MoE combine (down-projection, return, top-k weighted sum): fused, GEMM-only
    (grouped GEMM + return of the rows, no sum) and unfused (that, then a sum launch)."""
    w = I.MOE_COMBINE_R8_E64
    wd = I.MOE_R8_E64
    # the routing of the MoE layer: one dispatch on the layer's token/logit inputs
    x = [dev_normal((wd.T, wd.H), 1.0, wd.x_seed + r + seed_off, device) for r in range(wd.R)]
    lg = [I.zipf_logits(w.T, w.E, w.logit_seed + r + seed_off).to(device) for r in range(w.R)]
    we = [dev_normal((wd.E_loc, wd.H, wd.N), 0.02, wd.w_seed + d + seed_off, device) for d in range(wd.R)]
    ws = mk.Workspace(device)
    disp = mk.moe_dispatch_gemm(x, lg, we, E_loc=w.E_loc, topk=w.topk, workspace=ws, stream=stream)
    del x, we
    sets = []
    for s in range(2):
        h = [dev_normal((w.cap, w.N), 1.0, w.h_seed + d + 1000 * s + seed_off, device) for d in range(w.R)]
        w2 = [dev_normal((w.E_loc, w.N, w.H), 0.02, w.w2_seed + d + 1000 * s + seed_off, device)
              for d in range(w.R)]
        gen = torch.Generator(device=device)
        gen.manual_seed(w.gate_seed + 1000 * s + seed_off)
        gates = []
        for r in range(w.R):
            u = torch.rand((w.T, w.topk), generator=gen, device=device) * 0.95 + 0.05
            gates.append((u / u.sum(dim=1, keepdim=True)).contiguous())
        sets.append((h, w2, gates))
    outs = mk.moe_combine(*sets[0], disp["recv_src"], disp["counts"], E_loc=w.E_loc, topk=w.topk,
                          workspace=ws, stream=stream)
    fns = {}
    for name, cfg in (("fused", None), ("gemm_only", mk.Config(mode=mk.MODE_GEMM_ONLY)),
                      ("unfused", mk.Config(mode=mk.MODE_UNFUSED))):
        def step(i, cfg=cfg):
            h, w2, gates = sets[i % 2]
            mk.moe_combine(h, w2, gates, disp["recv_src"], disp["counts"], E_loc=w.E_loc, topk=w.topk,
                           out=outs, cfg=cfg, workspace=ws, stream=stream)
        fns[name] = step
    res = {name: tmax(t) for name, t in time_interleaved(fns, steps, 3, stream, dist).items()}
    st, _ = mk.device_status(ws, stream)
    flops = w.flops()
    rows = w.R * w.T * w.topk
    hbm_bytes = (rows * w.N * 2                     # expert hidden rows
                 + w.R * w.E_loc * w.N * w.H * 2    # down-projection weights
                 + rows * w.H * 2 * 2               # returned rows: written, read by the sum
                 + w.R * w.T * w.H * 2              # combined outputs
                 + rows * (4 + 4))                  # gates, recv_src
    fused_tf = flops / (res["fused"] * 1e-3) / 1e12
    t_tensor = flops / (bf16_peak * 1e12)
    t_hbm = hbm_bytes / (hbm_peak * 1e9)
    return {"fused_ms": res["fused"], "gemm_only_ms": res["gemm_only"], "unfused_ms": res["unfused"],
            "exposed_ms": res["fused"] - res["gemm_only"], "fused_tflops": fused_tf,
            "pct_of_peak": 100 * fused_tf / bf16_peak, "algorithmic_bytes": hbm_bytes,
            "roofline_ms": 1e3 * max(t_tensor, t_hbm),
            "roofline_frac": 1e3 * max(t_tensor, t_hbm) / res["fused"],
            "traffic": recorded_traffic(w.name),
            "status": mk.status_string(st)}


def bench_mlp(mk, device, stream, dist, steps, seed_off, tmax, bf16_peak, hbm_peak):
    """Chained TP MLP (AllGather+GEMM -> ReLU -> GEMM+ReduceScatter): fused, GEMM-only
    (pre-gathered input, ranks summed in tensor memory) and unfused (four launches)."""
    w = I.MLP_R8_TP8
    M = w.R * w.m
    x = [dev_normal((w.m, w.h), 1.0, w.x_seed + r + seed_off, device) for r in range(w.R)]
    w1 = [dev_normal((w.h, w.f_r), w.w_std, w.w1_seed + r + seed_off, device) for r in range(w.R)]
    w2 = [dev_normal((w.f_r, w.h), w.w_std, w.w2_seed + r + seed_off, device) for r in range(w.R)]
    xg = torch.empty((M, w.h), dtype=torch.bfloat16, device=device)
    hid = [torch.empty((M, w.f_r), dtype=torch.bfloat16, device=device) for _ in range(w.R)]
    y = [torch.empty((w.m, w.h), dtype=torch.bfloat16, device=device) for _ in range(w.R)]
    ws = mk.Workspace(device)
    fns = {}
    for name, cfg in (("fused", None), ("gemm_only", mk.Config(mode=mk.MODE_GEMM_ONLY)),
                      ("unfused", mk.Config(mode=mk.MODE_UNFUSED))):
        def step(i, cfg=cfg):
            mk.mlp_ag_rs(x, w1, w2, x_gathered=xg, hid=hid, y_blocks=y, cfg=cfg, workspace=ws,
                         stream=stream)
        fns[name] = step
    res = {name: tmax(t) for name, t in time_interleaved(fns, steps, 3, stream, dist).items()}
    st, _ = mk.device_status(ws, stream)
    flops = w.flops()
    fused_tf = flops / (res["fused"] * 1e-3) / 1e12
    return {"fused_ms": res["fused"], "gemm_only_ms": res["gemm_only"], "unfused_ms": res["unfused"],
            "exposed_ms": res["fused"] - res["gemm_only"], "fused_tflops": fused_tf,
            "pct_of_peak": 100 * fused_tf / bf16_peak, "bound": "tensor",
            "roofline_frac": fused_tf / bf16_peak, "traffic": recorded_traffic(w.name),
            "status": mk.status_string(st)}


def bench_ag_fp8(mk, device, stream, dist, steps, seed_off, tmax, bf16_peak, hbm_peak):
    """AllGather+GEMM of the headline shape with fp8 e4m3 operands (B given as B^T):
    fused, GEMM-only and unfused.  Peak: the measured bf16 peak times the nominal
    fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)."""
    w = I.AG_R8_TP8_UP
    nsets = 3
    sets = []
    for s in range(nsets):
        a = [dev_normal((w.m, w.k), 1.0, w.a_seed + r + 1000 * s + seed_off, device).to(mk.FP8)
             for r in range(w.R)]
        bt = dev_normal((w.n, w.k), 1.0, w.b_seed + 1000 * s + seed_off, device).to(mk.FP8)
        g = torch.empty((w.R * w.m, w.k), dtype=mk.FP8, device=device)
        c = torch.empty((w.R * w.m, w.n), dtype=torch.bfloat16, device=device)
        sets.append((a, bt, g, c))
    ws = mk.Workspace(device)
    fns = {}
    for name, cfg in (("fused", None), ("gemm_only", mk.Config(mode=mk.MODE_GEMM_ONLY)),
                      ("unfused", mk.Config(mode=mk.MODE_UNFUSED))):
        def step(i, cfg=cfg):
            a, bt, g, c = sets[i % nsets]
            mk.ag_gemm(a, bt, a_gathered=g, c=c, cfg=cfg, workspace=ws, stream=stream)
        fns[name] = step
    res = {name: tmax(t) for name, t in time_interleaved(fns, steps, 3, stream, dist).items()}
    st, _ = mk.device_status(ws, stream)
    fp8_peak = 2.0 * bf16_peak
    fused_tf = w.flops() / (res["fused"] * 1e-3) / 1e12
    return {"fused_ms": res["fused"], "gemm_only_ms": res["gemm_only"], "unfused_ms": res["unfused"],
            "exposed_ms": res["fused"] - res["gemm_only"], "fused_tflops": fused_tf,
            "fp8_peak_tflops": fp8_peak, "pct_of_fp8_peak": 100 * fused_tf / fp8_peak,
            "status": mk.status_string(st)}


def bench_ring(mk, device, stream, dist, steps, seed_off, tmax, bf16_peak, hbm_peak, causal=False):
    """Ring attention: fused (ring transfers overlapped), GEMM-only (no ring: K/V read from
    their source ranks) and unfused (a transfer launch, then the attention)."""
    w = I.RING_R8_H8_S4096_CAUSAL if causal else I.RING_R8_H8_S4096
    shape = (w.heads, w.s_r, w.d)
    q = [dev_normal(shape, 1.0, w.q_seed + r + seed_off, device) for r in range(w.R)]
    k = [dev_normal(shape, 1.0, w.k_seed + r + seed_off, device) for r in range(w.R)]
    v = [dev_normal(shape, 1.0, w.v_seed + r + seed_off, device) for r in range(w.R)]
    out = [torch.empty(shape, dtype=torch.bfloat16, device=device) for _ in range(w.R)]
    kr = [torch.empty(((w.R - 1) * w.heads, w.s_r, w.d), dtype=torch.bfloat16, device=device)
          for _ in range(w.R)]
    vr = [torch.empty_like(t) for t in kr]
    ws = mk.Workspace(device)
    fns = {}
    for name, cfg in (("fused", None), ("gemm_only", mk.Config(mode=mk.MODE_GEMM_ONLY)),
                      ("unfused", mk.Config(mode=mk.MODE_UNFUSED))):
        def step(i, cfg=cfg):
            mk.ring_attention(q, k, v, causal=causal, out=out, k_recv=kr, v_recv=vr, cfg=cfg,
                              workspace=ws, stream=stream)
        fns[name] = step
    res = {name: tmax(t) for name, t in time_interleaved(fns, steps, 3, stream, dist).items()}
    st, _ = mk.device_status(ws, stream)
    flops = w.flops()
    fused_tf = flops / (res["fused"] * 1e-3) / 1e12
    return {"fused_ms": res["fused"], "gemm_only_ms": res["gemm_only"], "unfused_ms": res["unfused"],
            "exposed_ms": res["fused"] - res["gemm_only"], "fused_tflops": fused_tf,
            "pct_of_peak": 100 * fused_tf / bf16_peak, "bound": "tensor",
            "roofline_frac": fused_tf / bf16_peak,
            "traffic": recorded_traffic(w.name, kernel="mk_ring_attn_kernel"),
            "status": mk.status_string(st)}


if __name__ == "__main__":
    sys.exit(main())
