"""Summaries of the in-kernel trace (mk_config.trace = 1) of one AG / RS / AR / MoE / MLP call.

`summarize(records, copy_records)` reduces the records of the newest call to
per-wave figures: wave w is the w-th work item of every CTA.  For each wave it
gives the median time between consecutive accumulator-ready stamps of a CTA (the
item's MMA time in steady state), in microseconds and in SM cycles, the median
wait for the item's inputs, the epilogue time and the SM clock; the copy warps'
records give when the AllGather copy-in started and ended and its rate.

Run as a module on one GPU to trace a bench workload:

    python -m comm_gemm_tile_gb300.trace ag|rs|ar|moe|mlp [--mode fused|gemm] [--calls N] [--pair auto|off|on]

It makes the workload's inputs (seeded normal bf16, drawn on the device), runs N
untraced calls back to back to reach a steady clock and power state, then one
traced call, and prints the summary of that call.
"""
from __future__ import annotations

import argparse
import statistics

import torch

import comm_gemm_tile_gb300 as mk


def _newest(rec: torch.Tensor):
    """Indices of the records written by the newest call."""
    ep = rec[:, mk.TRACE_ID] >> 32
    sel = (ep == ep.max()) & (rec[:, mk.TRACE_START] != 0)
    return torch.nonzero(sel).flatten()


def _med(xs):
    return statistics.median(xs) if xs else float("nan")


def summarize(rec: torch.Tensor, copy_rec: torch.Tensor | None = None, max_rows: int = 12,
              items: tuple | None = None) -> dict:
    """items = (lo, hi): only work items lo <= i < hi (waves counted inside that range)."""
    idx = _newest(rec)
    if items is not None:
        it_ = idx // 2
        idx = idx[(it_ >= items[0]) & (it_ < items[1])]
    r = rec[idx]
    t0i = int(r[:, mk.TRACE_START].min())
    # differences in int64 first: the stamps are ~1e18 ns, beyond a double's integer range
    us = lambda col: ((r[:, col] - t0i).double() / 1e3).tolist()   # noqa: E731
    start, inputs, ready, end = us(mk.TRACE_START), us(mk.TRACE_INPUTS), us(mk.TRACE_READY), us(mk.TRACE_END)
    c0 = int(r[:, mk.TRACE_CLK_START].min())
    clk_s = (r[:, mk.TRACE_CLK_START] - c0).double().tolist()
    clk_r = (r[:, mk.TRACE_CLK_READY] - c0).double().tolist()
    ident = rec[idx, mk.TRACE_ID]
    cta = ((ident >> 1) & 0x7FFFFFFF).tolist()
    item = (idx // 2).tolist()
    per_cta: dict = {}
    for j in range(len(item)):
        per_cta.setdefault(cta[j], []).append(j)
    waves: dict = {}
    for js in per_cta.values():
        js.sort(key=lambda j: item[j])
        prev_t, prev_c = 0.0, None
        for w, j in enumerate(js):
            dt_ns = (ready[j] - start[j]) * 1e3
            mhz = (clk_r[j] - clk_s[j]) / dt_ns * 1e3 if dt_ns > 2000 else None
            gap_cyc = clk_r[j] - prev_c if prev_c is not None else None
            waves.setdefault(w, []).append({
                "gap_us": ready[j] - prev_t, "gap_cycles": gap_cyc, "input_wait_us": inputs[j] - start[j],
                "epilogue_us": end[j] - ready[j], "start_us": start[j], "mhz": mhz})
            prev_t, prev_c = ready[j], clk_r[j]
    out = {"records": len(item), "items": len(set(item)), "ctas": len(per_cta),
           "span_us": max(end) if end else 0.0, "waves": []}
    # at most max_rows rows: consecutive waves pooled into groups
    ws_ = sorted(waves)
    per = max(1, -(-len(ws_) // max_rows))
    for g0 in range(0, len(ws_), per):
        grp = ws_[g0:g0 + per]
        v = [x for w in grp for x in waves[w]]
        out["waves"].append({
            "wave": f"{grp[0]}" if len(grp) == 1 else f"{grp[0]}-{grp[-1]}", "n": len(v),
            "start_us": _med([x["start_us"] for x in v]),
            "ready_gap_us": _med([x["gap_us"] for x in v]),
            "ready_gap_cycles": _med([x["gap_cycles"] for x in v if x["gap_cycles"] is not None]),
            "input_wait_us": _med([x["input_wait_us"] for x in v]),
            "input_wait_max_us": max(x["input_wait_us"] for x in v),
            "epilogue_us": _med([x["epilogue_us"] for x in v]),
            "sm_mhz": _med([x["mhz"] for x in v if x["mhz"] is not None]),
        })
    if copy_rec is not None and copy_rec.shape[0]:
        ep_new = int(rec[idx, mk.TRACE_ID].max()) >> 32
        c = copy_rec[(copy_rec[:, mk.TRACE_ID] >> 32) == ep_new]
        if c.shape[0]:
            s_ = ((c[:, 0] - t0i).double() / 1e3).tolist()
            e_ = ((c[:, 1] - t0i).double() / 1e3).tolist()
            nbytes = float(c[:, 3].sum())
            out["copy"] = {"warps": c.shape[0], "start_us": _med(s_), "end_med_us": _med(e_),
                           "end_max_us": max(e_), "bytes": nbytes,
                           "tb_per_s": nbytes / ((max(e_) - min(s_)) * 1e-6) / 1e12}
    return out


def format_summary(d: dict, title: str = "") -> str:
    lines = []
    if title:
        lines.append(title)
    lines.append(f"{d['items']} items on {d['ctas']} CTAs ({d['records']} records), "
                 f"span {d['span_us']:.1f} us")
    lines.append("| wave | CTA items | start us | ready gap us | ready gap cycles | input wait us "
                 "(max) | epilogue us | SM MHz |")
    lines.append("|---|---|---|---|---|---|---|---|")
    for w in d["waves"]:
        lines.append(f"| {w['wave']} | {w['n']} | {w['start_us']:.1f} | {w['ready_gap_us']:.2f} | "
                     f"{w['ready_gap_cycles']:.0f} | {w['input_wait_us']:.2f} ({w['input_wait_max_us']:.2f}) | "
                     f"{w['epilogue_us']:.2f} | {w['sm_mhz']:.0f} |")
    if "copy" in d:
        c = d["copy"]
        lines.append(f"copy warps: {c['warps']}, start {c['start_us']:.1f} us, end median "
                     f"{c['end_med_us']:.1f} / max {c['end_max_us']:.1f} us, {c['bytes'] / 1e6:.1f} MB "
                     f"at {c['tb_per_s']:.2f} TB/s")
    return "\n".join(lines)


def _dev_normal(shape, std, seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (x * std).to(torch.bfloat16)


def _trace_moe(mode: str, calls: int, dev) -> str:
    from comm_gemm_tile_gb300 import inputs as I
    w = I.MOE_R8_E64
    m_mode = {"fused": mk.MODE_FUSED, "gemm": mk.MODE_GEMM_ONLY}[mode]
    sets = []
    for s in range(2):
        x = [_dev_normal((w.T, w.H), 1.0, w.x_seed + r + 1000 * s, dev) for r in range(w.R)]
        lg = [I.zipf_logits(w.T, w.E, w.logit_seed + r + 1000 * s).to(dev) for r in range(w.R)]
        we = [_dev_normal((w.E_loc, w.H, w.N), 0.02, w.w_seed + d + 1000 * s, dev) for d in range(w.R)]
        sets.append((x, lg, we))
    ws = mk.Workspace(dev)
    out = mk.moe_dispatch_gemm(*sets[0], E_loc=w.E_loc, topk=w.topk, cap_rows=w.cap, workspace=ws)

    def call(i, cfg):
        mk.moe_dispatch_gemm(*sets[i % 2], E_loc=w.E_loc, topk=w.topk, cap_rows=w.cap, out=out,
                             cfg=cfg, workspace=ws)

    cfg = mk.Config(mode=m_mode, trace=1)
    for i in range(calls):
        call(i, mk.Config(mode=m_mode))
    call(calls, cfg)
    st, detail = mk.device_status(ws)
    if st != mk.MK_OK:
        raise RuntimeError(f"traced call reported {mk.status_string(st)} ({detail})")
    rec, crec = mk.moe_trace_records(ws, w.R, w.E_loc, w.topk, w.T, w.H, w.N, w.cap, cfg)
    return format_summary(summarize(rec), f"{w.name}, {mode}, after {calls} untraced calls")


def _trace_mlp(mode: str, calls: int, dev) -> str:
    """The chained MLP: the up-projection tiles and the down-projection items
    summarised apart (item order: every up-projection tile first)."""
    from comm_gemm_tile_gb300 import inputs as I
    w = I.MLP_R8_TP8
    m_mode = {"fused": mk.MODE_FUSED, "gemm": mk.MODE_GEMM_ONLY}[mode]
    sets = []
    for s in range(2):
        x = [_dev_normal((w.m, w.h), 1.0, 40 + r + 1000 * s, dev) for r in range(w.R)]
        w1 = [_dev_normal((w.h, w.f_r), 0.02, 50 + r + 1000 * s, dev) for r in range(w.R)]
        w2 = [_dev_normal((w.f_r, w.h), 0.02, 60 + r + 1000 * s, dev) for r in range(w.R)]
        sets.append((x, w1, w2))
    ws = mk.Workspace(dev)
    xg, hid, y = mk.mlp_ag_rs(*sets[0], workspace=ws)

    def call(i, cfg):
        mk.mlp_ag_rs(*sets[i % 2], x_gathered=xg, hid=hid, y_blocks=y, cfg=cfg, workspace=ws)

    cfg = mk.Config(mode=m_mode, trace=1)
    for i in range(calls):
        call(i, mk.Config(mode=m_mode))
    # the traced call on a zero-filled workspace of its own: the fused call's
    # staging, where GEMM-only's records go, holds running sums
    ws = mk.Workspace(dev)
    call(calls, cfg)
    st, detail = mk.device_status(ws)
    if st != mk.MK_OK:
        raise RuntimeError(f"traced call reported {mk.status_string(st)} ({detail})")
    rec, crec = mk.mlp_trace_records(ws, w.R, w.m, w.h, w.f_r, cfg)
    rows = w.R * w.m
    n1 = w.R * (-(-rows // 256)) * (-(-w.f_r // 256))   # up-projection items on CTA pairs
    t = f"{w.name}, {mode}, after {calls} untraced calls"
    return "\n".join([format_summary(summarize(rec, crec, items=(0, n1)), t + ": up-projection tiles"),
                      format_summary(summarize(rec, items=(n1, rec.shape[0] // 2)),
                                     t + ": down-projection items")])


def trace_workload(op: str, mode: str = "fused", calls: int = 30, device="cuda:0", pair: int = 0) -> str:
    from comm_gemm_tile_gb300 import build
    from comm_gemm_tile_gb300 import inputs as I
    build.build()
    dev = torch.device(device)
    if op == "moe":
        return _trace_moe(mode, calls, dev)
    if op == "mlp":
        return _trace_mlp(mode, calls, dev)
    w = {"ag": I.AG_R8_TP8_UP, "rs": I.RS_R8_TP8_DOWN, "ar": I.AR_R8_DECODE}[op]
    m_mode = {"fused": mk.MODE_FUSED, "gemm": mk.MODE_GEMM_ONLY}[mode]
    nsets = 2
    sets = []
    for s in range(nsets):
        a = [_dev_normal((w.m, w.k), 1.0, w.a_seed + r + 1000 * s, dev) for r in range(w.R)]
        if op == "ag":
            b = _dev_normal((w.k, w.n), w.b_std, w.b_seed + 1000 * s, dev)
            g = torch.empty((w.R * w.m, w.k), dtype=torch.bfloat16, device=dev)
            c = torch.empty((w.R * w.m, w.n), dtype=torch.bfloat16, device=dev)
            sets.append((a, b, g, c))
        else:
            b = [_dev_normal((w.k, w.n), w.b_std, w.b_seed + r + 1000 * s, dev) for r in range(w.R)]
            rows = w.m // w.R if op == "rs" else w.m
            o = [torch.empty((rows, w.n), dtype=torch.bfloat16, device=dev) for _ in range(w.R)]
            sets.append((a, b, o))
    ws = mk.Workspace(dev)
    op_code = {"ag": mk.OP_AG_GEMM, "rs": mk.OP_GEMM_RS, "ar": mk.OP_GEMM_AR}[op]

    def call(i, cfg):
        st = sets[i % nsets]
        if op == "ag":
            mk.ag_gemm(st[0], st[1], a_gathered=st[2], c=st[3], cfg=cfg, workspace=ws)
        elif op == "rs":
            mk.gemm_rs(st[0], st[1], c_blocks=st[2], cfg=cfg, workspace=ws)
        else:
            mk.gemm_ar(st[0], st[1], c_replicas=st[2], cfg=cfg, workspace=ws)

    if op == "ag" and m_mode == mk.MODE_GEMM_ONLY:
        for i in range(nsets):           # GEMM-only reads the gathered A as it stands
            call(i, mk.Config())
    cfg = mk.Config(mode=m_mode, trace=1, cta_pair=pair)
    for i in range(calls):
        call(i, mk.Config(mode=m_mode, cta_pair=pair))
    call(calls, cfg)
    st, detail = mk.device_status(ws)
    if st != mk.MK_OK:
        raise RuntimeError(f"traced call reported {mk.status_string(st)} ({detail})")
    rec = mk.trace_records(ws, op_code, w.R, w.m, w.n, w.k, cfg)
    crec = mk.trace_copy_records(ws, op_code, w.R, w.m, w.n, w.k, cfg) if op == "ag" else None
    return format_summary(summarize(rec, crec), f"{w.name}, {mode}, after {calls} untraced calls")


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("op", choices=["ag", "rs", "ar", "moe", "mlp"])
    ap.add_argument("--mode", choices=["fused", "gemm"], default="fused")
    ap.add_argument("--calls", type=int, default=30)
    ap.add_argument("--pair", choices=["auto", "off", "on"], default="auto",
                    help="CTA pairs for AG / RS / AR (mk_config.cta_pair)")
    args = ap.parse_args()
    pair = {"auto": mk.PAIR_AUTO, "off": mk.PAIR_OFF, "on": mk.PAIR_ON}[args.pair]
    print(trace_workload(args.op, args.mode, args.calls, pair=pair))


if __name__ == "__main__":
    main()
