"""Where the time of one decode call goes, read from %globaltimer stamps.

Builds libsanta_timeline.so (the library compiled with -DSANTA_TIMELINE), runs decode calls
on the synthetic inputs of a named workload, reads the stamps that every CTA wrote at its
phase boundaries and prints, per quantity, the median over the calls.  Every time is in
microseconds from the first CTA's entry into the first kernel of the call.  The timer ticks
in steps of about 0.26 us, so a phase shorter than that reads 0 or 0.26.

    python -m stochastic_sparse_kv_gb300.timeline --workload llama8b_b16_32k --S 256
    python -m stochastic_sparse_kv_gb300.timeline --workload llama8b_b1_32k --two-pass --json

One library build per process: run it as its own process, not after libsanta.so was loaded.
"""
from __future__ import annotations

import argparse
import json
import statistics

import numpy as np
import torch

from . import _build, santa, workloads

ROWS_SCORE = 1024  # rows [0, 1024): CTAs of the score or single-pass kernel
COLS = 16

# two-pass layout: the score kernel's stamps (columns) and the value stage's phases
SCORE_MARKS = {"producer done": 1, "roles done": 2, "cta end": 3}
VALUE_PHASES = (("A chunk data", 1, 2), ("B fixed point + hot", 2, 3), ("C heavy keys", 3, 4),
                ("D re-score", 4, 5), ("E prefix", 5, 6), ("F search", 6, 7), ("F discards", 7, 8),
                ("G index out + loads", 8, 9), ("G reduce + out", 9, 10))
# single-pass cluster kernel: absolute marks and the phases between consecutive stamps
CLUSTER_MARKS = {"setup done": 1, "producer done": 2, "score roles done": 3, "value stage start": 5,
                 "cta end": 11}
CLUSTER_PHASES = (("teardown", 3, 4), ("value init", 4, 5), ("1 max/scale exchange", 5, 6),
                  ("2 fixed point + heavy keys", 6, 7), ("3 prefix + range totals", 7, 8),
                  ("4 search", 8, 9), ("5 distinct rows + loads", 9, 10), ("slice exchange + out", 10, 11))


def _spread(x: np.ndarray) -> dict:
    if x.size == 0:
        return {"min": None, "med": None, "max": None}
    return {"min": float(x.min()), "med": float(np.median(x)), "max": float(x.max())}


def _durations(x: np.ndarray) -> dict:
    if x.size == 0:
        return {"med": None, "p90": None, "max": None}
    return {"med": float(np.median(x)), "p90": float(np.percentile(x, 90)), "max": float(x.max())}


def analyse(stamps: np.ndarray, single_pass: bool) -> dict:
    """The quantities of one call from its stamp array [rows, 16] (uint64 ns, 0 = not
    written).  Pure host arithmetic, so that it can be checked without a GPU."""
    st = stamps.astype(np.int64)
    sc = st[:ROWS_SCORE]
    sc = sc[sc[:, 0] != 0]
    if sc.shape[0] == 0:
        raise ValueError("no stamps: was the call made through libsanta_timeline.so?")
    t0 = int(sc[:, 0].min())
    us = lambda a: (a - t0) / 1e3  # noqa: E731
    r = {"ctas": int(sc.shape[0])}
    if single_pass:
        r["marks"] = {k: _spread(us(sc[sc[:, c] != 0, c])) for k, c in CLUSTER_MARKS.items()}
        r["phases"] = {k: _durations((sc[:, c1] - sc[:, c0])[(sc[:, c0] != 0) & (sc[:, c1] != 0)] / 1e3)
                       for k, c0, c1 in CLUSTER_PHASES}
        r["end"] = float(us(sc[:, 11].max()))
        return r
    r["marks"] = {k: _spread(us(sc[sc[:, c] != 0, c])) for k, c in SCORE_MARKS.items()}
    va = st[ROWS_SCORE:]
    va = va[va[:, 0] != 0]
    r["value_ctas"] = int(va.shape[0])
    r["value_entry"] = _spread(us(va[:, 0]))
    waited = va[va[:, 1] != 0]
    r["value_wait_done"] = _spread(us(waited[:, 1]))
    stream_end = int(sc[:, 3].max())
    r["value_ctas_entered_before_score_end"] = int((va[:, 0] < stream_end).sum())
    r["phases"] = {k: _durations((va[:, c1] - va[:, c0])[(va[:, c0] != 0) & (va[:, c1] != 0)] / 1e3)
                   for k, c0, c1 in VALUE_PHASES}
    full = va[va[:, 10] != 0]
    r["value_total"] = _durations((full[:, 10] - full[:, 1]) / 1e3)
    r["end"] = float(us(va[:, 1:11].max())) if va.size else float(us(sc[:, 3].max()))
    return r


def _median_over_calls(results: list) -> dict:
    """Each numeric leaf: its median over the calls."""
    first = results[0]
    if isinstance(first, dict):
        return {k: _median_over_calls([x[k] for x in results]) for k in first}
    vals = [x for x in results if x is not None]
    return float(statistics.median(vals)) if vals else None


def run(w: workloads.Workload, S: int, mode: str = "systematic", two_pass: bool = False, bernoulli: bool = False,
        group_dedup: bool = False, calls: int = 20, warmup: int = 5, device: str = "cuda:0",
        library: str | None = None) -> dict:
    """`library`: a stamped build to load instead of building libsanta_timeline.so."""
    lib = santa.load(library or _build.build(timeline=True))
    dev = torch.device(device)
    torch.cuda.set_device(dev)
    q, k, v, sl = workloads.make_inputs_device(w, dev)
    shape = santa.make_shape(w.B, w.H_q, w.H_kv, w.d, w.n_max, 0.0)
    launches = santa.call_info(shape, S, mode, group_dedup, bernoulli, two_pass)
    single = launches == 1 + (1 if bernoulli else 0) and mode != "dense"
    rows = ROWS_SCORE + w.B * w.H_q
    buf = torch.zeros((rows, COLS), dtype=torch.int64, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)  # larger than L2
    plan = santa.DecodePlan(q, k, v, sl, S, mode, group_dedup=group_dedup, bernoulli=bernoulli, two_pass=two_pass)
    rc = lib.santa_timeline_buffer(buf.data_ptr(), buf.numel() * 8)
    if rc != 0:
        raise santa.SantaError(rc, "santa_timeline_buffer")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per_call, event_us = [], []
    try:
        for i in range(warmup + calls):
            buf.zero_()
            flush.zero_()
            torch.cuda.synchronize()
            ev0.record()
            plan(1000 + i)
            ev1.record()
            torch.cuda.synchronize()
            if i >= warmup:
                event_us.append(ev0.elapsed_time(ev1) * 1e3)
                per_call.append(analyse(buf.cpu().numpy(), single))
    finally:
        lib.santa_timeline_buffer(None, 0)
    out = _median_over_calls(per_call)
    out.update({"workload": w.name, "S": S, "mode": mode, "two_pass": two_pass, "bernoulli": bernoulli,
                "group_dedup": group_dedup, "layout": "single-pass cluster kernel" if single else "two launches",
                "launches": launches, "calls": calls, "event_us": float(statistics.median(event_us))})
    return out


def report(r: dict) -> str:
    f = lambda x: "   -  " if x is None else f"{x:6.2f}"  # noqa: E731
    flags = "".join(f", {k.replace('_', ' ')}" for k in ("group_dedup", "bernoulli") if r.get(k))
    lines = [f"== {r['workload']} S={r['S']} {r['mode']}{flags} ({r['layout']}, {r['launches']} launches): "
             f"event {r['event_us']:.1f} us (stamped build), end of last CTA {r['end']:.1f} us, CTAs {r['ctas']:.0f}"]
    for k, m in r["marks"].items():
        lines.append(f"  {k:28s} min {f(m['min'])} med {f(m['med'])} max {f(m['max'])}")
    if "value_entry" in r:
        for k in ("value_entry", "value_wait_done"):
            m = r[k]
            lines.append(f"  {k:28s} min {f(m['min'])} med {f(m['med'])} max {f(m['max'])}")
        lines.append(f"  value CTAs entered before the score grid ended: {r['value_ctas_entered_before_score_end']:.0f}"
                     f" of {r['value_ctas']:.0f}")
    lines.append("  phase durations per CTA (us):")
    for k, m in r["phases"].items():
        lines.append(f"    {k:28s} med {f(m['med'])} p90 {f(m['p90'])} max {f(m['max'])}")
    if "value_total" in r:
        m = r["value_total"]
        lines.append(f"    {'value stage, wait done -> end':28s} med {f(m['med'])} p90 {f(m['p90'])} max {f(m['max'])}")
    return "\n".join(lines)


def _workload(name: str) -> workloads.Workload:
    table = {x.name: x for x in (workloads.LLAMA_B1, workloads.BATCHED, workloads.RAGGED, *workloads.LONG,
                                 workloads.LONG_GLOBAL)}
    if name not in table:
        raise SystemExit(f"unknown workload {name}; one of {sorted(table)}")
    return table[name]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--workload", default=workloads.BATCHED.name)
    ap.add_argument("--S", type=int, default=256)
    ap.add_argument("--mode", default="systematic", choices=("systematic", "stratified", "iid"))
    ap.add_argument("--two-pass", action="store_true")
    ap.add_argument("--bernoulli", action="store_true")
    ap.add_argument("--group-dedup", action="store_true")
    ap.add_argument("--calls", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--json", action="store_true")
    ap.add_argument("--library", default=None, help="a stamped build (-DSANTA_TIMELINE) to load instead")
    a = ap.parse_args(argv)
    r = run(_workload(a.workload), a.S, a.mode, a.two_pass, a.bernoulli, a.group_dedup, a.calls, a.warmup,
            library=a.library)
    print(json.dumps(r) if a.json else report(r))


if __name__ == "__main__":
    main()
