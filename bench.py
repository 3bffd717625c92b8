"""Benchmark: SANTA decode-step attention on synthetic Llama-3.1-8B-shaped KV caches.

One step = one santa_decode call over a batch: scores over all cached keys, softmax CDF,
S sample points per query head, and the gather-add of the sampled V rows.  Default
workload: B=16, H_q=32, H_kv=8, d=128, n_k=32768, S=256, systematic sampling.  Prints ONE
JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The line carries the headline (`value`, µs per step, one pair of CUDA events around the
timed steps), `roofline` (algorithmic bytes per call over the measured copy peak, and the
DRAM traffic of an ncu record taken on the same sources), `clocks` sampled during the
timed region, `e2e` (host buffers copied in and out every step), `cpu_baseline` (the
oracle) and `gpu_launches`.  Unless --no-extras: the other sampling modes and dense, S
sweeps, Bernoulli qK^T, group dedup, a 32-layer CUDA-graph stack and (unless
--no-workloads) every other configuration of the workload table.

--impl reference times the fp64 CPU oracle on this machine's host cores on a bounded
sample of the same workload, scaled to the same unit.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SANTA decode-attn µs/step @32k ctx, B=16, S=256; achieved HBM GB/s vs dense"
UNIT = "us/step"
FALLBACK_HBM_GBS = 6800.0
# GB300's nominal HBM3e bandwidth: the denominator of the 70%-of-roofline target as the
# target is stated.  `frac` uses the measured copy bandwidth; `frac_of_nominal` this.
NOMINAL_HBM_GBS = 8000.0
# GB300's L2 is 129 MB: timed configurations whose K/V cache is smaller than three times
# that rotate among copies of it (each step then reads data no recent step touched)
L2_ROTATE_BYTES = 3 * 129 * 1000 * 1000
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "santa_decode_b16_32k_traffic.txt")
CSRC = os.path.join("stochastic_sparse_kv_gb300", "csrc")
KERNEL_SOURCES = [os.path.join(CSRC, f) for f in ("santa_common.cuh", "santa_sample.cuh", "santa_tcgen05.cuh", "santa_score.cuh",
                                                   "santa_gather.cuh", "santa_dense.cuh", "santa_cluster.cuh",
                                                   "santa_kernels.h", "santa_kernels_d128.cu", "santa_kernels_d64.cu",
                                                   "santa_api.cu")]
# The sampled path is two launches chained by programmatic dependent launch (the value
# stage's launch and prologue overlap the score grid's end), so one santa_decode call is
# timed as the unit.
ROOFLINE_UNIT = "santa_decode: santa_score_kernel<128,4> + santa_gather_kernel<128,4,0,256> (PDL-chained)"
ROOFLINE_UNIT_DENSE = "santa_decode (dense): santa_dense_kernel<128,4> + santa_dense_merge_kernel<128> (PDL-chained)"


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def algorithmic_bytes(B, H_q, H_kv, d, seq_lens, S, mode):
    """All of K (each valid key row once), the S gathered V rows per query head (dense:
    all of V), q and the fp32 output."""
    nk = sum(int(n) for n in seq_lens)
    kbytes = H_kv * nk * d * 2
    q = B * H_q * d * 2
    out = B * H_q * d * 4
    if mode == "dense":
        return 2 * kbytes + q + out + 4 * B
    nz = sum(1 for n in seq_lens if n > 0)
    return kbytes + nz * H_q * S * d * 2 + q + out + 4 * B


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def sources_sha():
    h = hashlib.sha256()
    for s in KERNEL_SOURCES:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """dram read+write bytes per launch from the committed ncu summary, or None when the
    kernel sources changed since the capture."""
    try:
        kv = {}
        with open(PROFILE_TRAFFIC) as f:
            for line in f:
                if "=" in line and not line.startswith("#"):
                    a, b = line.strip().split("=", 1)
                    kv[a.strip()] = b.strip()
        if kv.get("source_sha") != sources_sha():
            return None
        return float(kv["traffic_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
                self.lines = [l for l in out.splitlines() if l.strip()]
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus):
    if n_gpus <= 1 or "RANK" not in os.environ:
        return 0, 1, None
    import torch.distributed as dist
    dist.init_process_group("nccl")
    return dist.get_rank(), dist.get_world_size(), dist


def time_steps(fn, steps, warmup, stream, dist=None):
    """W untimed steps, then exactly `steps` timed steps bracketed by barrier + sync and one
    pair of CUDA events on the launching stream (no events between the steps: at small
    batches their own cost would show); returns (total ms over the max of ranks, the mean
    ms of one step on this rank, repeated per step)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        fn()
    t1.record(stream)
    torch.cuda.synchronize()
    local = t0.elapsed_time(t1)
    total = max_over_ranks(local, dist, "cuda")
    torch.cuda.synchronize()
    return total, [local / steps] * steps


def max_over_ranks(value, dist=None, device="cpu"):
    """The largest `value` over all ranks (each rank runs an independent replica; the
    step takes as long as the slowest), followed by a barrier.  `dist` is
    torch.distributed or None (one process)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def multi_layer(n_layers, w, S, dev, peak, reps=20):
    """Attention of one decode step through an n_layers-deep model without weights: every
    layer has its own KV cache (so nothing is reused from L2 between layers) and writes a
    bf16 output, and the whole stack of calls is captured in one CUDA graph and replayed.
    Returns per-token times for the sampled (systematic) and the dense path."""
    import torch
    from stochastic_sparse_kv_gb300 import santa
    B, H_q, H_kv, d, n = w.B, w.H_q, w.H_kv, w.d, w.n_max
    try:
        gen = torch.Generator(device=dev)
        gen.manual_seed(20261202)
        kv, qs = [], []
        for _ in range(n_layers):
            kv.append((torch.randn(B, H_kv, n, d, device=dev, generator=gen).to(torch.bfloat16),
                       torch.randn(B, H_kv, n, d, device=dev, generator=gen).to(torch.bfloat16)))
            g = torch.randn(B, H_q, d, device=dev, generator=gen)
            qs.append((3.0 * d ** 0.5 * g / g.norm(dim=-1, keepdim=True)).to(torch.bfloat16))
    except torch.cuda.OutOfMemoryError as e:
        return {"skipped": f"out of device memory for {n_layers} layers: {e}"[:200]}
    sl = torch.full((B,), n, dtype=torch.int32, device=dev)
    outs = [torch.empty(B, H_q, d, dtype=torch.bfloat16, device=dev) for _ in range(n_layers)]
    shape = santa.make_shape(B, H_q, H_kv, d, n)
    ws = santa.new_workspace(max(santa.workspace_size(shape, S, "systematic"),
                                 santa.workspace_size(shape, 1, "dense")), dev)
    res = {"layers": n_layers, "kv_cache_gb": round(n_layers * 2 * B * H_kv * n * d * 2 / 1e9, 1),
           "out": "bf16", "graph": True}
    for mode in ("systematic", "dense"):
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for li in range(n_layers):  # eager warm-up (kernel attributes, tensor maps)
                santa.decode(qs[li], kv[li][0], kv[li][1], sl, S, mode, seed=li, out=outs[li], want_idx=False,
                             workspace=ws, stream=side)
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for li in range(n_layers):
                    santa.decode(qs[li], kv[li][0], kv[li][1], sl, S, mode, seed=li, out=outs[li],
                                 want_idx=False, workspace=ws, stream=side)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        us_tok = e0.elapsed_time(e1) * 1000.0 / reps
        ab = n_layers * algorithmic_bytes(B, H_q, H_kv, d, [n] * B, S, mode)
        res[mode] = {"us_per_token": round(us_tok, 1), "us_per_layer": round(us_tok / n_layers, 2),
                     "frac_of_peak": round(ab / (us_tok * 1e-6) / 1e9 / peak, 4)}
        del graph
    res["speedup_vs_dense"] = round(res["dense"]["us_per_token"] / res["systematic"]["us_per_token"], 3)
    del kv, qs, outs
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    import numpy as np
    import torch
    from stochastic_sparse_kv_gb300 import santa, workloads

    rank, world, dist = dist_setup(args.gpus)
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    santa.load()
    w = pick_workload(args.workload)
    S = args.S
    log(f"[bench] generating inputs {w.name} (B={w.B}, n={w.n_max}) ...")
    q, k, v, sl = workloads.make_inputs(w)
    qd, kd, vd, sld = q.to(dev), k.to(dev), v.to(dev), sl.to(dev)
    stream = torch.cuda.current_stream()
    B, H_q, H_kv, d = w.B, w.H_q, w.H_kv, w.d
    out = torch.empty(B, H_q, d, dtype=torch.float32, device=dev)
    idx = torch.empty(B, H_q, S, dtype=torch.int32, device=dev)
    seq = sl.tolist()

    plans = {}  # one prepared call per configuration: each step is a single foreign call

    def step_mode(mode, S_=S, seed_box=[0], group_dedup=False, bernoulli=False):
        key = (mode, S_, group_dedup, bernoulli)
        if key not in plans:
            with_idx = mode != "dense" and S_ == S
            plans[key] = santa.DecodePlan(qd, kd, vd, sld, S_, mode, out=out, idx_out=(idx if with_idx else None),
                                          want_idx=with_idx, group_dedup=group_dedup, stream=stream,
                                          bernoulli=bernoulli)
        plan = plans[key]

        def f():
            seed_box[0] += 1
            plan(seed_box[0])
        return f

    peak, peak_kind = measured_peak()
    mode = args.mode
    launches_per_step = santa.call_info(santa.make_shape(B, H_q, H_kv, d, w.n_max), S, mode)
    with ClockSampler(local) as clk:
        total_ms, per = time_steps(step_mode(mode), args.steps, args.warmup, stream, dist)
    clocks = clk.summary()
    us_step = total_ms * 1000.0 / args.steps
    avg_launch_ms = sum(per) / len(per)
    abytes = algorithmic_bytes(B, H_q, H_kv, d, seq, S, mode)
    achieved = abytes / (avg_launch_ms * 1e-3) / 1e9

    # the other modes and the S sweep (same inputs, shorter runs)
    extra_steps = max(10, min(args.steps, 50))
    modes = {}
    for m in (() if args.no_extras else ("systematic", "stratified", "dense")):
        tm, pm = time_steps(step_mode(m), extra_steps, 3, stream, dist)
        ab = algorithmic_bytes(B, H_q, H_kv, d, seq, S, m)
        al = sum(pm) / len(pm)
        modes[m] = {"us_per_step": round(tm * 1000 / extra_steps, 2),
                    "achieved_gbs": round(ab / (al * 1e-3) / 1e9, 1),
                    "frac_of_peak": round(ab / (al * 1e-3) / 1e9 / peak, 4),
                    "algorithmic_bytes": ab}
    for m in (() if args.no_extras else ("systematic", "stratified")):
        modes[m]["speedup_vs_dense"] = round(modes["dense"]["us_per_step"] / modes[m]["us_per_step"], 3)
    sweep = {}
    for S2 in (() if args.no_extras else workloads.BATCHED_S_SWEEP):
        tm, pm = time_steps(step_mode("systematic", S2), extra_steps, 3, stream, dist)
        ab = algorithmic_bytes(B, H_q, H_kv, d, seq, S2, "systematic")
        al = sum(pm) / len(pm)
        sweep[str(S2)] = {"us_per_step": round(tm * 1000 / extra_steps, 2),
                          "frac_of_peak": round(ab / (al * 1e-3) / 1e9 / peak, 4)}

    sweep_strat = {}
    for S2 in (() if args.no_extras else workloads.BATCHED_S_SWEEP):
        tm, pm = time_steps(step_mode("stratified", S2), extra_steps, 3, stream, dist)
        ab = algorithmic_bytes(B, H_q, H_kv, d, seq, S2, "stratified")
        al = sum(pm) / len(pm)
        sweep_strat[str(S2)] = {"us_per_step": round(tm * 1000 / extra_steps, 2),
                                "frac_of_peak": round(ab / (al * 1e-3) / 1e9 / peak, 4)}

    # Bernoulli qK^T (the ternary query draws), same inputs
    variants = {}
    for name, kw in (() if args.no_extras else (("bernoulli_qk", {"bernoulli": True}),)):
        row = {}
        for m in ("systematic", "dense") if name == "bernoulli_qk" else ("systematic",):
            tm, _ = time_steps(step_mode(m, **kw), extra_steps, 3, stream, dist)
            row[m] = round(tm * 1000 / extra_steps, 2)
        variants[name] = row
    if "bernoulli_qk" in variants:
        # the fraction of key features the ternary queries select: per head, and the union
        # over the G heads that share a KV head (what a feature-major cache could skip)
        qt = santa.ternary_query(qd, 1).view(B, H_kv, H_q // H_kv, d) != 0
        variants["bernoulli_qk"]["feature_density_per_head"] = round(float(qt.float().mean()), 4)
        variants["bernoulli_qk"]["feature_density_per_kv_group"] = round(float(qt.any(2).float().mean()), 4)

    # the opt-in group deduplication of V loads (SANTA_GROUP_DEDUP) against the default
    gdd = {}
    for S2 in (() if args.no_extras else (256, 2048)):
        row = {}
        for flag in (False, True):
            tm, _ = time_steps(step_mode("systematic", S2, group_dedup=flag), extra_steps, 3, stream, dist)
            row["group_dedup" if flag else "per_head"] = round(tm * 1000 / extra_steps, 2)
        gdd[str(S2)] = row

    # every configuration of the workload table, each mode (inputs drawn on the device)
    wl, gdd_w = {}, {}
    if not args.no_extras and not args.no_workloads:
        for w2, S_list in workload_table(workloads):
            log(f"[bench] workload {w2.name} ...")
            q2, k2, v2, sl2 = workloads.make_inputs_device(w2, dev)
            seq2 = sl2.tolist()
            o2 = torch.empty(w2.B, w2.H_q, w2.d, dtype=torch.float32, device=dev)
            # a cache smaller than L2 would stay in it from one step to the next: rotate
            # among enough copies that each step reads memory the previous ones did not
            kv_bytes = 2 * k2.numel() * k2.element_size()
            ncopy = max(1, -(-L2_ROTATE_BYTES // kv_bytes))
            caches = [(k2, v2)] + [(k2.clone(), v2.clone()) for _ in range(ncopy - 1)]
            for S2 in S_list:
                for m in ("systematic", "stratified", "dense"):
                    if m == "dense" and S2 != S_list[-1]:
                        continue
                    plans2 = [santa.DecodePlan(q2, kc, vc, sl2, S2, m, out=o2, want_idx=False, stream=stream)
                              for kc, vc in caches]
                    sb = [0]

                    def f(plans2=plans2, sb=sb):
                        sb[0] += 1
                        plans2[sb[0] % len(plans2)](sb[0])
                    tm, pm = time_steps(f, extra_steps, 3, stream, dist)
                    ab = algorithmic_bytes(w2.B, w2.H_q, w2.H_kv, w2.d, seq2, S2, m)
                    al = sum(pm) / len(pm)
                    key = f"{w2.name}/{m}" + ("" if m == "dense" else f"/S{S2}")
                    wl[key] = {"us_per_step": round(tm * 1000 / extra_steps, 2),
                               "frac_of_peak": round(ab / (al * 1e-3) / 1e9 / peak, 4),
                               "l2": (f"rotates {ncopy} copies of the K/V cache ({ncopy * kv_bytes / 1e6:.0f} MB)"
                                      if ncopy > 1 else f"K/V cache {kv_bytes / 1e6:.0f} MB > L2"),
                               "launches": santa.call_info(santa.make_shape(w2.B, w2.H_q, w2.H_kv, w2.d, w2.n_max),
                                                           S2, m)}
                    del plans2
            if w2.heavy_frac > 0:
                # the heavy-hitter batch is where the heads of a group share sampled rows: the
                # opt-in group deduplication against the default, as for the headline batch
                row_all = {}
                for S2 in (256, 2048):
                    row = {}
                    for flag in (False, True):
                        pl = santa.DecodePlan(q2, k2, v2, sl2, S2, "systematic", out=o2, want_idx=False,
                                              stream=stream, group_dedup=flag)
                        sb = [0]

                        def f(pl=pl, sb=sb):
                            sb[0] += 1
                            pl(sb[0])
                        tm, _ = time_steps(f, extra_steps, 3, stream, dist)
                        row["group_dedup" if flag else "per_head"] = round(tm * 1000 / extra_steps, 2)
                        del pl
                    row_all[str(S2)] = row
                gdd_w[w2.name] = row_all
            del q2, k2, v2, sl2, o2, caches
            torch.cuda.empty_cache()
        for key in list(wl):
            if "/dense" in key:
                continue
            dk = key.rsplit("/", 2)[0] + "/dense"
            if dk in wl:
                wl[key]["speedup_vs_dense"] = round(wl[dk]["us_per_step"] / wl[key]["us_per_step"], 3)

    # end to end through the C ABI with host buffers: H2D inputs, decode, D2H result
    e2e = None
    if args.e2e_steps > 0:
        qh, kh, vh, slh = (t.cpu().pin_memory() for t in (q, k, v, sl))
        outh = torch.empty(B, H_q, d, dtype=torch.float32).pin_memory()
        idxh = torch.empty(B, H_q, S, dtype=torch.int32).pin_memory()

        def e2e_step():
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            sld.copy_(slh, non_blocking=True)
            santa.decode(qd, kd, vd, sld, S, mode, seed=1, out=out, idx_out=idx)
            outh.copy_(out, non_blocking=True)
            idxh.copy_(idx, non_blocking=True)
        te, _ = time_steps(e2e_step, args.e2e_steps, 2, stream, dist)
        h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh, slh))
        d2h = outh.numel() * 4 + idxh.numel() * 4
        e2e = {"value": round(te * 1000 / args.e2e_steps, 2), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    # CPU baseline: the fp64 oracle, as it stands, on a bounded sample (rank 0, N=1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(q, k, v, sl, w, S, mode, args.cpu_rows)

    # the attention of a whole decode step through a 32-layer stack (CUDA graph, bf16 out)
    ml = None
    if not args.no_extras and args.layers > 0 and world == 1:
        log(f"[bench] multi-layer decode: {args.layers} layers ...")
        ml = multi_layer(args.layers, w, S, dev, peak)

    if rank == 0:
        # the committed DRAM record covers the sampled path's launch pair only
        traffic = profiled_traffic() if mode != "dense" else None
        rec = {
            "metric": METRIC, "value": round(us_step, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us_step / 1000, 5),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded N(0,1) bf16 K/V, q scaled to score std 3; Llama-3.1-8B attention shape)",
            "config": {"workload": w.name, "B": B, "H_q": H_q, "H_kv": H_kv, "d": d, "n_k": w.n_max, "S": S,
                       "mode": mode,
                       "l2": f"inputs larger than L2 (K/V cache {2 * kd.numel() * kd.element_size() / 1e9:.2f} GB > 129 MB L2)"
                       if 2 * kd.numel() * kd.element_size() > L2_ROTATE_BYTES else
                       "K/V cache smaller than 3x L2: these steps may partly hit L2 (the workloads table rotates copies)",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic, "peak_kind": peak_kind,
                         "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                         "nominal_peak": NOMINAL_HBM_GBS,
                         "kernel": ROOFLINE_UNIT_DENSE if mode == "dense" else ROOFLINE_UNIT,
                         "algorithmic_bytes_per_launch": abytes,
                         "avg_launch_us": round(avg_launch_ms * 1000, 2)},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps * launches_per_step,
            "clocks": clocks,
            "modes": modes,
            "S_sweep_systematic": sweep,
            "S_sweep_stratified": sweep_strat,
            "variants_us_per_step": variants,
            "workloads": wl,
            "group_dedup_us_per_step": {args.workload: gdd, **gdd_w},
            "multi_layer": ml,
        }
        print(json.dumps(rec), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def workload_table(workloads):
    """The configurations timed under `workloads` (each with its S values)."""
    table = [(workloads.LLAMA_B1, (256,))]
    table += [(lw, (128, 256)) for lw in workloads.LONG]
    table.append((workloads.RAGGED, (256,)))
    table.append((workloads.LONG_GLOBAL, (256,)))
    return table


def pick_workload(name):
    from stochastic_sparse_kv_gb300 import workloads
    table = {workloads.BATCHED.name: workloads.BATCHED, workloads.LLAMA_B1.name: workloads.LLAMA_B1,
             workloads.RAGGED.name: workloads.RAGGED, workloads.LONG_GLOBAL.name: workloads.LONG_GLOBAL}
    for lw in workloads.LONG:
        table[lw.name] = lw
    if name not in table:
        raise SystemExit(f"unknown workload {name}; one of {sorted(table)}")
    return table[name]


def cpu_baseline(q, k, v, sl, w, S, mode, rows):
    """Time the oracle on `rows` batch rows of the workload; scale to one full step."""
    import oracle
    rows = max(1, min(rows, w.B))
    qs, ks, vs, ss = q[:rows].contiguous(), k[:rows].contiguous(), v[:rows].contiguous(), sl[:rows]
    om = "dense" if mode == "dense" else mode
    t0 = time.perf_counter()
    oracle.decode(qs, ks, vs, ss, S if om != "dense" else 0, om, seed=1)
    dt = time.perf_counter() - t0
    us_step = dt * 1e6 * (w.B / rows)
    return {"value": round(us_step, 1), "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{rows} of {w.B} batch rows ({rows * w.H_q} query heads x {w.n_max} keys), "
                      f"{dt:.2f} s wall, scaled x{w.B / rows:g} to one step"}


def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores (the pages ship no code)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    import oracle
    from stochastic_sparse_kv_gb300 import workloads
    w = workloads.BATCHED
    S = args.S
    # one batch row per step keeps the run within minutes; generate just those rows
    w1 = workloads.Workload(w.name, 1, w.H_q, w.H_kv, w.d, w.n_max, S, w.modes)
    q, k, v, sl = workloads.make_inputs(w1)
    for _ in range(args.warmup):
        oracle.decode(q, k, v, sl, S, args.mode if args.mode != "dense" else "dense", seed=0)
    ts = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        oracle.decode(q, k, v, sl, S if args.mode != "dense" else 0, args.mode, seed=i)
        ts.append(time.perf_counter() - t0)
    per_row = sum(ts) / len(ts)
    us_step = per_row * 1e6 * w.B
    sample = f"1 of {w.B} batch rows per step ({w.H_q} query heads x {w.n_max} keys), scaled x{w.B}"
    cores = oracle.num_threads()
    rec = {"metric": METRIC, "value": round(us_step, 1), "unit": UNIT, "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us_step / 1000, 3),
           "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "config": {"workload": w.name, "B": w.B, "H_q": w.H_q, "H_kv": w.H_kv, "d": w.d, "n_k": w.n_max,
                      "S": S, "mode": args.mode},
           "cpu_baseline": {"value": round(us_step, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(us_step, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(rec), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--mode", default="systematic", choices=["systematic", "stratified", "dense", "iid"])
    ap.add_argument("--S", type=int, default=256)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-rows", type=int, default=16)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the other modes and the S sweep")
    ap.add_argument("--workload", default="llama8b_b16_32k")
    ap.add_argument("--layers", type=int, default=32, help="depth of the multi-layer extra (0: skip it)")
    ap.add_argument("--no-workloads", action="store_true", help="skip timing the other configurations")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
