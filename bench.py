#!/usr/bin/env python
"""Decode steps/s and effective KV GB/s of the sparse KV-cache decode step on GB300.

Workload (default): Llama-3.1-8B-shaped attention, 32 layers, 32 q / 8 kv heads, d = 128, batch 8,
context 32768, block 16, budget 2048 tokens (128 blocks, 1 sink + 2 recent), cache cap 192 blocks
(1.5x budget), 4 lookahead draft queries per step (q_draft = q_{t+j} + N(0, 0.3^2)), full KV history
(32 GiB) in pinned host memory.  Seeded synthetic data (workload/), no dataset.

One step = every layer, in order, for every request: attention over the selection made by the
previous step, scoring with the drafts, selection, cache update, and the host -> slot fetch on a
side stream.  Each timed step is its own CUDA graph (its queries baked in).  Per-step reads
(about 3 GiB) exceed the 129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a bounded sample of the
same workload on the host cores.
"""
import argparse
import json
import os
import resource
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workload as W  # noqa: E402

METRIC = "sparse decode steps/s (effective KV GB/s and HBM/host-link roofline alongside)"
UNIT = "steps/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_32k_lookahead")
    ap.add_argument("--timed-kernel", default="attn", choices=["attn", "score", "fetch", "update", "topk"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--threads", type=int, default=0, help="generator threads (0: all cores)")
    return ap.parse_args()


def log(*a):
    print("[bench]", *a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------- distributed

class Dist:
    def __init__(self, n_gpus):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl" if self._has_cuda() else "gloo")
            self.pg = dist

    @staticmethod
    def _has_cuda():
        import torch
        return torch.cuda.is_available()

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device="cuda" if self._has_cuda() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- peaks

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j.get("hbm_gbs", 6800.0), "measured (MEASURED_PEAKS.json)"
    return 6800.0, "fallback (6.8 TB/s)"


def host_link_peak_gbs():
    """Host -> device copy of 1 GiB of pinned memory (copy engine), best of 3: the measured link."""
    import torch
    n = 1 << 30
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    h.fill_(1)
    d = torch.empty(n, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(4):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        d.copy_(h, non_blocking=True)
        b.record()
        b.synchronize()
        best = max(best, n / (a.elapsed_time(b) * 1e-3) / 1e9)
    del h, d
    return best


# ----------------------------------------------------------------------------- algorithmic bytes

def algorithmic_bytes(w, lens, link_bytes_per_step):
    """HBM bytes one step must move (per layer: index scan, attention reads of the selected
    K/V rows, queries, the slot writes of fetched rows) and host-link bytes."""
    rows_per_unit = []
    for L in lens:
        nb = (L + w.block_size - 1) // w.block_size
        k = min(w.budget_blocks, nb)
        rows_per_unit += [min(k * w.block_size, L)] * w.n_kv_head
    row_b = 2 * (w.d_k + (0 if w.v_shares_k else w.d_v))
    idx_b = sum(((L + w.block_size - 1) // w.block_size) * w.d_k * 2 for L in lens) * w.n_kv_head
    attn_b = sum(rows_per_unit) * row_b
    q_b = w.n_req * w.n_q_head * w.d_k * 2 * (1 + (w.n_draft if w.lookahead else 0))
    out_b = w.n_req * w.n_q_head * w.d_v * 4
    per_layer = {"index": idx_b, "attn": attn_b + w.n_req * w.n_q_head * w.d_k * 2 + out_b}
    hbm = w.n_layer * (idx_b + attn_b + q_b + out_b) + link_bytes_per_step   # fetched rows are written to HBM
    return hbm, link_bytes_per_step, per_layer


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample_time(w, steps_warm: int, steps_timed: int, n_layers: int):
    """Run the oracle on request 0 and the first n_layers layers; returns (seconds per timed
    step of the sample, units in the sample, cores used, description)."""
    from oracle import OracleDecoder
    ws = w.with_(n_req=1, n_layer=n_layers)
    k, v = W.kv_numpy(ws)
    dec = OracleDecoder(ws, k, v, [ws.ctx0])
    qs = W.QueryStream(ws)
    inputs = []
    for t in range(steps_warm + steps_timed):
        q = qs.queries(t)
        d = qs.drafts(t) if ws.lookahead else None
        tok = W.token(ws, ws.ctx0 + t) if ws.append else (None, None)
        inputs.append((q, d, tok))
    for t in range(steps_warm):
        q, d, (nk, nv) = inputs[t]
        dec.step(q, d, nk, nv)
    r0 = resource.getrusage(resource.RUSAGE_SELF)
    t0 = time.perf_counter()
    for t in range(steps_warm, steps_warm + steps_timed):
        q, d, (nk, nv) = inputs[t]
        dec.step(q, d, nk, nv)
    wall = time.perf_counter() - t0
    r1 = resource.getrusage(resource.RUSAGE_SELF)
    cpu = (r1.ru_utime - r0.ru_utime) + (r1.ru_stime - r0.ru_stime)
    cores = max(1, int(round(cpu / wall))) if wall > 0 else 1
    units = ws.n_req * ws.n_layer * ws.n_kv_head
    desc = (f"oracle (numpy, fp64) on request 0 of {w.n_req}, layers 0-{n_layers - 1} of {w.n_layer}, all "
            f"{w.n_kv_head} kv-heads ({units} of {w.n_req * w.n_layer * w.n_kv_head} units), {steps_timed} step(s) after "
            f"{steps_warm} warm-up; time scaled by units to the full step")
    return wall / steps_timed, units, cores, desc


def run_reference(args, dist):
    if dist.rank != 0:
        return 0
    w = W.WORKLOADS[args.workload]
    total_units = w.n_req * w.n_layer * w.n_kv_head
    n_layers = max(1, min(w.n_layer, 2))
    per_step, units, cores, desc = oracle_sample_time(w, max(1, args.warmup), max(1, args.steps), n_layers)
    full_step = per_step * total_units / units
    value = 1.0 / full_step
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": full_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_of(w):
    return {"workload": w.name, "batch": w.n_req, "layers": w.n_layer, "q_heads": w.n_q_head,
            "kv_heads": w.n_kv_head, "d_k": w.d_k, "d_v": w.d_v, "context": w.ctx0, "block": w.block_size,
            "budget_tokens": w.budget_blocks * w.block_size, "cache_blocks_per_head": w.cap_blocks,
            "lookahead_drafts": w.n_draft if w.lookahead else 0, "append": w.append,
            "layer_prefetch": w.layer_prefetch, "host_kv_gib": round(w.host_kv_bytes / 2**30, 2),
            "l2": "no flush: each step reads > 3 GiB, far above the 129 MB L2",
            "parallelism": "one replica per GPU (requests are independent)"}


# ----------------------------------------------------------------------------- our path

def run_ours(args, dist):
    import torch
    import sparse_kv_cache_decode_gb300 as K
    from sparse_kv_cache_decode_gb300 import build as kbuild

    kbuild.build()
    torch.cuda.set_device(dist.local)
    w = W.WORKLOADS[args.workload]
    if dist.world > 1:
        w = w.with_(seed=w.seed + dist.rank)       # each GPU serves its own batch of requests
    B, NL, Hkv = w.n_req, w.n_layer, w.n_kv_head
    T = args.warmup + args.steps
    T_e2e = 0 if args.no_e2e else args.steps
    t0 = time.time()
    k_host = torch.empty((NL, B, Hkv, w.max_ctx, w.d_k), dtype=torch.int16, pin_memory=True)
    v_host = None if w.v_shares_k else torch.empty((NL, B, Hkv, w.max_ctx, w.d_v), dtype=torch.int16,
                                                   pin_memory=True)
    W.fill_kv(w, k_host, v_host, args.threads)
    log(f"host KV {w.host_kv_bytes / 2**30:.1f} GiB generated in {time.time() - t0:.1f}s")

    ctx = K.Context(K.make_config(w))
    ctx.bind_host_kv(k_host, v_host)
    lens = [w.ctx0] * B
    ctx_len = torch.tensor(lens, dtype=torch.int32, device="cuda")
    index = torch.zeros((NL, B, Hkv, w.max_blocks, w.d_k), dtype=torch.int16, device="cuda")
    for l in range(NL):
        ctx.index_build(l, index, ctx_len)
    torch.cuda.synchronize()

    # per-step inputs (device copies for the device-resident timing, pinned copies for e2e)
    t0 = time.time()
    qs = W.QueryStream(w)
    nq = w.n_score_q
    q_all = torch.empty((T + T_e2e, NL, B, w.n_q_head, w.d_k), dtype=torch.int16)
    d_all = torch.empty((T + T_e2e, NL, B, w.n_draft, w.n_q_head, w.d_k), dtype=torch.int16) if w.lookahead else None
    tok_all = []
    for t in range(T + T_e2e):
        q_all[t] = torch.from_numpy(qs.queries(t).view(np.int16))
        if d_all is not None:
            d_all[t] = torch.from_numpy(qs.drafts(t).view(np.int16))
        if w.append:
            nk, nv = W.token(w, w.ctx0 + t)
            tok_all.append((torch.from_numpy(nk.view(np.int16)),
                            None if nv is None else torch.from_numpy(nv.view(np.int16))))
    log(f"queries for {T + T_e2e} steps generated in {time.time() - t0:.1f}s")
    q_dev = q_all[:T].cuda()
    d_dev = d_all[:T].cuda() if d_all is not None else None
    tok_dev = [(a.cuda(), None if b is None else b.cuda()) for a, b in tok_all[:T]]

    out = torch.zeros((NL, B, w.n_q_head, w.d_v), dtype=torch.float32, device="cuda")
    sel = torch.zeros((NL, B, Hkv, w.budget_blocks), dtype=torch.int32, device="cuda")
    nsel = torch.zeros((NL, B, Hkv), dtype=torch.int32, device="cuda")
    stats = torch.zeros((NL, 7), dtype=torch.int64, device="cuda")
    s = torch.cuda.Stream()
    cs = torch.cuda.Stream()

    def step(qt, dt, tok):
        if w.append:
            ctx.advance_ctx(ctx_len)
        for l in range(NL):
            if w.layer_prefetch and l > 0:
                ctx.layer_prefetch(l, sel[l - 1], nsel[l - 1], ctx_len, stats, stream=cs)
            ctx.decode_step(l, qt[l], None if dt is None else dt[l], nq if dt is not None else 1, index, ctx_len,
                            out[l], stats, None if tok is None else tok[0][l],
                            None if tok is None or tok[1] is None else tok[1][l], sel[l], nsel[l], stream=s,
                            copy_stream=cs)
        ctx.join(s)

    # step 0 eagerly (bootstraps lookahead selections), then one graph per remaining step
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        step(q_dev[0], None if d_dev is None else d_dev[0], tok_dev[0] if w.append else None)
    s.synchronize()
    graphs = {}

    def capture(t, qt, dt, tok):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step(qt, dt, tok)
        return g

    for t in range(1, args.warmup):
        graphs[t] = capture(t, q_dev[t], None if d_dev is None else d_dev[t], tok_dev[t] if w.append else None)
    n_timed_kernel_per_step = {"attn": NL, "score": NL, "fetch": NL + (NL - 1 if w.layer_prefetch else 0),
                               "update": NL, "topk": NL}[args.timed_kernel]
    ctx.kernel_timer_arm(args.timed_kernel, args.steps * n_timed_kernel_per_step)
    launches0 = ctx.launch_count()
    for t in range(args.warmup, T):
        graphs[t] = capture(t, q_dev[t], None if d_dev is None else d_dev[t], tok_dev[t] if w.append else None)
    launches = ctx.launch_count() - launches0
    with torch.cuda.stream(s):
        for t in range(1, args.warmup):
            graphs[t].replay()
    torch.cuda.synchronize()
    stats0 = stats.cpu().numpy().copy()

    hbm_peak, hbm_src = measured_peaks()
    link_peak = host_link_peak_gbs()
    clocks = ClockSampler(dist.local)
    clocks.start()
    time.sleep(0.3)
    dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        ev0.record(s)
        for t in range(args.warmup, T):
            graphs[t].replay()
        ev1.record(s)
    torch.cuda.synchronize()
    dist.barrier()
    elapsed = ev0.elapsed_time(ev1) * 1e-3
    clk = clocks.stop()
    elapsed = dist.max(elapsed)
    stats1 = stats.cpu().numpy()
    dstat = (stats1 - stats0).sum(axis=0)
    kernel_ms, kernel_n = ctx.kernel_timer_read()
    dev_status = ctx.poll_error()
    if dev_status != 0:
        raise RuntimeError(f"device status {K.STATUS.get(dev_status, dev_status)}")

    ms_per_step = elapsed / args.steps * 1e3
    value = dist.world * args.steps / elapsed
    link_per_step = float(dstat[6]) / args.steps
    hbm_step, link_step, per_layer = algorithmic_bytes(w, lens, link_per_step)
    t_step = elapsed / args.steps
    step_roof = max(hbm_step / (hbm_peak * 1e9), link_step / (link_peak * 1e9))
    kv_gbs = hbm_step / t_step / 1e9
    misses, hits = float(dstat[1]), float(dstat[0])

    # dominant-kernel roofline: algorithmic bytes per launch / live CUDA-event duration
    per_launch_ms = kernel_ms / max(1, kernel_n)
    if args.timed_kernel == "attn":
        alg = per_layer["attn"]
    elif args.timed_kernel == "score":
        alg = per_layer["index"] + w.n_req * nq * w.n_q_head * w.d_k * 2
    elif args.timed_kernel == "fetch":
        alg = link_per_step / max(1, n_timed_kernel_per_step)
    else:
        alg = 0
    achieved = alg / (per_launch_ms * 1e-3) / 1e9 if per_launch_ms > 0 else 0.0
    bound_peak = link_peak if args.timed_kernel == "fetch" else hbm_peak
    roofline = {"bound": "hbm" if args.timed_kernel != "fetch" else "host-link", "kernel": args.timed_kernel,
                "achieved": round(achieved, 1), "peak": round(bound_peak, 1), "unit": "GB/s",
                "frac": round(achieved / bound_peak, 4), "traffic": None,
                "bytes_per_launch": alg, "avg_launch_ms": round(per_launch_ms, 5), "launches_timed": kernel_n,
                "peak_source": hbm_src if args.timed_kernel != "fetch" else "measured in this run (H2D copy)"}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, ctx, ctx_len, index, out, sel, nsel, stats, s, cs, q_all, d_all, tok_all, T,
                      step, dist)

    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(w),
            "effective_kv_gbs": round(kv_gbs, 1),
            "step_roofline": {"hbm_bytes": hbm_step, "link_bytes": link_step, "hbm_peak_gbs": hbm_peak,
                              "link_peak_gbs": round(link_peak, 1), "bound_ms": round(step_roof * 1e3, 4),
                              "frac": round(step_roof / t_step, 4),
                              "bound": "host-link" if link_step / link_peak > hbm_step / hbm_peak else "hbm"},
            "miss_fraction": round(misses / max(1.0, misses + hits), 4),
            "roofline": roofline, "clocks": clk, "gpu_launches": int(launches)}
    if e2e:
        line["e2e"] = e2e
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        per_step, units, cores, desc = oracle_sample_time(w, 1, 3, min(w.n_layer, 8))
        full = per_step * (w.n_req * w.n_layer * w.n_kv_head) / units
        line["cpu_baseline"] = {"value": round(1.0 / full, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc}
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    ctx.close()
    return 0


def run_e2e(args, w, ctx, ctx_len, index, out, sel, nsel, stats, s, cs, q_all, d_all, tok_all, T, step, dist):
    """The same steps through the public API with host buffers: each step copies its queries
    (and drafts) from pinned host memory into fixed device buffers, runs the step graph, and
    copies the attention output back to pinned host memory."""
    import torch
    K_steps = args.steps
    q_pin = q_all[T:T + K_steps].pin_memory()
    d_pin = d_all[T:T + K_steps].pin_memory() if d_all is not None else None
    q_fix = torch.empty_like(q_all[0], device="cuda")
    d_fix = torch.empty_like(d_all[0], device="cuda") if d_all is not None else None
    tok_fix = None
    tok_pin = []
    if w.append:
        tok_pin = [(a.pin_memory(), None if b is None else b.pin_memory()) for a, b in tok_all[T:T + K_steps]]
        tok_fix = (torch.empty_like(tok_all[0][0], device="cuda"),
                   None if tok_all[0][1] is None else torch.empty_like(tok_all[0][1], device="cuda"))
    out_pin = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(q_fix, d_fix, tok_fix)
    torch.cuda.synchronize()
    h2d = q_fix.numel() * 2 + (d_fix.numel() * 2 if d_fix is not None else 0)
    if tok_fix is not None:
        h2d += tok_fix[0].numel() * 2 + (tok_fix[1].numel() * 2 if tok_fix[1] is not None else 0)
    d2h = out.numel() * 4
    dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    with torch.cuda.stream(s):
        for i in range(K_steps):
            q_fix.copy_(q_pin[i], non_blocking=True)
            if d_fix is not None:
                d_fix.copy_(d_pin[i], non_blocking=True)
            if tok_fix is not None:
                tok_fix[0].copy_(tok_pin[i][0], non_blocking=True)
                if tok_fix[1] is not None:
                    tok_fix[1].copy_(tok_pin[i][1], non_blocking=True)
            g.replay()
            out_pin.copy_(out, non_blocking=True)
    e1.record(s)
    torch.cuda.synchronize()
    el = dist.max(e0.elapsed_time(e1) * 1e-3)
    return {"value": round(dist.world * K_steps / el, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h)}


def main():
    args = parse()
    dist = Dist(args.gpus)
    try:
        if args.impl == "reference":
            return run_reference(args, dist)
        return run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    sys.exit(main())
