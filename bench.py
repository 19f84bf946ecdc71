#!/usr/bin/env python
"""Decode steps/s and effective KV GB/s of the sparse KV-cache decode step on GB300.

Workload (default): Llama-3.1-8B-shaped attention, 32 layers, 32 q / 8 kv heads, d = 128, batch 8,
context 32768, block 16, budget 2048 tokens (128 blocks, 1 sink + 2 recent), cache cap 192 blocks
(1.5x budget), 4 lookahead draft queries per step (q_draft = q_{t+j} + N(0, 0.3^2) noise), full KV
history (32 GiB) in pinned host memory.  Seeded synthetic data (workload/), no dataset.

One step = every layer, in order, for every request: attention over the selection made by the
previous step, scoring with the drafts, selection, cache update, and the host -> slot fetch on a
side stream.  The step is captured once as a CUDA graph over fixed input buffers; every timed
step copies its own device-resident inputs into them and replays the graph.  Per-step reads
(about 3 GiB) exceed the 129 MB L2, so no flush is needed between steps.

The default run also measures the other workloads, each in a child process of its own (its
history is freed when it ends): the 128K host-resident case with a per-step append, the MLA
token-level case with cross-layer prefetch, and a reduced budget/eviction sweep (one process,
one shared history); their lines go under `per_config`.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload NAME]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a bounded sample of the
same workload on the host cores.
"""
import argparse
import hashlib
import json
import os
import re
import resource
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# The step runs on several streams (compute, copy, selection) and as a CUDA graph whose branches
# run concurrently; all of them map onto the context's hardware work queues, 8 by default.  More
# queues keep the copy-stream fetch from sharing one with the compute stream (where it would wait
# behind the layer kernels).  Read when CUDA initialises, so it is set before torch touches it;
# children inherit it.
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")

import numpy as np  # noqa: E402

import workload as W  # noqa: E402

METRIC = "sparse decode steps/s (effective KV GB/s and HBM/host-link roofline alongside)"
UNIT = "steps/s"

# Workloads measured beside the headline by the default run (child processes).
PER_CONFIG = ["llama8b_128k_append", "mla_128k_token_topk", "llama8b_32k_lookahead_fp8"]
# Reduced budget/eviction sweep: block size x budget tokens x target step overlap (%).
SWEEP_POINTS = [f"sweep_bs{bs}_b{b}_ov{ov}" for bs in (16, 64) for b in (512, 2048, 4096) for ov in (50, 80, 95)]


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_32k_lookahead",
                    help="a named workload, or 'sweep' (with --sweep-points) for several sweep cases on one history")
    ap.add_argument("--sweep-points", default=",".join(SWEEP_POINTS))
    ap.add_argument("--timed-kernel", default="auto", choices=["auto", "attn", "score", "fetch"],
                    help="kernel of the roofline object (auto: the one with the most time per step)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="measure the selected workload only")
    ap.add_argument("--child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--threads", type=int, default=0, help="generator threads (0: all cores)")
    ap.add_argument("--serial", action="store_true", help="fetch on the compute stream (kernels run one at a time)")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (smaller profiling cases)")
    ap.add_argument("--batch", type=int, default=0, help="override the request count (smaller profiling cases)")
    ap.add_argument("--no-io", action="store_true",
                    help="control run: every step replays the first step's inputs, so the selection repeats, every "
                         "selected block is resident and the timed steps fetch nothing over the host link")
    ap.add_argument("--numa-local", action="store_true",
                    help="give the host history an explicit memory policy (preferred node = the local CPU node), "
                         "which keeps automatic NUMA balancing off it")
    ap.add_argument("--link-peak-only", action="store_true",
                    help="measure the host link (copy engine and SM zero-copy reads) on the workload's history and "
                         "print the figures")
    return ap.parse_args(argv)


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

def upload_graphs(graphs, stream):
    """Upload every instantiated graph before timing, so no first launch pays for it."""
    import ctypes
    import torch
    cands = [os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", n)
             for n in ("libcudart.so.13", "libcudart.so")]
    rt = None
    for c in cands:
        if os.path.exists(c):
            rt = ctypes.CDLL(c)
            break
    if rt is None or not all(hasattr(g, "raw_cuda_graph_exec") for g in graphs):
        return False
    rt.cudaGraphUpload.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    for g in graphs:
        rc = rt.cudaGraphUpload(ctypes.c_void_p(g.raw_cuda_graph_exec()), ctypes.c_void_p(stream.cuda_stream))
        if rc != 0:
            raise RuntimeError(f"cudaGraphUpload failed ({rc})")
    torch.cuda.synchronize()
    return True


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j.get("hbm_gbs", 6800.0), "measured (MEASURED_PEAKS.json)"
    return 6800.0, "fallback (6.8 TB/s)"


def _time_ms(fn, reps=3):
    import torch
    best = None
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    return best


def burst_fit(bursts):
    """Least-squares line through (bytes, microseconds) points of host-link bursts: time = fixed
    cost + bytes / streaming rate.  Returns (fixed cost in us, streaming rate in GB/s)."""
    x = np.array([b for b, _ in bursts], dtype=np.float64)
    y = np.array([t for _, t in bursts], dtype=np.float64)
    slope, icpt = np.polyfit(x, y, 1)
    return float(icpt), float(1e-3 / slope)


def link_peaks(K, host_tensors):
    """The host link measured three ways; the largest is the link peak of the step roofline.
      ce_pinned   copy engine, 1 GiB of cudaHostAlloc memory -> device
      ce_history  copy engine, 1 GiB of the bound history (the memory the fetch reads) -> device
      sm_seq      SM zero-copy reads of consecutive 8 KiB items of that 1 GiB (kvs_probe_host_read)
      sm_rand     SM zero-copy reads of 8 KiB items at random 8 KiB-aligned places in the whole history
    The SM probes take the best of a few grid shapes."""
    import torch
    n = 1 << 30
    out = {}
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    h.fill_(1)
    d = torch.empty(n, dtype=torch.uint8, device="cuda")
    out["ce_pinned"] = n / (_time_ms(lambda: d.copy_(h, non_blocking=True)) * 1e-3) / 1e9
    del h
    hist = host_tensors[0]
    flat = hist.view(-1).view(torch.uint8)
    region = flat.numel()
    if region >= n:
        src = flat[:n]
        out["ce_history"] = n / (_time_ms(lambda: d.copy_(src, non_blocking=True)) * 1e-3) / 1e9
    del d
    item = 8192
    sink = torch.zeros(2, dtype=torch.int32, device="cuda")
    seq = torch.arange(0, min(n, region) // item, dtype=torch.int64, device="cuda") * item
    rng = np.random.default_rng(12345)
    rnd = torch.from_numpy(rng.integers(0, region // item, size=65536, dtype=np.int64) * item).cuda()
    for name, offs in (("sm_seq", seq), ("sm_rand", rnd)):
        best, shape = 0.0, None
        for ctas, threads in ((152, 256), (304, 256), (608, 128), (1216, 128)):
            ms = _time_ms(lambda: K.probe_host_read(hist, region, offs, item, ctas, threads, sink))
            gbs = offs.numel() * item / (ms * 1e-3) / 1e9
            if gbs > best:
                best, shape = gbs, f"{ctas}x{threads}"
        out[name] = best
        out[name + "_grid"] = shape
    # bursts of the size a layer's fetch moves: time = fixed latency + bytes / streaming rate
    bursts = []
    for nit in (278, 490, 2000, 65536):
        offs = rnd[:nit] if nit <= rnd.numel() else rnd
        ms = _time_ms(lambda: K.probe_host_read(hist, region, offs, item, 152, 128, sink))
        bursts.append((offs.numel() * item, ms * 1e3))
    fixed_us, stream_gbs = burst_fit(bursts)
    out["bursts"] = [{"mb": round(b / 1e6, 2), "us": round(t, 1), "gbs": round(b / (t * 1e-6) / 1e9, 1)} for b, t in bursts]
    out["burst_fixed_us"] = round(fixed_us, 1)
    out["burst_stream_gbs"] = round(stream_gbs, 1)
    torch.cuda.synchronize()
    if int(sink[1].item()) != 0:
        raise RuntimeError("link probe skipped items")
    vals = {k: v for k, v in out.items() if k in ("ce_pinned", "ce_history", "sm_seq", "sm_rand")}
    best_key = max(vals, key=vals.get)
    res = {k: (round(v, 1) if isinstance(v, float) else v) for k, v in out.items()}
    res["peak_gbs"] = round(vals[best_key], 1)
    res["peak_source"] = f"{best_key} (largest of the measurements in this run; profiles/host_link_peak.md)"
    res["history_bytes"] = int(region)
    return res


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        fields = dict(ln.split(":", 1) for ln in out.splitlines() if ":" in ln)
        name = fields.get("Model name", "").strip()
        vendor = fields.get("Vendor ID", "").strip()
        arch = fields.get("Architecture", "").strip()
        return " ".join(x for x in (vendor, name, f"({arch})" if arch else "") if x) or "unknown"
    except (OSError, subprocess.SubprocessError, ValueError):
        return "unknown"


# ----------------------------------------------------------------------------- algorithmic bytes

def algorithmic_bytes(w, lens, link_bytes_per_step):
    """HBM bytes one step must move (per layer: index scan, attention reads of the selected
    K/V rows, queries, the slot writes of fetched rows) and host-link bytes."""
    rows_per_unit = []
    for L in lens:
        nb = (L + w.block_size - 1) // w.block_size
        k = min(w.budget_blocks, nb)
        rows_per_unit += [min(k * w.block_size, L)] * w.n_kv_head
    row_b = w.elt_bytes * (w.d_k + (0 if w.v_shares_k else w.d_v))          # bf16 or E4M3 rows
    idx_b = sum(((L + w.block_size - 1) // w.block_size) * w.d_idx * 2 for L in lens) * w.n_kv_head
    attn_b = sum(rows_per_unit) * row_b
    q_b = w.n_req * w.n_q_head * w.d_k * 2 * (1 + (w.n_draft if w.lookahead else 0))
    out_b = w.n_req * w.n_q_head * w.d_v * 4
    per_layer = {"index": idx_b, "attn": attn_b + w.n_req * w.n_q_head * w.d_k * 2 + out_b}
    hbm = w.n_layer * (idx_b + attn_b + q_b + out_b) + link_bytes_per_step   # fetched rows are written to HBM
    return hbm, link_bytes_per_step, per_layer


def dependency_bound_ms(w, per_layer, link_per_layer, hbm_peak, link_peak):
    """Sync-mode bound under the layer dependency: per layer the index scan, then the larger of
    the attention reads and the layer's own fetch, summed over layers (ms)."""
    t = 0.0
    for lb in link_per_layer:
        t_ik = per_layer["index"] / (hbm_peak * 1e9)
        t_attn = per_layer["attn"] / (hbm_peak * 1e9)
        t_fetch = lb / (link_peak * 1e9)
        t += t_ik + max(t_attn, t_fetch)
    return t * 1e3


# ----------------------------------------------------------------------------- ncu traffic

# the sources that define each timed kernel ("attn": the TMA-fed GQA attention kernel that the
# committed traffic figures were taken from)
KERNEL_SOURCES = {"attn": ["k_attn_tma.cu", "kvs_attn_tma.cuh"],
                  "score": ["k_score.cu", "kvs_score.cuh", "k_score_tc.cu"],
                  "fetch": ["k_cache.cu"]}


def source_sha(kname) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kname, []):
        with open(os.path.join(ROOT, "sparse_kv_cache_decode_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic(kname, workload):
    """DRAM bytes (read + write) per launch of a kernel on a workload, from a committed ncu summary
    under profiles/ that records them for the current kernel source (a `traffic` block naming the
    kernel, the workload, the sources' sha256 prefix and the bytes per full launch); None when no
    summary matches or the kernel changed since the counters were taken."""
    pdir = os.path.join(ROOT, "profiles")
    want = source_sha(kname)
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".md"):
            continue
        with open(os.path.join(pdir, f)) as fh:
            text = fh.read()
        for block in re.findall(r"```traffic\n(.*?)```", text, flags=re.S):
            kv = dict(ln.split(":", 1) for ln in block.strip().splitlines() if ":" in ln)
            kv = {k.strip(): v.strip() for k, v in kv.items()}
            if kv.get("kernel") == kname and kv.get("workload") == workload and kv.get("source_sha") == want:
                return {"bytes": int(kv["dram_bytes_per_launch"]), "profile": f"profiles/{f}",
                        "note": kv.get("note", "")}
    return None


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
    coverage = dense_softmax_coverage(ws, dec, inputs[-1][0])
    return wall / steps_timed, units, cores, desc, coverage


def dense_softmax_coverage(ws, dec, q):
    """Share of the exact dense softmax mass (over every present token, fp64) that falls on the
    tokens the step attended to, for the last oracle step: mean over the q heads of layer 0 of
    request 0 (outside any timed region)."""
    from oracle import bf16_to_f64
    g, bs = ws.group, ws.block_size
    shares = []
    for h in range(ws.n_kv_head):
        u = (0, 0, h)
        L = dec.L[0]
        k = bf16_to_f64(dec.k[u][:L])
        qh = bf16_to_f64(q[0, 0, h * g:(h + 1) * g])
        logits = float(ws.softmax_scale) * (qh @ k.T)
        p = np.exp(logits - logits.max(axis=1, keepdims=True))
        attended = np.zeros(L, bool)
        for b in dec.records[u].attn_sel:
            attended[b * bs:min(L, (b + 1) * bs)] = True
        shares += list(p[:, attended].sum(axis=1) / p.sum(axis=1))
    return {"value": round(float(np.mean(shares)), 4), "min": round(float(np.min(shares)), 4),
            "sample": f"oracle, last step of the CPU-baseline sample, layer 0 of request 0, {len(shares)} q heads"}


def coverage_study(w, q):
    """Dense-softmax coverage of the selection each block-scoring rule makes, on request 0, layer 0,
    every kv head, with the step's current query (oracle, fp64; outside any timed region): the share
    of the exact attention mass over all present tokens that the selected tokens carry, mean and
    minimum over the q heads.  Rules: the block-mean key ("mean"), the [max | min] upper bound
    ("bound"), and two references that need every key: the block's largest token logit
    ("token_max") and the block's exact softmax mass ("mass", the best any block selection can do)."""
    from oracle import bf16_to_f64, block_scores, block_scores_bound, index_keys, index_minmax, select_blocks
    ws = w.with_(n_req=1, n_layer=1)
    k, _ = W.kv_numpy(ws)
    g, bs, L = ws.group, ws.block_size, ws.ctx0
    nb = (L + bs - 1) // bs
    cov = {m: [] for m in ("mean", "bound", "token_max", "mass")}
    for h in range(ws.n_kv_head):
        kr = k[0, 0, h, :L]
        rows = q[0, 0, h * g:(h + 1) * g]
        logits = float(ws.softmax_scale) * (bf16_to_f64(rows) @ bf16_to_f64(kr).T)      # (G, L)
        p = np.exp(logits - logits.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        pad = nb * bs - L
        lp = np.pad(logits, ((0, 0), (0, pad)), constant_values=-np.inf).reshape(g, nb, bs)
        mass = np.pad(p, ((0, 0), (0, pad))).reshape(g, nb, bs).sum(axis=2)
        scores = {"mean": block_scores(rows, index_keys(kr, L, bs), ws.softmax_scale)[0],
                  "bound": block_scores_bound(rows, index_minmax(kr, L, bs), ws.softmax_scale)[0],
                  "token_max": lp.max(axis=2).max(axis=0),
                  "mass": mass.max(axis=0)}
        for m, sc in scores.items():
            sel = select_blocks(sc.astype(np.float32), nb, ws.budget_blocks, ws.n_sink, ws.n_recent)
            taken = np.zeros(nb, bool)
            taken[sel] = True
            cov[m] += list(mass[:, taken].sum(axis=1))
    return {m: {"value": round(float(np.mean(v)), 4), "min": round(float(np.min(v)), 4)} for m, v in cov.items()} | {
        "sample": f"oracle, request 0, layer 0, {ws.n_kv_head} kv heads x {g} q heads, the step's own query scoring, "
                  f"budget {ws.budget_blocks} blocks of {bs}"}


def run_reference(args, dist):
    if dist.rank != 0:
        return 0
    w = W.get(args.workload)
    total_units = w.n_req * w.n_layer * w.n_kv_head
    n_layers = max(1, min(w.n_layer, 2))
    per_step, units, cores, desc, coverage = oracle_sample_time(w, max(1, args.warmup), max(1, args.steps), n_layers)
    full_step = per_step * total_units / units
    value = 1.0 / full_step
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": full_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "cpu": cpu_model(), "kind": "oracle",
                             "sample": desc},
            "dense_softmax_coverage": coverage,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_of(w):
    return {"workload": w.name, "batch": w.n_req, "layers": w.n_layer, "q_heads": w.n_q_head,
            "kv_heads": w.n_kv_head, "d_k": w.d_k, "d_v": w.d_v, "context": w.ctx0, "block": w.block_size,
            "budget_tokens": w.budget_blocks * w.block_size, "cache_blocks_per_head": w.cap_blocks,
            "lookahead_drafts": w.n_draft if w.lookahead else 0, "append": w.append,
            "layer_prefetch": w.layer_prefetch, "rho": w.rho, "draft_rho": w.draft_rho,
            "host_kv_gib": round(w.host_kv_bytes / 2**30, 2),
            "l2": "no flush: each step reads > 1 GiB, far above the 129 MB L2",
            "parallelism": "one replica per GPU (requests are independent)"}


def prefetch_report(w, dstat, steps: int):
    """Cross-layer prefetch per step from the device counters (hits, misses, evictions, prefetched,
    prefetch hits, pin fallbacks, bytes fetched): blocks prefetched, how many of them the layer's own
    selection then used, and the miss bytes that use hid from the step's critical path."""
    if not w.layer_prefetch or steps <= 0:
        return None
    prefetched, used = float(dstat[3]) / steps, float(dstat[4]) / steps
    block_bytes = w.block_size * (w.d_k + (0 if w.v_shares_k else w.d_v)) * w.elt_bytes
    return {"blocks_per_step": round(prefetched, 1), "used_per_step": round(used, 1),
            "used_fraction": round(used / prefetched, 4) if prefetched else None,
            "hidden_miss_bytes_per_step": int(used * block_bytes)}


def check_host_memory(history_bytes: int):
    """Refuse to start when the host cannot hold every local rank's page-locked history (with 10%
    slack): page-locking more than the host has would end in the OOM killer, not in an error."""
    ranks = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    try:
        with open("/proc/meminfo") as f:
            avail = next(int(ln.split()[1]) * 1024 for ln in f if ln.startswith("MemAvailable:"))
    except (OSError, StopIteration):
        return
    need = int(history_bytes * 1.1) * ranks
    if need > avail:
        raise RuntimeError(f"host memory: {ranks} rank(s) x {history_bytes / 2**30:.1f} GiB of history need "
                           f"{need / 2**30:.1f} GiB, {avail / 2**30:.1f} GiB available")


def selection_overlap(prev_sel, prev_n, sel, n):
    """Mean over units of |S_t & S_t-1| / |S_t| (host arrays [..., K_b] and counts [...])."""
    a = prev_sel.reshape(-1, prev_sel.shape[-1])
    b = sel.reshape(-1, sel.shape[-1])
    na, nb = prev_n.reshape(-1), n.reshape(-1)
    vals = []
    for i in range(b.shape[0]):
        if nb[i] <= 0:
            continue
        vals.append(len(np.intersect1d(a[i, :na[i]], b[i, :nb[i]])) / nb[i])
    return vals


# ----------------------------------------------------------------------------- our path

class History:
    """The page-locked host history of a workload (huge pages when the kernel gives them)."""

    def __init__(self, K, w, threads, numa_local=False):
        import torch
        NL, B, Hkv = w.n_layer, w.n_req, w.n_kv_head
        check_host_memory(w.host_kv_bytes)
        t0 = time.time()
        self.K = K
        self.vm0 = K.numa_vmstat()
        if w.kv_dtype == "fp8":
            # generate bf16, quantise to E4M3 through the GPU into the history that is then bound
            kb = K.HostArray((NL, B, Hkv, w.max_ctx, w.d_k))
            vb = K.HostArray((NL, B, Hkv, w.max_ctx, w.d_v))
            W.fill_kv(w, kb.tensor, vb.tensor, threads)
            k8 = K.HostArray((NL, B, Hkv, w.max_ctx, w.d_k), dtype=torch.uint8, local_node=numa_local)
            v8 = K.HostArray((NL, B, Hkv, w.max_ctx, w.d_v), dtype=torch.uint8, local_node=numa_local)
            K.quantize_history_e4m3(kb.tensor, k8.tensor, w.k_scale)
            K.quantize_history_e4m3(vb.tensor, v8.tensor, w.v_scale)
            kb.close()
            vb.close()
            del kb, vb
            frac = min(k8.huge_fraction(), v8.huge_fraction())
            k8.register()
            v8.register()
            self.k, self.v, self.k_keep, self.v_keep = k8.tensor, v8.tensor, k8, v8
            self.desc = f"E4M3 codes (scales {w.k_scale:g} / {w.v_scale:g}); mmap + huge pages ({frac:.0%}) + cudaHostRegister"
        elif w.v_shares_k:
            self.k, self.k_keep, self.desc = K.pinned_host_history((NL, B, Hkv, w.max_ctx, w.d_k),
                                                                   lambda t: W.fill_kv(w, t, None, threads),
                                                                   local_node=numa_local)
            self.v, self.v_keep = None, None
        else:
            k_arr = K.HostArray((NL, B, Hkv, w.max_ctx, w.d_k), local_node=numa_local)
            v_arr = K.HostArray((NL, B, Hkv, w.max_ctx, w.d_v), local_node=numa_local)
            W.fill_kv(w, k_arr.tensor, v_arr.tensor, threads)
            fk, fv = k_arr.huge_fraction(), v_arr.huge_fraction()
            if min(fk, fv) >= 0.95:
                k_arr.register()
                v_arr.register()
                self.k, self.v, self.k_keep, self.v_keep = k_arr.tensor, v_arr.tensor, k_arr, v_arr
                self.desc = f"mmap + transparent huge pages ({min(fk, fv):.0%}) + cudaHostRegister"
            else:
                self.k = torch.empty(k_arr.tensor.shape, dtype=torch.int16, pin_memory=True)
                self.v = torch.empty(v_arr.tensor.shape, dtype=torch.int16, pin_memory=True)
                self.k.copy_(k_arr.tensor)
                self.v.copy_(v_arr.tensor)
                del k_arr, v_arr
                self.k_keep = self.v_keep = None
                self.desc = f"cudaHostAlloc (huge pages covered only {min(fk, fv):.0%})"
        if numa_local:
            node = getattr(self.k_keep, "node", None)
            self.desc += f"; preferred NUMA node {node}" if node is not None else "; NUMA policy not set"
        log(f"host memory: {self.desc}; {w.host_kv_bytes / 2**30:.1f} GiB generated in {time.time() - t0:.1f}s")

    def vmstat_delta(self):
        now = self.K.numa_vmstat()
        return {k: now[k] - self.vm0.get(k, 0) for k in now if now[k] != self.vm0.get(k, 0)}

    def huge_arrays(self):
        return [a for a in (self.k_keep, self.v_keep) if isinstance(a, self.K.HostArray)]

    def repair_after_first_step(self, ctx):
        """On some hosts the first scattered device reads of the mapped history split part of its
        transparent huge pages; the device then translates 64 KiB pages on every later fetch into
        them, and fetches slow down many times over.  Collapse the pages again (or, failing that,
        move the history to driver-pinned memory) and bind again, before any graph captures the
        host pointers."""
        import torch
        arrays = self.huge_arrays()
        if not arrays:
            return
        left = min(a.huge_fraction() for a in arrays)
        log(f"host memory after the first step: huge {left:.2%}; vmstat since allocation {self.vmstat_delta()}")
        if left >= 0.999:
            return
        again = min(a.recollapse() for a in arrays)
        log(f"host memory: the first step split huge pages ({left:.1%} left); collapsed again: {again:.1%}")
        if again >= 0.999:
            ctx.bind_host_kv(self.k, self.v)
            self.desc += f" (huge pages split by the first step, {left:.0%} left, collapsed again)"
            return
        k_new = torch.empty(self.k.shape, dtype=self.k.dtype, pin_memory=True)
        k_new.copy_(self.k)
        v_new = None
        if self.v is not None:
            v_new = torch.empty(self.v.shape, dtype=self.v.dtype, pin_memory=True)
            v_new.copy_(self.v)
        ctx.bind_host_kv(k_new, v_new)
        for a in arrays:
            a.close()
        self.k, self.v, self.k_keep, self.v_keep = k_new, v_new, None, None
        self.desc = f"cudaHostAlloc (the first step split huge pages of the mapped history: {again:.0%} left)"
        log(f"host memory: {self.desc}")

    def huge_after(self):
        arrays = self.huge_arrays()
        return [round(a.huge_fraction(), 4) for a in arrays] if arrays else None

    def close(self):
        for a in self.huge_arrays():
            a.close()
        self.k = self.v = self.k_keep = self.v_keep = None


class LinkPeak:
    """The link peak of a history, measured once, when first asked for (after a timed region, so
    that the probe's scattered reads of the history never precede one)."""

    def __init__(self, K, hist):
        self.K, self.hist, self.v = K, hist, None

    def get(self):
        if self.v is None:
            self.v = link_peaks(self.K, [self.hist.k])
        return self.v


def run_point(args, dist, w, hist, link, e2e: bool, cpu_baseline: bool):
    """Measure one workload on a bound history; returns its JSON line (a dict)."""
    import torch
    K = hist.K
    B, NL, Hkv = w.n_req, w.n_layer, w.n_kv_head
    T = args.warmup + args.steps
    T_e2e = args.steps if e2e else 0
    ctx = K.Context(K.make_config(w))
    ctx.bind_host_kv(hist.k, hist.v)
    lens = [w.ctx0] * B
    ctx_len = torch.tensor(lens, dtype=torch.int32, device="cuda")
    index = torch.zeros((NL, B, Hkv, w.max_blocks, w.d_idx), dtype=torch.int16, device="cuda")
    for l in range(NL):
        ctx.index_build(l, index, ctx_len)
    torch.cuda.synchronize()

    # per-step inputs (device copies for the device-resident timing, pinned copies for e2e)
    t0 = time.time()
    qs = W.QueryStream(w)
    nq = w.n_score_q
    n_meas = max(2, min(args.steps, 8))
    T_all = T + n_meas + T_e2e
    q_all = torch.empty((T_all, NL, B, w.n_q_head, w.d_k), dtype=torch.int16)
    d_all = torch.empty((T_all, NL, B, w.n_draft, w.n_q_head, w.d_k), dtype=torch.int16) if w.lookahead else None
    tok_all = []
    for t in range(T_all):
        q_all[t] = torch.from_numpy(qs.queries(t).view(np.int16))
        if d_all is not None:
            d_all[t] = torch.from_numpy(qs.drafts(t).view(np.int16))
        if w.append:
            nk, nv = W.token(w, w.ctx0 + t)
            tok_all.append((torch.from_numpy(nk.view(np.int16)),
                            None if nv is None else torch.from_numpy(nv.view(np.int16))))
    log(f"{w.name}: queries for {T_all} steps generated in {time.time() - t0:.1f}s")
    T_dev = T + n_meas
    q_dev = q_all[:T_dev].cuda()
    d_dev = d_all[:T_dev].cuda() if d_all is not None else None
    tok_dev = [(a.cuda(), None if b is None else b.cuda()) for a, b in tok_all[:T_dev]]

    out = torch.zeros((NL, B, w.n_q_head, w.d_v), dtype=torch.float32, device="cuda")
    sel = torch.zeros((NL, B, Hkv, w.budget_blocks), dtype=torch.int32, device="cuda")
    nsel = torch.zeros((NL, B, Hkv), dtype=torch.int32, device="cuda")
    stats = torch.zeros((NL, 7), dtype=torch.int64, device="cuda")
    s = torch.cuda.Stream()
    cs = torch.cuda.Stream(priority=-1)   # fetch CTAs are scheduled ahead of compute CTAs

    def step(qt, dt, tok, serial=False):
        if w.append:
            ctx.advance_ctx(ctx_len)
        for l in range(NL):
            if w.layer_prefetch and l > 0:
                ctx.layer_prefetch(l, sel[l - 1], nsel[l - 1], ctx_len, stats, stream=s if serial else cs)
            ctx.decode_step(l, qt[l], None if dt is None else dt[l], nq if dt is not None else 1, index, ctx_len,
                            out[l], stats, None if tok is None else tok[0][l],
                            None if tok is None or tok[1] is None else tok[1][l], sel[l], nsel[l], stream=s,
                            copy_stream=None if serial else cs)
        ctx.join(s)

    q_fix = torch.empty_like(q_dev[0])
    d_fix = torch.empty_like(d_dev[0]) if d_dev is not None else None
    tok_fix = None
    if w.append:
        tok_fix = (torch.empty_like(tok_dev[0][0]),
                   None if tok_dev[0][1] is None else torch.empty_like(tok_dev[0][1]))

    def stage_inputs(t):
        if args.no_io:
            t = 0
        q_fix.copy_(q_dev[t], non_blocking=True)
        if d_fix is not None:
            d_fix.copy_(d_dev[t], non_blocking=True)
        if tok_fix is not None:
            tok_fix[0].copy_(tok_dev[t][0], non_blocking=True)
            if tok_fix[1] is not None:
                tok_fix[1].copy_(tok_dev[t][1], non_blocking=True)

    def capture(serial=False):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step(q_fix, d_fix, tok_fix, serial)
        return g

    # Step 0 eagerly (bootstraps the lookahead selections).  Then one graph over fixed input
    # buffers; each step copies its device-resident inputs into them (inside the timed region)
    # and replays the graph.
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        stage_inputs(0)
        step(q_fix, d_fix, tok_fix, args.serial)
    s.synchronize()
    hist.repair_after_first_step(ctx)
    launches0 = ctx.launch_count()
    graph = capture(args.serial)
    launches_per_step = ctx.launch_count() - launches0
    upload_graphs([graph], s)
    with torch.cuda.stream(s):
        for t in range(1, args.warmup):
            stage_inputs(t)
            graph.replay()
    torch.cuda.synchronize()
    stats0 = stats.cpu().numpy().copy()

    hbm_peak, hbm_src = measured_peaks()
    clocks = ClockSampler(dist.local)
    clocks.start()
    time.sleep(0.3)
    dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        ev0.record(s)
        for t in range(args.warmup, T):
            stage_inputs(t)
            graph.replay()
        ev1.record(s)
    torch.cuda.synchronize()
    dist.barrier()
    elapsed = ev0.elapsed_time(ev1) * 1e-3
    huge_after = hist.huge_after()
    clk = clocks.stop()
    elapsed = dist.max(elapsed)
    stats1 = stats.cpu().numpy()
    dstat = (stats1 - stats0).sum(axis=0)
    link_layers = (stats1 - stats0)[:, 6] / args.steps        # per layer, bytes fetched per step
    launches = launches_per_step * args.steps
    dev_status = ctx.poll_error()
    if dev_status != 0:
        raise RuntimeError(f"device status {K.STATUS.get(dev_status, dev_status)}")

    # Kernel durations: a measurement pass right after the timed region, with the fetch on the
    # compute stream so that the kernels run one at a time; CUDA events around every launch of each
    # kernel, in graphs of their own (one per step, events recorded as graph nodes).  The same pass
    # snapshots each step's selection for the achieved step-to-step overlap.
    per_step_launches = {"attn": NL, "score": NL, "fetch": NL + (NL - 1 if w.layer_prefetch else 0),
                         "update": NL, "topk": NL}
    if w.layer_prefetch:
        per_step_launches["prefetch"] = NL - 1
    for kname, n in per_step_launches.items():
        ctx.kernel_timer_arm(kname, n_meas * n)
    meas_graphs = [capture(serial=True) for _ in range(n_meas)]
    upload_graphs(meas_graphs, s)
    snaps = []
    for i, g in enumerate(meas_graphs):
        with torch.cuda.stream(s):
            stage_inputs(T + i)
            g.replay()
        s.synchronize()
        snaps.append((sel.cpu().numpy(), nsel.cpu().numpy()))
    torch.cuda.synchronize()
    kernel_times = {k: ctx.kernel_timer_read(k) for k in per_step_launches}
    for kname in per_step_launches:
        ctx.kernel_timer_arm(kname, 0)
    if ctx.poll_error() != 0:
        raise RuntimeError("device status set in the measurement pass")
    ov = []
    for (a, na), (b, nb) in zip(snaps, snaps[1:]):
        ov += selection_overlap(a, na, b, nb)
    achieved_overlap = round(float(np.mean(ov)), 4) if ov else None

    link = link.get()
    ms_per_step = elapsed / args.steps * 1e3
    value = dist.world * args.steps / elapsed
    link_per_step = float(dstat[6]) / args.steps
    hbm_step, link_step, per_layer = algorithmic_bytes(w, lens, link_per_step)
    t_step = elapsed / args.steps
    link_peak = link["peak_gbs"]
    step_roof = max(hbm_step / (hbm_peak * 1e9), link_step / (link_peak * 1e9))
    kv_gbs = hbm_step / t_step / 1e9
    misses, hits = float(dstat[1]), float(dstat[0])

    # kernel rooflines: algorithmic bytes per launch / CUDA-event duration per launch (kernels one at
    # a time), against the kernel's own bound (HBM for scoring and attention, the host link for the
    # fetch); `roofline` is the kernel with the most time per step
    def kernel_roofline(kname):
        kms, kn = kernel_times[kname]
        per_launch_ms = kms / max(1, kn)
        if kname == "attn":
            alg = per_layer["attn"]
        elif kname == "score":
            alg = per_layer["index"] + w.n_req * nq * w.n_q_head * w.d_k * 2
        else:
            alg = link_per_step / max(1, per_step_launches["fetch"])
        achieved = alg / (per_launch_ms * 1e-3) / 1e9 if per_launch_ms > 0 else 0.0
        peak = link_peak if kname == "fetch" else hbm_peak
        tr = profile_traffic(kname, w.name)
        r = {"bound": "host-link" if kname == "fetch" else "hbm", "kernel": kname,
             "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "GB/s",
             "frac": round(achieved / peak, 4), "traffic": tr["bytes"] if tr else None,
             "bytes_per_launch": int(alg), "avg_launch_ms": round(per_launch_ms, 5), "launches_timed": kn,
             "peak_source": link["peak_source"] if kname == "fetch" else hbm_src,
             "timing": "CUDA events around each launch; measurement pass after the timed region with the fetch "
                       "on the compute stream (kernels one at a time)"}
        if tr:
            r["traffic_source"] = f"{tr['profile']} ({tr['note']})" if tr["note"] else tr["profile"]
        return r

    rooflines = {k: kernel_roofline(k) for k in ("attn", "score", "fetch")}
    step_ms = {k: ms / max(1, n) * per_step_launches[k] for k, (ms, n) in kernel_times.items()}
    if kernel_times["topk"][1] == 0 and kernel_times["update"][1] > 0:   # fused top-K + update kernel
        step_ms["topk+update"] = step_ms.pop("update")
        step_ms.pop("topk")
    dominant = args.timed_kernel if args.timed_kernel != "auto" else max(rooflines, key=lambda k: step_ms[k])
    roofline = dict(rooflines[dominant])
    roofline["dominant_by"] = "most CUDA-event time per step among attn, score, fetch (kernels one at a time)"
    roofline["kernel_ms_per_step"] = round(step_ms[dominant], 4)

    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(w),
            "effective_kv_gbs": round(kv_gbs, 1),
            "step_roofline": {"hbm_bytes": hbm_step, "link_bytes": link_step, "hbm_peak_gbs": hbm_peak,
                              "link_peak_gbs": link_peak, "bound_ms": round(step_roof * 1e3, 4),
                              "frac": round(step_roof / t_step, 4),
                              "bound": "host-link" if link_step / link_peak > hbm_step / hbm_peak else "hbm"},
            "achieved_overlap": achieved_overlap,
            "miss_fraction": round(misses / max(1.0, misses + hits), 4),
            "prefetch": prefetch_report(w, dstat, args.steps),
            "roofline": roofline, "rooflines": rooflines, "clocks": clk, "gpu_launches": int(launches),
            "kernel_ms_per_step": {k: round(v, 4) for k, v in step_ms.items()},
            "fetch": "inline" if args.serial else "side stream", "host_memory": hist.desc,
            "host_huge_fraction_after_timing": huge_after,
            "launches_per_step": int(launches_per_step)}
    if not w.lookahead:
        dep = dependency_bound_ms(w, per_layer, link_layers, hbm_peak, link_peak)
        line["dependency_bound"] = {"ms": round(dep, 4), "frac": round(dep / (t_step * 1e3), 4),
                                    "what": "sum over layers of index scan + max(attention reads, that layer's "
                                            "fetch), each at its peak: the bound under the layer dependency"}
    if e2e:
        line["e2e"] = run_e2e(args, w, ctx, out, s, q_all, d_all, tok_all, T + n_meas, step, dist)
    if dist.rank == 0 and dist.world == 1 and cpu_baseline:
        per_step, units, cores, desc, coverage = oracle_sample_time(w, 1, 3, min(w.n_layer, 8))
        full = per_step * (w.n_req * w.n_layer * w.n_kv_head) / units
        line["cpu_baseline"] = {"value": round(1.0 / full, 6), "unit": UNIT, "cores": cores, "cpu": cpu_model(),
                                "kind": "oracle", "sample": desc}
        line["dense_softmax_coverage"] = coverage
        line["coverage_study"] = coverage_study(w, q_all[0].numpy().view(np.uint16))
    ctx.close()
    del index, q_dev, d_dev, tok_dev
    torch.cuda.empty_cache()
    return line


def run_e2e(args, w, ctx, out, s, q_all, d_all, tok_all, T, step, dist):
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
        step(q_fix, d_fix, tok_fix, args.serial)
    upload_graphs([g], s)
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


def workload_of(args, name, dist):
    w = W.get(name)
    if args.layers:
        w = w.with_(n_layer=args.layers)
    if args.batch:
        w = w.with_(n_req=args.batch)
    if args.no_io:
        w = w.with_(name=w.name + "_no_io")
    if dist.world > 1:
        w = w.with_(seed=w.seed + dist.rank)       # each GPU serves its own batch of requests
    if w.append:   # history capacity for every appended token of the run (timed, measured, e2e)
        T = args.warmup + args.steps
        w = w.with_(steps=max(w.steps, T + 8 + (0 if args.no_e2e else args.steps) + 1))
    return w


# Policy variants of the headline workload, measured on its history: the [max | min] upper-bound
# block score, and least-important-first eviction.
VARIANTS = {"score_mode=bound": {"score_mode": "bound"}, "evict_policy=importance": {"evict_policy": "importance"}}

SUMMARY_KEYS = ("value", "ms_per_step", "effective_kv_gbs", "step_roofline", "dependency_bound", "achieved_overlap",
                "miss_fraction", "prefetch", "roofline", "kernel_ms_per_step", "clocks", "gpu_launches", "host_memory")


def run_children(args):
    """The other workloads, one child process each (the sweep: one process over a shared history)."""
    res = {}
    jobs = [(name, ["--workload", name, "--steps", "20", "--warmup", "4"]) for name in PER_CONFIG]
    jobs.append(("sweep", ["--workload", "sweep", "--steps", "10", "--warmup", "3"]))
    for name, extra in jobs:
        cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--child", "--no-e2e", "--no-cpu-baseline",
               "--no-per-config"] + extra
        t0 = time.time()
        try:
            r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
        except subprocess.TimeoutExpired:
            res[name] = {"error": "timed out after 900 s"}
            continue
        sys.stderr.write(r.stderr[-4000:])
        lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
        if r.returncode != 0 or not lines:
            tail = (r.stderr.strip().splitlines() or ["no output"])[-1]
            res[name] = {"error": f"exit {r.returncode}: {tail[:300]}"}
            continue
        j = json.loads(lines[-1])
        log(f"{name}: done in {time.time() - t0:.0f}s")
        if name == "sweep":
            res["sweep"] = j
        else:
            res[name] = {k: j[k] for k in SUMMARY_KEYS if k in j}
            res[name]["config"] = j["config"]
    return res


def run_ours(args, dist):
    import torch
    import sparse_kv_cache_decode_gb300 as K
    from sparse_kv_cache_decode_gb300 import build as kbuild

    kbuild.build()
    torch.cuda.set_device(dist.local)
    if args.workload == "sweep":
        return run_sweep(args, dist, K)
    w = workload_of(args, args.workload, dist)
    hist = History(K, w, args.threads, args.numa_local)
    link = LinkPeak(K, hist)
    if args.link_peak_only:
        if dist.rank == 0:
            print(json.dumps({"workload": w.name, "host_memory": hist.desc, "link": link.get()}), flush=True)
        hist.close()
        return 0
    line = run_point(args, dist, w, hist, link, e2e=not args.no_e2e,
                     cpu_baseline=not args.no_cpu_baseline and not args.child)
    line["link_peak"] = link.get()
    if dist.rank == 0 and dist.world == 1 and not args.child and not args.no_per_config:
        line["variants"] = {}
        for vname, kw in VARIANTS.items():
            j = run_point(args, dist, w.with_(name=f"{w.name}_{vname.split('=')[1]}", **kw), hist, link, e2e=False,
                          cpu_baseline=False)
            line["variants"][vname] = {k: j[k] for k in SUMMARY_KEYS if k in j}
    line["host_vmstat_delta"] = hist.vmstat_delta()
    hist.close()
    del hist
    torch.cuda.empty_cache()
    if dist.rank == 0 and dist.world == 1 and not args.child and not args.no_per_config:
        line["per_config"] = run_children(args)
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_sweep(args, dist, K):
    """Several budget/eviction sweep cases over one history (the cases differ only in block size,
    budget and query correlation, none of which changes the stored K/V)."""
    import torch
    names = [n for n in args.sweep_points.split(",") if n]
    ws = [workload_of(args, n, dist) for n in names]
    base = ws[0]
    for w in ws:
        if (w.n_layer, w.n_req, w.n_kv_head, w.max_ctx, w.d_k, w.d_v, w.seed, w.n_heavy) != \
                (base.n_layer, base.n_req, base.n_kv_head, base.max_ctx, base.d_k, base.d_v, base.seed, base.n_heavy):
            raise ValueError("sweep cases must share one history shape")
    hist = History(K, base, args.threads, args.numa_local)
    link = LinkPeak(K, hist)
    points = {}
    for w in ws:
        t0 = time.time()
        try:
            j = run_point(args, dist, w, hist, link, e2e=False, cpu_baseline=False)
            points[w.name] = {k: j[k] for k in SUMMARY_KEYS if k in j}
        except Exception as e:   # one refused case does not end the sweep
            points[w.name] = {"error": str(e)[:300]}
        log(f"{w.name}: {time.time() - t0:.0f}s")
    line = {"metric": METRIC, "unit": UNIT, "workload": "sweep", "n_layer": base.n_layer, "batch": base.n_req,
            "context": base.ctx0, "host_memory": hist.desc, "link_peak": link.get(), "points": points,
            "host_vmstat_delta": hist.vmstat_delta()}
    hist.close()
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    return 0


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
