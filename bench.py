#!/usr/bin/env python3
"""Benchmark of the Hybrid-SWA dual-KV-pool attention path on GB300.

Headline workload: decode, 70-layer stack (60 sliding W=128 + 10 full, 6:1),
32 q / 4 KV heads, d = 128, batch 32, contexts U[8K, 64K], one new token per
sequence.  A step is the whole hot path for one batch: for every layer the
decode attention and the append of the new token (hsa_decode_attn_append, one
fused launch per layer), captured once in a CUDA graph and replayed.

The default run then measures, in the same JSON line, the other workloads of the
metric, each as an object of its own with the same keys (value, ms_per_step,
roofline, e2e, clocks, cpu_baseline): "prefill" (8 requests, prefix 16K-128K,
chunk 2K-8K: chunked prefill attention + append on all 70 layers; TFLOP/s),
"long" (batch 4, contexts 256K-1M) and "mtp" (batch 48, mixed buckets, 4 query
tokens + 1000 window-safe cases).  --workload NAME measures one workload alone
(its line then carries it at the top level).  Inputs are seeded synthetic bf16
N(0,1); the KV pools (tens of GB) are far larger than L2, so no extra flush is
needed.

Prints ONE JSON line (rank 0).  Under torchrun every rank runs an independent
replica of the workload (sequences are independent: weak scaling, no
collective on the data path).
"""
import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np
import torch

import workload

METRIC = ("decode attn tokens/s & KV-read GB/s (% HBM peak); prefill attn TFLOP/s (% peak)")
DATA = "synthetic (seeded bf16 N(0,1), drawn lengths, random page permutation)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# --------------------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return dict(hbm=float(j["hbm_gbs"]), bf16=float(j["bf16_tflops"]),
                    bf16_sustained=float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                    source="measured")
    except Exception:
        return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS, bf16_sustained=1700.0,
                    source="fallback")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.out = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.out = open(self.path, "w")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.out is not None:
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [r for r in rows if r[2] > 300.0] or rows
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "samples": len(rows),
                "power_w_max": max(r[2] for r in rows), "reasons": sorted(reasons)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def max_over_ranks(x, ws, device="cuda"):
    """Slowest rank's value (timings are taken as the max over ranks)."""
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- accounting
def decode_bytes(inst, layer_full, fp8=False):
    """Algorithmic bytes of one decode attention launch on one layer.

    KV: every key some query of the step may see, once (2048 B per token per
    layer: K and V, 4 KV heads, d = 128, bf16): full layers c + T tokens, sliding
    layers min(c + T, W + T - 1).  Plus q read and out written.  An FP8 full layer
    holds its c cached tokens as FP8 codes (E4M3 or E5M2) plus one fp32 scale per
    (token, head) row: 2 * Hkv * (d + 4) bytes per token; the T new rows are read
    as bf16.
    """
    cfg = inst.cfg
    per_tok = 2 * cfg.Hkv * cfg.d * 2
    c = inst.prefix.astype(np.int64)
    qo = 2 * inst.R * cfg.T * cfg.Hq * cfg.d * 2
    if layer_full and fp8:
        return int(c.sum()) * 2 * cfg.Hkv * (cfg.d + 4) + inst.R * cfg.T * per_tok + qo
    if layer_full:
        keys = c + cfg.T
    else:
        keys = np.minimum(c + cfg.T, cfg.W + cfg.T - 1)
    qo = 2 * inst.R * cfg.T * cfg.Hq * cfg.d * 2
    return int(keys.sum()) * per_tok + qo


def pool_ratio(inst):
    """Bytes the dual pool allocates for this workload (bf16 layout: pages of the
    full layers, one W-slot ring row per sequence for each sliding layer) over the
    bytes an all-full stack would allocate for the same pages."""
    cfg = inst.cfg
    row = cfg.Hkv * cfg.d * 2 * 2          # K and V of one position, bf16
    full = inst.num_blocks * cfg.page * row
    ring = inst.n_ring_rows * cfg.W * row
    n_full = sum(1 for f in inst.full if f)
    return (n_full * full + (len(inst.full) - n_full) * ring) / (len(inst.full) * full)


def keys_per_row(inst, layer_full):
    """Keys each new row attends (int64 [rows])."""
    cfg = inst.cfg
    out = np.zeros(inst.rows, np.int64)
    for r in range(inst.R):
        a, b = int(inst.cu_new[r]), int(inst.cu_new[r + 1])
        pos = int(inst.prefix[r]) + np.arange(b - a, dtype=np.int64)
        out[a:b] = pos + 1 if layer_full else np.minimum(pos + 1, cfg.W)
    return out


def prefill_flops(inst, layer_full):
    """4 d Hq x (keys attended per row), masked work excluded."""
    cfg = inst.cfg
    total = 0
    for P, C in zip(inst.prefix.astype(np.int64), inst.new.astype(np.int64)):
        i = np.arange(C, dtype=np.int64)
        if layer_full:
            keys = P + i + 1
        else:
            keys = np.minimum(P + i + 1, cfg.W)
        total += int(keys.sum())
    return 4 * cfg.d * cfg.Hq * total


def prefill_swa_bytes(inst):
    """Algorithmic bytes of one sliding-layer prefill launch: q read and out
    written (rows x Hq x d bf16 each), the chunk's k_new / v_new read, and the
    ring positions some row still sees (min(P, W - 1) per request, 2048 B each)."""
    cfg = inst.cfg
    rows = inst.rows
    qo = 2 * rows * cfg.Hq * cfg.d * 2
    kv_new = 2 * rows * cfg.Hkv * cfg.d * 2
    per_tok = 2 * cfg.Hkv * cfg.d * 2
    ring = int(np.minimum(inst.prefix.astype(np.int64), cfg.W - 1).sum()) * per_tok
    return qo + kv_new + ring


# --------------------------------------------------------------------------- reference arm
def run_reference(args, inst):
    """The CPU oracle as it stands on this host's cores, bounded samples.

    One timed call = the oracle on one full and one sliding layer of the sampled
    sequences (rows).  Returns (value, unit, extrapolated 70-layer step seconds,
    threads, sample description, median measured seconds per call); the value is
    the workload's throughput at the extrapolated step time."""
    import oracle
    import harness  # noqa: F401  (host-only use below)
    cfg = inst.cfg
    nthreads = oracle.num_threads()
    full_layer = next(l for l in range(cfg.n_layers) if inst.full[l])
    swa_layer = next(l for l in range(cfg.n_layers) if not inst.full[l])
    rng = np.random.default_rng(7)
    n_full = sum(inst.full)
    n_swa = cfg.n_layers - n_full
    if cfg.kind == "decode":
        seqs = list(range(inst.R))
        if inst.prefix.sum() > 3_000_000:  # keep host memory and time bounded
            seqs = sorted(rng.choice(inst.R, size=max(1, inst.R // 8), replace=False).tolist())
    else:
        seqs = [0]
    times = []
    cases = {}
    for l in (full_layer, swa_layer):
        rows = [r for s in seqs for r in range(int(inst.cu_new[s]), int(inst.cu_new[s + 1]))]
        if cfg.kind == "prefill":
            rows = rows[:: max(1, len(rows) // 64)]  # a row subsample
        items = np.array([(r, h) for r in rows for h in range(cfg.Hq)], np.int32)
        cases[l] = (_host_case(inst, l, seqs), rows, items)
    calls = []
    for step in range(args.warmup + args.steps):
        t_layer = {}
        call = 0.0
        for l in (full_layer, swa_layer):
            c, rows, items = cases[l]
            t0 = time.perf_counter()
            oracle.attention(window=0 if inst.full[l] else cfg.W, scale=cfg.scale, items=items,
                             nthreads=nthreads, **c)
            dt = time.perf_counter() - t0
            call += dt
            kpr = keys_per_row(inst, inst.full[l])
            t_layer[l] = dt * (kpr.sum() / kpr[rows].sum())  # extrapolate by keys attended
        if step >= args.warmup:
            times.append(t_layer[full_layer] * n_full + t_layer[swa_layer] * n_swa)
            calls.append(call)
    step_s = statistics.median(times)
    call_s = statistics.median(calls)
    if cfg.kind == "decode":
        value = inst.R * cfg.T / step_s
        unit = "tokens/s"
    else:
        flops = sum(prefill_flops(inst, f) for f in inst.full)
        value = flops / step_s / 1e12
        unit = "TFLOP/s"
    sample = ("%s: 1 full + 1 sliding layer, %d of %d sequences%s, extrapolated x(%d, %d) "
              "to %d layers and to all rows" % (cfg.name, len(seqs), inst.R,
                                                 ", row subsample" if cfg.kind == "prefill" else "",
                                                 n_full, n_swa, cfg.n_layers))
    return value, unit, step_s, nthreads, sample, call_s


def _host_case(inst, layer, seqs):
    """Oracle inputs generated on the host (CPU generator stream)."""
    cfg = inst.cfg
    q, k, v = workload.new_tokens(inst, layer, "cpu")
    hk, hv, off, start = [], [], [0], []
    want = set(seqs)
    for s in range(inst.R):
        if s in want:
            a, b, st = workload.history(inst, layer, s, "cpu")
            hk.append(a)
            hv.append(b)
            off.append(off[-1] + a.shape[0])
            start.append(st)
        else:
            off.append(off[-1])
            start.append(int(inst.prefix[s]))
    empty = torch.zeros((0, cfg.Hkv, cfg.d), dtype=torch.bfloat16)
    return dict(cu_rows=inst.cu_new, prefix_len=inst.prefix, q=q, k_new=k, v_new=v,
                hist_k=torch.cat(hk) if hk else empty, hist_v=torch.cat(hv) if hv else empty,
                hist_off=np.array(off, np.int64), hist_start=np.array(start, np.int32))


# --------------------------------------------------------------------------- our arm
class DecodeStep:
    """All layers: decode attention fused with the append of the step's new tokens
    (hsa_decode_attn_append, one launch per layer)."""

    def __init__(self, inst, device, layers=None, swa_prefetch=False, kv_fp8=False,
                 early_pool_read=True, swa_prefetch_frac=1.0):
        import full_attention_kv_gb300 as hsa
        import harness
        self.hsa = hsa
        self.inst = inst
        self.kv_fp8 = kv_fp8
        # each layer's attention is queued right behind the previous layer's, which
        # writes only its own layer's pool: sliding layers may read their ring before
        # that kernel ends (HSA_DECODE_EARLY_POOL_READ)
        self.early = early_pool_read
        cfg = inst.cfg
        self.model_layers = list(range(cfg.n_layers)) if layers is None else list(layers)
        self.layers = list(range(len(self.model_layers)))  # pool layer indices
        self.pool = harness.make_pool(inst, self.model_layers, device=device, stale="zero",
                                      fp8=kv_fp8)
        # layerwise SWA prefetch: every sliding layer's rings also live in a pinned
        # host tier and are brought back each step on a side stream
        self.prefetch = swa_prefetch
        self.swa = [i for i, l in enumerate(self.model_layers) if not inst.full[l]]
        if swa_prefetch:
            self.host_k = {i: self.pool.k[i].cpu().pin_memory() for i in self.swa}
            self.host_v = {i: self.pool.v[i].cpu().pin_memory() for i in self.swa}
            # the sequences whose rings come back from the host tier each step: all of
            # them, or a seeded fraction (requests returning to a cached conversation)
            n = max(1, int(round(swa_prefetch_frac * inst.R)))
            seqs = (np.arange(inst.R) if n >= inst.R else
                    np.sort(np.random.default_rng(inst.cfg.seed).choice(inst.R, n, replace=False)))
            self.host_rows = torch.from_numpy(inst.ring_row[seqs].astype(np.int32)).to(device)
            self.seqs = torch.from_numpy(seqs.astype(np.int32)).to(device)
            self.side = torch.cuda.Stream(device, priority=0)  # below the attention stream
            # one event per run of consecutive sliding layers, recorded once the run's
            # rings are back: the run's first layer waits on it, and the layers after it
            # keep their programmatic launch behind the layer before (a wait on another
            # stream's event before every launch would break that chain)
            self.runs = []
            for i in self.swa:
                if self.runs and self.runs[-1][-1] == i - 1:
                    self.runs[-1].append(i)
                else:
                    self.runs.append([i])
            self.ready = {r[0]: torch.cuda.Event() for r in self.runs}
            ring_bytes = cfg.Hkv * cfg.W * cfg.d * 2 * 2  # K and V of one sequence's ring
            self.prefetch_bytes = len(seqs) * ring_bytes * len(self.swa)
            self.prefetch_frac = len(seqs) / inst.R
        self.q, self.k, self.v = [], [], []
        for l in self.model_layers:
            q, k, v, cl = harness.decode_inputs(inst, l, device)
            self.q.append(q)
            self.k.append(k)
            self.v.append(v)
        self.cl = cl
        B, T = inst.R, cfg.T
        self.out = [torch.empty_like(q) for q in self.q]
        self.ws = hsa.decode_workspace(self.pool, B, T, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.cu = torch.arange(0, B * T + 1, T, dtype=torch.int32, device=device)
        self.seq = torch.arange(B, dtype=torch.int32, device=device)
        self.window = None
        if cfg.n_window_cases:
            m, slots, _ = workload.window_cases(cfg.n_window_cases, cfg.W, seed=cfg.seed)
            self.window = (torch.from_numpy(m).to(device), torch.from_numpy(slots).to(device),
                           torch.empty(len(m), dtype=torch.int32, device=device))
        self.launches_per_step = len(self.layers) + (1 if self.window else 0)

    def attn(self, l, stream=None):
        # attention fused with the append of the step's new rows (accept-all for T > 1)
        self.hsa.hsa_decode_attn_append(self.pool, l, self.q[l], self.k[l], self.v[l], self.cl,
                                        self.inst.cfg.scale, out=self.out[l], workspace=self.ws,
                                        dev_err=self.err, stream=stream,
                                        early_pool_read=self.early)

    def prefetch_all(self, stream):
        with torch.cuda.stream(stream):
            for r in self.runs:
                for i in r:
                    self.hsa.hsa_swa_prefetch(self.pool, i, self.host_k[i], self.host_v[i],
                                              self.host_rows, self.seqs, dev_err=self.err)
                self.ready[r[0]].record(stream)

    def __call__(self):
        if self.prefetch:
            cur = torch.cuda.current_stream()
            self.side.wait_stream(cur)
            self.prefetch_all(self.side)
            for l in self.layers:
                if l in self.ready:
                    cur.wait_event(self.ready[l])
                self.attn(l)
            cur.wait_stream(self.side)
        else:
            for l in self.layers:
                self.attn(l)
        if self.window is not None:
            m, s, o = self.window
            self.hsa.hsa_window_safe_len(m, s, self.inst.cfg.W, out=o)

    def inputs(self):
        return self.q + self.k + self.v

    def outputs(self):
        return self.out

    def kernels(self):
        """The step's kernels, dominant first: (key, name, pool layers, algorithmic
        bytes per launch, bound)."""
        full = [i for i, l in enumerate(self.model_layers) if self.inst.full[l]]
        swa = [i for i, l in enumerate(self.model_layers) if not self.inst.full[l]]
        out = []
        if full:
            key = {"e4m3": "full_fp8", "e5m2": "full_e5m2"}.get(self.kv_fp8, "full")
            out.append((key,
                        "decode_kernel (full layers%s)" % (
                            ", FP8 %s KV" % self.kv_fp8.upper() if self.kv_fp8 else ""),
                        full, decode_bytes(self.inst, True, self.kv_fp8), "hbm", self.attn))
        if swa:
            out.append(("sliding", "decode_kernel (sliding layers, ring)", swa,
                        decode_bytes(self.inst, False), "hbm", self.attn))
        return out

    def units_per_step(self):
        return self.inst.R * self.inst.cfg.T


class PrefillStep:
    """All layers: chunked prefill attention then append of the chunk.

    Replayed steps re-append the same chunk, so after the first step a sliding
    layer's ring holds the chunk's tail instead of the prefix's: values change, the
    work (masks depend only on lengths) does not.
    """

    def __init__(self, inst, device, layers=None):
        import full_attention_kv_gb300 as hsa
        import harness
        self.hsa = hsa
        self.inst = inst
        cfg = inst.cfg
        self.model_layers = list(range(cfg.n_layers)) if layers is None else list(layers)
        self.layers = list(range(len(self.model_layers)))
        self.pool = harness.make_pool(inst, self.model_layers, device=device, stale="zero")
        self.q, self.k, self.v = [], [], []
        for l in self.model_layers:
            q, k, v, cu, pl, seq = harness.prefill_inputs(inst, l, device)
            self.q.append(q)
            self.k.append(k)
            self.v.append(v)
        self.cu, self.pl, self.seq = cu, pl, seq
        self.max_chunk = int(inst.new.max())
        self.out = [torch.empty_like(q) for q in self.q]
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.launches_per_step = 2 * len(self.layers)

    def attn(self, l, stream=None):
        self.hsa.hsa_prefill_attn(self.pool, l, self.q[l], self.k[l], self.v[l], self.cu,
                                  self.pl, self.seq, self.max_chunk, self.inst.cfg.scale,
                                  out=self.out[l], dev_err=self.err, stream=stream)

    def append(self, l, stream=None):
        self.hsa.hsa_kv_append(self.pool, l, self.k[l], self.v[l], self.cu, self.seq,
                               self.pl, dev_err=self.err, stream=stream)

    def layer(self, l):
        self.attn(l)
        self.append(l)

    def __call__(self):
        for l in self.layers:
            self.layer(l)

    def inputs(self):
        return self.q + self.k + self.v

    def outputs(self):
        return self.out

    def kernels(self):
        full = [i for i, l in enumerate(self.model_layers) if self.inst.full[l]]
        swa = [i for i, l in enumerate(self.model_layers) if not self.inst.full[l]]
        out = []
        # appends move each written row once in and once out: 2 x 2048 B per token
        # (a sliding layer writes only the last W rows of each request)
        row = 2 * self.inst.cfg.Hkv * self.inst.cfg.d * 2
        if full:
            out.append(("full", "prefill_kernel (full layers)", full,
                        prefill_flops(self.inst, True), "tensor", self.attn))
        if swa:
            out.append(("sliding", "prefill_swa_kernel (sliding layers)", swa,
                        prefill_swa_bytes(self.inst), "hbm", self.attn))
        if full:
            out.append(("append_full", "append_kernel (full layers)", full,
                        2 * self.inst.rows * row, "hbm", self.append))
        if swa:
            kept = int(np.minimum(self.inst.new, self.inst.cfg.W).sum())
            out.append(("append_sliding", "append_kernel (sliding layers, last W rows)", swa,
                        2 * kept * row, "hbm", self.append))
        return out

    def units_per_step(self):
        return sum(prefill_flops(self.inst, self.inst.full[l]) for l in self.model_layers)


def time_kernel(launch, layers, iters):
    """Average duration of one kernel's launches (launch(layer, stream=...)) on
    `layers`, CUDA events recorded on the stream the launches go to."""
    stream = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in layers]
    ends = [torch.cuda.Event(enable_timing=True) for _ in layers]
    total_ms = 0.0
    n = 0
    for it in range(iters + 1):
        for i, l in enumerate(layers):
            starts[i].record(stream)
            launch(l, stream=stream)
            ends[i].record(stream)
        torch.cuda.synchronize()
        if it == 0:
            continue  # warm-up pass
        for i in range(len(layers)):
            total_ms += starts[i].elapsed_time(ends[i])
            n += 1
    return total_ms / n / 1e3


def _prefetch_report(step, args, stream):
    """Step time without the prefetch, and the prefetch alone, on the same GPU."""
    step.prefetch = False
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        step()
    for _ in range(3):
        g2.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        g2.replay()
    e1.record()
    torch.cuda.synchronize()
    plain_ms = e0.elapsed_time(e1) / args.steps
    step.prefetch = True
    s = torch.cuda.current_stream()
    step.prefetch_all(s)
    torch.cuda.synchronize()
    e0.record(s)
    for _ in range(args.steps):
        step.prefetch_all(s)
    e1.record(s)
    torch.cuda.synchronize()
    alone_ms = e0.elapsed_time(e1) / args.steps
    return {"bytes_per_step": step.prefetch_bytes, "step_ms_without_prefetch": plain_ms,
            "prefetch_alone_ms": alone_ms,
            "prefetch_alone_gbs": step.prefetch_bytes / (alone_ms / 1e3) / 1e9}


def _swap_io(step, ins, outs):
    """Point a step's input (q, k, v per layer) and output lists at other tensors;
    returns the previous (inputs, outputs) for restoring."""
    prev = (step.inputs(), step.outputs())
    n = len(step.q)
    step.q, step.k, step.v = list(ins[:n]), list(ins[n:2 * n]), list(ins[2 * n:3 * n])
    step.out = list(outs)
    return prev


def _graph_step(step, stream, warmup):
    """Warm the step eagerly, capture it in one CUDA graph, replay `warmup` times."""
    with torch.cuda.stream(stream):
        for _ in range(2):
            step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    torch.cuda.synchronize()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    if int(step.err.item()) != 0:
        raise SystemExit("device error flag set: %d" % int(step.err.item()))
    return graph


def _e2e_layered(step, steps, ws):
    """End to end through the C ABI with host buffers, the copies pipelined by layer:
    seconds per step, H2D and D2H bytes per step.

    A serving loop issued eagerly on three streams: every layer's q, k_new and v_new
    go from pinned host memory to the device on one stream, layer l's kernels start
    once its own inputs are in (and the previous step's read-back of its output is
    done), and layer l's output goes back to pinned host memory on a third stream as
    soon as layer l ends.  A step's copies overlap its own kernels and the
    neighbouring steps'; everything is inside the timed region."""
    n = len(step.layers)
    h_in = [t.cpu().pin_memory() for t in step.inputs()]
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in step.outputs()]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    main, s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_done = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]

    def serve(k):
        for _ in range(k):
            with torch.cuda.stream(s_in):
                for l in range(n):
                    s_in.wait_event(ev_done[l])  # the previous step's layer l has read them
                    for h, d in ((h_in[l], step.q[l]), (h_in[n + l], step.k[l]),
                                 (h_in[2 * n + l], step.v[l])):
                        d.copy_(h, non_blocking=True)
                    ev_in[l].record(s_in)
            with torch.cuda.stream(main):
                for l in range(n):
                    main.wait_event(ev_in[l])
                    main.wait_event(ev_out[l])  # the previous step's output l is read back
                    step.layer(l)
                    ev_done[l].record(main)
            with torch.cuda.stream(s_out):
                for l in range(n):
                    s_out.wait_event(ev_done[l])
                    h_out[l].copy_(step.out[l], non_blocking=True)
                    ev_out[l].record(s_out)

    serve(2)
    torch.cuda.synchronize()
    barrier(ws)
    t0 = time.perf_counter()
    serve(steps)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / steps
    if int(step.err.item()) != 0:
        raise SystemExit("device error flag set: %d" % int(step.err.item()))
    del h_in, h_out
    return max_over_ranks(e2e_s, ws), h2d, d2h


def _e2e(step, graph, stream, steps, ws):
    """End to end through the C ABI with host buffers: seconds per step, H2D and
    D2H bytes per step.

    A serving loop: every step copies its inputs from pinned host memory and reads
    its outputs back, all inside the timed region.  Two device input / output sets,
    each with its own captured step, let step i+1's host-to-device copies (one
    stream) and step i's device-to-host read (another) overlap step i's kernels."""
    h_in = [t.cpu().pin_memory() for t in step.inputs()]
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in step.outputs()]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    sets = [(step.inputs(), step.outputs(), graph)]
    alt_in = [torch.empty_like(t) for t in step.inputs()]
    alt_out = [torch.empty_like(t) for t in step.outputs()]
    saved = _swap_io(step, alt_in, alt_out)
    with torch.cuda.stream(stream):
        step()  # warm the second set once before capture
    torch.cuda.synchronize()
    graph_b = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_b, stream=stream):
        step()
    torch.cuda.synchronize()
    _swap_io(step, *saved)
    sets.append((alt_in, alt_out, graph_b))
    cur = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]

    def serve(n):
        for i in range(n):
            b = i & 1
            d_in, d_out, g = sets[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[b])   # step i-2 has consumed this input set
                for h, d in zip(h_in, d_in):
                    d.copy_(h, non_blocking=True)
                ev_in[b].record(s_in)
            cur.wait_event(ev_in[b])
            if i >= 2:
                cur.wait_event(ev_out[b])         # step i-2's outputs are read back
            g.replay()
            ev_done[b].record(cur)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                for h, d in zip(h_out, d_out):
                    h.copy_(d, non_blocking=True)
                ev_out[b].record(s_out)

    serve(2)
    torch.cuda.synchronize()
    barrier(ws)
    t0 = time.perf_counter()
    serve(steps)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / steps
    del sets, alt_in, alt_out, graph_b, h_in, h_out
    return max_over_ranks(e2e_s, ws), h2d, d2h


def _roofline(cfg_name, key, name, per_launch, bound, launch_s, pk):
    """Roofline entry of one kernel: algorithmic work per launch / launch time."""
    if bound == "hbm":
        achieved = per_launch / launch_s / 1e9
        r = {"kernel": name, "bound": "hbm", "achieved": achieved, "peak": pk["hbm"],
             "unit": "GB/s", "frac": achieved / pk["hbm"], "traffic": _traffic(cfg_name, key),
             "peak_source": pk["source"], "launch_us": launch_s * 1e6,
             "bytes_per_launch": per_launch}
    else:
        achieved = per_launch / launch_s / 1e12
        r = {"kernel": name, "bound": "tensor", "achieved": achieved, "peak": pk["bf16"],
             "unit": "TFLOP/s", "frac": achieved / pk["bf16"],
             "frac_sustained": achieved / pk["bf16_sustained"],
             "traffic": _traffic(cfg_name, key),
             "peak_source": pk["source"] + " (burst: each launch timed alone)",
             "launch_us": launch_s * 1e6, "flops_per_launch": per_launch}
    return r


def measure(args, inst, ws, rank, local, cpu_repeats=None):
    """One workload on this rank's GPU: the graph-timed step (max over ranks), every
    kernel of the step against its roofline, the end-to-end serving loop, clocks
    during the timed region, and (rank 0) the CPU oracle on a bounded sample."""
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import full_attention_kv_gb300 as hsa
    hsa.lib()
    cfg = inst.cfg
    layers = None if args.layers is None else [int(x) for x in args.layers.split(",")]
    if cfg.kind == "decode":
        step = DecodeStep(inst, device, layers, swa_prefetch=args.swa_prefetch,
                          kv_fp8=args.kv_fp8, early_pool_read=not args.no_early_pool_read,
                          swa_prefetch_frac=args.swa_prefetch_frac)
    else:
        step = PrefillStep(inst, device, layers)
    # the attention stream runs at high priority (a side stream, if any, at the default)
    stream = torch.cuda.Stream(device, priority=-1)
    if args.profile_step:
        # one eager step between cudaProfilerStart / Stop (for ncu --profile-from-start off)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                step()
        torch.cuda.synchronize()
        torch.cuda.cudart().cudaProfilerStart()
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        torch.cuda.cudart().cudaProfilerStop()
        return {"profile_step": cfg.name, "launches": step.launches_per_step,
                "dev_err": int(step.err.item())}
    graph = _graph_step(step, stream, args.warmup)

    # ---- timed region: K graph replays ------------------------------------
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    kernels = step.kernels()
    with ClockSampler(local) as clk:
        barrier(ws)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            graph.replay()
        e1.record()
        torch.cuda.synchronize()
        barrier(ws)
        step_ms = e0.elapsed_time(e1) / args.steps
        # each kernel of the step, same stream, per-launch events
        iters = max(3, min(args.steps, 10))
        launch_s = [time_kernel(k[5], k[2], iters) for k in kernels]
        prefetch_info = None
        if getattr(step, "prefetch", False):
            prefetch_info = _prefetch_report(step, args, stream)
    clocks = clk.summary()
    step_ms = max_over_ranks(step_ms, ws)
    if hasattr(step, "layer"):
        e2e_s, h2d, d2h = _e2e_layered(step, args.steps, ws)
    else:
        e2e_s, h2d, d2h = _e2e(step, graph, stream, args.steps, ws)

    units = step.units_per_step()
    pk = peaks()
    roofs = [_roofline(cfg.name, k[0], k[1], k[3], k[4], s, pk) for k, s in zip(kernels, launch_s)]
    if cfg.kind == "decode":
        value = units * ws / (step_ms / 1e3)
        unit = "tokens/s"
        e2e_value = units * ws / e2e_s
        kv_step = sum(decode_bytes(inst, inst.full[l], args.kv_fp8 and inst.full[l])
                      for l in step.model_layers)
        extra = {"kv_read_gbs": kv_step / (step_ms / 1e3) / 1e9,
                 "hbm_frac_step": kv_step / (step_ms / 1e3) / 1e9 / pk["hbm"]}
    else:
        value = units * ws / (step_ms / 1e3) / 1e12
        unit = "TFLOP/s"
        e2e_value = units * ws / e2e_s / 1e12
        extra = {"step_tflops_frac": value / ws / pk["bf16"],
                 "step_tflops_frac_sustained": value / ws / pk["bf16_sustained"],
                 "prefill_rows": inst.rows}
    line = {
        "value": value, "unit": unit, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_ms,
        "config": dict(
            workload_config(inst, ws),
            l2="inputs larger than L2 (KV pools %.1f GB)" % (_pool_bytes(step.pool) / 1e9),
            graph="one CUDA graph per step (%d launches)" % step.launches_per_step),
        "roofline": roofs[0],
        "kernels": roofs,
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": step.launches_per_step * args.steps,
    }
    if cfg.kind == "decode":
        line["config"]["early_pool_read"] = step.early
    line.update(extra)
    if args.kv_fp8:
        line["dtype"] = ("%s Full KV Pool (fp16 MMA, fp32 accumulate), bf16 rings / q / out"
                         % args.kv_fp8)
        line["config"]["kv_fp8"] = ("full layers stored as %s codes + one fp32 scale per "
                                    "(token, KV head) row; sliding rings bf16"
                                    % args.kv_fp8.upper())
    if prefetch_info is not None:
        line["swa_prefetch"] = prefetch_info
        line["config"]["swa_prefetch"] = ("every step reloads the sliding layers' rings of %.0f%% "
                                          "of the sequences from a pinned host tier on a side "
                                          "stream, layer by layer" % (100 * step.prefetch_frac))
    del graph, step
    gc.collect()
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline and not args.kv_fp8:
        reps = args.steps if cpu_repeats is None else cpu_repeats
        v, unit_c, _, cores, sample, call_s = run_reference(
            argparse.Namespace(steps=reps, warmup=1), inst)
        line["cpu_baseline"] = {"value": v, "unit": unit_c, "cores": cores, "kind": "oracle",
                                "sample": sample + "; median of %d timed calls after 1 "
                                "untimed (%.3f s per call)" % (reps, call_s)}
    return line


def workload_config(inst, ws):
    """The `config` object both arms report: the workload by what it is, its sizes."""
    cfg = inst.cfg
    return {"workload": "%s: %d-layer 6:1 Hybrid-SWA stack (W=%d), Hq=%d Hkv=%d d=%d, "
                        "batch %d, T=%d, contexts %s" % (
                            cfg.name, cfg.n_layers, cfg.W, cfg.Hq, cfg.Hkv, cfg.d, inst.R,
                            cfg.T, _ctx_desc(cfg)),
            "global_batch": inst.R * ws, "T": cfg.T,
            "context_total_tokens": int(inst.prefix.sum()),
            "parallelism": "replicas x%d" % ws,
            "kv_pool_vs_all_full": pool_ratio(inst)}


def _pool_bytes(pool):
    return sum(t.numel() * t.element_size() for t in pool.k + pool.v)


def _ctx_desc(cfg):
    if cfg.contexts:
        return "/".join(str(c) for c in cfg.contexts)
    if cfg.buckets:
        return "buckets " + ", ".join("%d-%d:%.1f" % b for b in cfg.buckets)
    if cfg.kind == "prefill":
        return "prefix U[%d,%d], chunk U[%d,%d]" % (cfg.prefix_lo, cfg.prefix_hi, cfg.chunk_lo,
                                                     cfg.chunk_hi)
    return "U[%d,%d]" % (cfg.ctx_lo, cfg.ctx_hi)


# DRAM bytes per launch of a kernel from an ncu capture, keyed by (workload, kernel)
# and by the code digest (code_digest) of the source the capture was taken on; a
# kernel whose source has changed since reports None.  Captures of fewer
# sequences / requests are scaled to the full launch by the units processed.
TRAFFIC = {
    # decode_kernel, full layer: 389.2 MB on 4 sequences, scaled by units
    ("decode", "full"): ("decode.cu", "4f3057adad2ada52", 2829665666),
    # decode_kernel, sliding layer: full-size launch (32 sequences)
    ("decode", "sliding"): ("decode.cu", "4f3057adad2ada52", 8786944),
    # decode_kernel, FP8 full layer: 202.1 MB (E4M3 and E5M2) on 4
    # sequences, scaled by units
    ("decode", "full_fp8"): ("decode.cu", "4f3057adad2ada52", 1469597851),
    ("decode", "full_e5m2"): ("decode.cu", "4f3057adad2ada52", 1469201390),
    # decode_kernel, full layer: 1.608 GB on 1 sequence, scaled by units
    ("long", "full"): ("decode.cu", "4f3057adad2ada52", 5674878985),
    ("long", "sliding"): ("decode.cu", "4f3057adad2ada52", 1169664),
    # decode_kernel, full layer, T = 4: 1.658 GB on 8 sequences, scaled by units
    ("mtp", "full"): ("decode.cu", "4f3057adad2ada52", 11699016334),
    ("mtp", "sliding"): ("decode.cu", "4f3057adad2ada52", 14617344),
    # prefill_kernel, full layer: 4.985 GB on 2 requests, scaled by flops
    ("prefill", "full"): ("prefill.cu", "7128fc2d6f16d75e", 15703684589),
    # prefill_swa_kernel, sliding layer: full-size launch
    ("prefill", "sliding"): ("prefill_swa.cu", "40cbea755aac5f81", 808964352),
    # append_kernel, full-size launches (writes still held in L2 at the kernel's end
    # reach DRAM after it)
    ("prefill", "append_full"): ("append.cu", "436d89e400666e68", 143246080),
    ("prefill", "append_sliding"): ("append.cu", "436d89e400666e68", 2110464),
}


def code_digest(path):
    """First 16 hex digits of the SHA-256 of a CUDA source with its comments and
    blank lines removed, so that editing a comment keeps a capture valid."""
    import hashlib
    import re
    with open(path) as f:
        s = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    lines = [re.sub(r"//.*$", "", l).rstrip() for l in s.splitlines()]
    return hashlib.sha256("\n".join(l for l in lines if l).encode()).hexdigest()[:16]


def _traffic(name, key):
    t = TRAFFIC.get((name, key))
    if not t:
        return None
    digest = code_digest(os.path.join(ROOT, "full_attention_kv_gb300", "csrc", t[0]))
    return t[2] if t[1] == digest else None


EXTRA_WORKLOADS = ("prefill", "long", "mtp")
# CPU oracle repeats for the extra workloads (each call already covers a bounded
# sample of the workload; the headline workload repeats as many times as --steps)
EXTRA_CPU_REPEATS = 2


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=None, choices=sorted(workload.CONFIGS),
                    help="measure one workload alone (default: decode as the headline, then "
                         "%s in the same line)" % ", ".join(EXTRA_WORKLOADS))
    ap.add_argument("--batch", type=int, default=None, help="truncate the draw (profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--swa-prefetch", action="store_true",
                    help="decode: reload every sliding layer's rings from pinned host memory "
                         "each step, layer by layer on a side stream")
    ap.add_argument("--swa-prefetch-frac", type=float, default=1.0,
                    help="with --swa-prefetch: the seeded fraction of sequences whose rings "
                         "come back each step (default: all)")
    ap.add_argument("--kv-fp8", nargs="?", const="e4m3", default=None, choices=["e4m3", "e5m2"],
                    help="decode: full layers as an FP8 Full KV Pool of that format (default "
                         "e4m3; no CPU baseline)")
    ap.add_argument("--no-early-pool-read", action="store_true",
                    help="decode: sliding layers wait for the previous kernel before reading "
                         "their ring (the default reads it early, HSA_DECODE_EARLY_POOL_READ)")
    ap.add_argument("--layers", default=None,
                    help="comma-separated model layers (profiling sub-stack; default all)")
    ap.add_argument("--profile-step", action="store_true",
                    help="run one eager step inside cudaProfilerStart/Stop and exit")
    args = ap.parse_args()
    head_name = args.workload or "decode"
    single = (args.workload is not None or args.swa_prefetch or args.kv_fp8 or
              args.layers is not None or args.batch is not None or args.profile_step or
              args.no_early_pool_read)
    if args.kv_fp8 and workload.CONFIGS[head_name].kind != "decode":
        ap.error("--kv-fp8 is a decode variant (prefill reads bf16 pools)")
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    ws, rank, local = dist_env()
    cfg = workload.shard(workload.CONFIGS[head_name], rank)
    inst = workload.draw(cfg, R=args.batch)

    if args.impl == "reference":
        if rank != 0:
            return
        v, unit, step_s, cores, sample, call_s = run_reference(args, inst)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": unit,
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": call_s * 1e3,
                "extrapolated_ms_per_step": step_s * 1e3,
                "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64",
                "data": DATA,
                "config": dict(workload_config(inst, 1),
                               parallelism="oracle on the host cores (rank 0's workload)"),
                "cpu_baseline": {"value": v, "unit": unit, "cores": cores, "kind": "oracle",
                                 "sample": sample + "; ms_per_step is the measured time of "
                                 "one call on the sample (median of %d after %d untimed), "
                                 "extrapolated_ms_per_step the %d-layer step time the value "
                                 "is computed from" % (args.steps, args.warmup,
                                                       cfg.n_layers)},
                "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if ws > 1:
        torch.distributed.init_process_group("nccl")
    res = measure(args, inst, ws, rank, local)
    if "profile_step" in res:
        if rank == 0:
            print(json.dumps(res))
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    line = {"metric": METRIC, "value": res.pop("value"), "unit": res.pop("unit"),
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": res.pop("ms_per_step"), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": res.pop("dtype", "bf16"),
            "data": DATA}
    res.pop("steps")
    res.pop("warmup")
    line.update(res)
    line["env"] = {"gpu": torch.cuda.get_device_name(local),
                   "sms": torch.cuda.get_device_properties(local).multi_processor_count,
                   "torch": torch.__version__, "cuda": torch.version.cuda}
    if not single:
        # the metric's other workloads, each with the same keys, in the same line
        for name in EXTRA_WORKLOADS:
            sub = workload.draw(workload.shard(workload.CONFIGS[name], rank))
            r = measure(args, sub, ws, rank, local, cpu_repeats=EXTRA_CPU_REPEATS)
            r["dtype"] = "bf16"
            line[name] = r
            line["gpu_launches"] += r["gpu_launches"]
    if rank == 0:
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
