"""Benchmark: paged decode attention on GB300 (tokens/s and HBM GB/s).

Headline workload: the ragged continuous batch -- 256 sequences, q_len 1,
context lengths log-uniform in 1..4096, 30% of the sequences sharing a
refcounted 512-token prefix (the same physical blocks), 16 query / 8 KV
heads, head_dim 128, block 16, bf16, pool 1.2x the blocks needed. One step is
one attention layer's decode step: the slot-mapped write of the 256 new
tokens' K/V into the block pool, then paged decode attention over the pool
(balanced split with its merge) -- one ``pa_append_decode`` call (three
kernels). Inputs are device resident when the timed region starts; the e2e
figure moves each step's inputs from pinned host memory and reads the result
back, through the library's public calls.

A model has one KV cache per layer, so the benchmark keeps 28 layers' pools
(the Qwen3-0.6B shape) and each step reads the next layer's pool: no step
finds the previous step's pool in L2. Steps are replayed from CUDA graphs of
up to 28 steps each, so the per-step figure does not depend on ``--steps``.

The same measurement (device-timed steps, the decode call's roofline, e2e,
and the fp64 oracle timed on the host cores) is repeated for the engine batch
(64 x 384) and the long-context batch (8 x 32768, balanced and split-K
16/32/64) under ``secondary``, together with the verify + chunked-prefill
call, the INT8 pool and the cascade decode.

Launch: ``python bench.py [--gpus N --steps K --warmup W]``; for N > 1 under
torchrun, each rank runs its own replica batch (the path shards by sequence
with no exchange) and rank 0 prints one JSON line. ``--impl reference`` times
the fp64 CPU oracle on the headline workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = ("paged decode attention tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU")
UNIT = "tokens/s"
LAYERS = 28                     # one KV cache per layer of the Qwen3-0.6B shape
GRAPH_STEPS = 28                # steps per captured graph (fewer when --steps is smaller)
FALLBACK_HBM_GBS = 6800.0       # only if MEASURED_PEAKS.json is missing
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")

WORKLOADS = {
    "ragged": ("ragged continuous batch: batch 256, q_len 1, context lengths log-uniform "
               "1-4096, 30% of sequences share a refcounted 512-token prefix, 16 Q / 8 KV "
               "heads, head_dim 128, block 16, bf16, pool 1.2x the blocks needed; step = "
               "cache write of 256 new tokens + paged decode attention"),
    "engine": ("engine-shaped decode: batch 64, q_len 1, every context 384, 16 Q / 8 KV heads, "
               "head_dim 128, block 16, bf16, shuffled pool; step = cache write of 64 new "
               "tokens + paged decode attention"),
    "long": ("long-context decode: batch 8, q_len 1, context 32768 each, 16 Q / 8 KV heads, "
             "head_dim 128, block 16, bf16, 1% outlier keys x8; step = cache write of 8 new "
             "tokens + paged decode attention (balanced split)"),
    "mixed": ("mixed verify + chunked prefill: 48 sequences with q_len 5 at contexts "
              "256-8192 + 2 prefill chunks of 512 queries at offsets 0 and 1536, causal, "
              "16 Q / 8 KV heads, head_dim 128, block 16, bf16"),
}
HEADLINE = "ragged"


# ---------------------------------------------------------------------------
# byte and flop counts
# ---------------------------------------------------------------------------

def decode_algorithmic_bytes(w, unique: bool = False, kv_bytes_per_token: int | None = None) -> int:
    """Bytes one decode call must move at least: every context token's K and V
    for all KV heads (4096 B per token at 8 x 128 bf16), q in, out and lse
    out, context lengths and the block-table entries it reads. unique: a
    shared prefix's rows are counted once (its physical blocks are the same
    for every sharer, so HBM has to deliver them only once per call)."""
    ctx = w.context_lens.to(torch.int64)
    tokens = int(ctx.sum())
    if unique:
        for seqs, t in w.meta.get("prefix_groups", []):
            tokens -= t * (len(seqs) - 1)
    per_tok = kv_bytes_per_token or w.num_kv_heads * w.head_dim * 2 * 2
    S, Hq, D = w.num_seqs, w.num_q_heads, w.head_dim
    rows = w.num_q_tokens
    q_out = rows * Hq * D * 2 * 2 + rows * Hq * 4
    tables = int(((ctx + w.block_size - 1) // w.block_size).sum()) * 4 + S * 4
    return tokens * per_tok + q_out + tables


def int8_bytes_per_token(w) -> int:
    """8-bit pools (int8, FP8): 1-byte K and V codes plus one fp32 scale per (token, KV head)
    row each (2112 B per token at 8 x 128)."""
    return w.num_kv_heads * (w.head_dim + 4) * 2


def attention_flops(w) -> int:
    """Useful flops of one call: 4 * D per (query row, head, visible key)."""
    n = 0
    for c, l in zip(w.context_lens.tolist(), w.q_lens.tolist()):
        n += sum(c - l + j + 1 for j in range(l)) if w.causal else l * c
    return n * 4 * w.head_dim * w.num_q_heads


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_18_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f in ("pa_decode.cu", "pa_device.cuh"):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_for(workload: str):
    """DRAM bytes per pa_decode call from the committed ncu summary, if it was
    taken on the current decode kernel source; else None."""
    try:
        d = json.load(open(TRAFFIC_FILE))
        e = d.get(workload)
        if e and e.get("source_hash") == kernel_source_hash():
            return int(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def replica_seed(base_seed: int, rank: int) -> int:
    """Each rank benchmarks its own replica batch, drawn with its own seed."""
    return base_seed + rank


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_step: int, steps: int, world: int, max_total_ms: float) -> float:
    """Tokens/s of the whole job: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_step * steps / (max_total_ms / 1e3)


def graph_plan(K: int, chunk: int = GRAPH_STEPS):
    """Split K steps into graph replays of at most `chunk` steps: (steps per
    full graph, number of full replays, steps of the remainder graph)."""
    c = max(1, min(K, chunk))
    return c, K // c, K % c


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        t0, t1 = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (0, 1e18)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 - 0.15 <= ts <= t1 + 0.15):
                continue
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------

def capture(fn, n: int, first: int = 0):
    """A CUDA graph of n calls fn(first), fn(first + 1), ... ."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(first, first + n):
            fn(i)
    return g


def timed_replays(graphs, stream):
    """CUDA-event time (ms) of each graph replay, in order, on `stream`."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in graphs]
    chunk = 128
    for c0 in range(0, len(graphs), chunk):
        # park the stream briefly so the host can queue a chunk of replays ahead
        torch.cuda._sleep(2_000_000)
        for i in range(c0, min(len(graphs), c0 + chunk)):
            ev[i][0].record(stream)
            graphs[i].replay()
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def mean_call_ms(fn, n_layers: int, reps: int, stream, per_graph: int = GRAPH_STEPS):
    """Mean time of one call when `per_graph` calls (rotating over n_layers
    inputs) run back to back in one graph."""
    fn(0)
    g = capture(lambda i: fn(i % n_layers), per_graph)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    ms = timed_replays([g] * reps, stream)
    return statistics.fmean(ms) / per_graph, statistics.median(ms) / per_graph


# ---------------------------------------------------------------------------
# one decode workload on the device
# ---------------------------------------------------------------------------

class DecodeBench:
    """A decode workload's inputs on the device and `layers` KV pools, each
    filled by the CUDA cache write (history, then the step's new tokens)."""

    def __init__(self, w, dev, B, layers):
        self.w, self.dev, self.B = w, dev, B
        names = ("q", "k_new", "v_new", "slot_new", "block_tables", "context_lens")
        self.d = {k: getattr(w, k).to(dev) for k in names}
        kh, vh, sh_ = w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev)
        self.pools = []
        for _ in range(layers):
            kc, vc = w.empty_pool(dev)
            if w.k_hist.shape[0]:
                B.pa_reshape_and_cache(kh, vh, sh_, kc, vc)
            B.pa_reshape_and_cache(self.d["k_new"], self.d["v_new"], self.d["slot_new"], kc, vc)
            self.pools.append((kc, vc))
        del kh, vh, sh_
        self.out = torch.empty_like(self.d["q"])
        self.lse = torch.empty(self.d["q"].shape[:2], dtype=torch.float32, device=dev)
        self.shape = B.shape_of(self.d["q"], self.pools[0][0], self.d["block_tables"])
        self.ws = {}
        torch.cuda.synchronize()
        if B.pa_debug_read_error() != 0:
            raise RuntimeError("device error while filling the pools")

    def workspace(self, P):
        if P not in self.ws:
            self.ws[P] = self.B.workspace(self.B.pa_decode_workspace_size(self.shape, P), self.dev)
        return self.ws[P]

    def step_calls(self):
        """One prepared pa_append_decode call per layer pool."""
        d, w = self.d, self.w
        return [self.B.prepare_append_decode(d["k_new"], d["v_new"], d["slot_new"], d["q"], kc, vc,
                                             d["block_tables"], d["context_lens"], w.scale,
                                             self.out, self.lse, workspace=self.workspace(0))
                for kc, vc in self.pools]

    def decode_calls(self, P):
        d, w = self.d, self.w
        return [self.B.prepare_decode(d["q"], kc, vc, d["block_tables"], d["context_lens"],
                                      w.scale, self.out, self.lse, num_splits=P,
                                      workspace=self.workspace(P))
                for kc, vc in self.pools]


def measure_decode(name, w, dev, B, args, layers, splits=(0,), world=1, clocks=None,
                   e2e=True):
    """Device-timed steps (exactly args.steps), the decode call's roofline for
    each split mode, and the e2e step through host buffers."""
    stream = torch.cuda.current_stream()
    bench = DecodeBench(w, dev, B, layers)
    n = len(bench.pools)
    steps = bench.step_calls()
    step = lambda i: steps[i % n]()  # noqa: E731
    K = args.steps
    chunk, full, rem = graph_plan(K)
    # warm the plain calls up once outside capture (first-call setup)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(n):
            step(i)
    stream.wait_stream(side)
    g_full = capture(step, chunk)
    g_rem = capture(step, rem, first=chunk) if rem else None
    torch.cuda.synchronize()
    for _ in range(max(1, -(-args.warmup // chunk))):
        g_full.replay()
    torch.cuda.synchronize()
    plan = [g_full] * full + ([g_rem] if g_rem is not None else [])
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if clocks is not None:
        clocks.mark()
    step_ms = timed_replays(plan, stream)
    if clocks is not None:
        clocks.mark()
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(sum(step_ms), world, dev)

    peak, peak_kind = peaks()
    alg = decode_algorithmic_bytes(w, unique=True)
    alg_logical = decode_algorithmic_bytes(w)
    reps = max(3, min(K, 2000) // GRAPH_STEPS)
    rooflines = {}
    for P in splits:
        calls = bench.decode_calls(P)
        mean_ms, med_ms = mean_call_ms(lambda i: calls[i % n](), n, reps, stream)
        achieved = alg / (mean_ms / 1e3) / 1e9
        rooflines[P] = {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic_for(name) if P == 0 else None,
            "kernel": ("pa_decode (paged_decode_kernel + decode_fixup_kernel)" if P == 0 else
                       f"pa_decode num_splits={P} (paged_decode_kernel + splitk_reduce_kernel)"),
            "alg_bytes_per_launch": alg, "alg_bytes_logical": alg_logical,
            "achieved_logical": round(alg_logical / (mean_ms / 1e3) / 1e9, 1),
            "launch_ms": round(mean_ms, 5), "launch_ms_median": round(med_ms, 5),
            "peak_source": f"{peak_kind} hbm_gbs",
        }
    err = B.pa_debug_read_error()
    if err != 0:
        raise RuntimeError(f"device error word {err:#x} after the timed region ({name})")
    res = {
        "workload": WORKLOADS.get(name, name),
        "value": whole_job_rate(w.num_q_tokens, K, world, total_ms),
        "ms_per_step": total_ms / K,
        "steps": K,
        "roofline": rooflines[splits[0]],
        "launches": 3 * K,  # cache write, decode, merge per step
        "l2": (f"inputs larger than L2: {n} layer pools of "
               f"{2 * bench.pools[0][0].numel() * 2 / 1e6:.1f} MB rotated per step"),
    }
    for P in splits[1:]:
        res[f"roofline_splits{P}"] = rooflines[P]
    if e2e:
        res["e2e"] = run_e2e(args, bench)
    del bench
    torch.cuda.empty_cache()
    return res


def run_e2e(args, bench):
    """The step through the public calls with host buffers, every step: the
    step's inputs (q, new K/V, slots, block tables, context lengths) staged in
    one pinned buffer and copied host-to-device in one copy, the library call,
    and out + lse (views of one device buffer) copied back in one copy and
    read on the host.

    `value` runs a forward of the layer steps as an engine captures it: one
    CUDA graph holding every layer's step, each step's upload on a side
    stream overlapping the previous step's call and its download on another
    side stream after its call (two sets of device staging buffers, events
    ordering their reuse, one pinned result slot per step); the host replays
    it and reads every step's result, host-timed over whole forwards.
    `serial_value` runs copy, call, copy back and a stream sync one after the
    other through the binding; `graph_value` is that serial step captured in
    a CUDA graph per layer."""
    w, dev, B = bench.w, bench.dev, bench.B
    names = ("q", "k_new", "v_new", "slot_new", "block_tables", "context_lens")

    def packed(tensors, device, pinned):
        offs, off = [], 0
        for t in tensors:
            offs.append(off)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(off, dtype=torch.uint8, device=device)
        if pinned:
            buf = buf.pin_memory()
        views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                 for o, t in zip(offs, tensors)]
        return buf, views

    src = [getattr(w, k).contiguous() for k in names]
    outs = [torch.empty(w.q.shape, dtype=torch.bfloat16),
            torch.empty(w.q.shape[:2], dtype=torch.float32)]
    n = len(bench.pools)
    stream = torch.cuda.current_stream()
    nbuf = 2
    host_in, dev_in, host_out, dev_out, calls_b, views = [], [], [], [], [], []
    for _ in range(nbuf):
        hb, hv = packed(src, "cpu", True)
        for v, t in zip(hv, src):
            v.copy_(t)
        db, dv = packed(src, dev, False)
        do, (out, lse) = packed(outs, dev, False)
        ho, _ = packed(outs, "cpu", True)
        d = dict(zip(names, dv))
        views.append((d, out, lse))
        host_in.append(hb)
        dev_in.append(db)
        host_out.append(ho)
        dev_out.append(do)
        calls_b.append([B.prepare_append_decode(d["k_new"], d["v_new"], d["slot_new"], d["q"],
                                                kc, vc, d["block_tables"], d["context_lens"],
                                                w.scale, out, lse, workspace=bench.workspace(0),
                                                stream=stream)
                        for kc, vc in bench.pools])
    # One forward of the n layer steps, pipelined and captured in one CUDA
    # graph: step i's upload runs on a side stream while step i-1 computes,
    # its download on another side stream after its call, each into its own
    # pinned slot; events order the reuse of the two device buffer sets. The
    # host replays the graph and then reads every step's result.
    steps = max(1, min(args.steps, 2000))
    host_outs = [packed(outs, "cpu", True)[0] for _ in range(n)]
    sink = [0.0]
    calls_gb = []
    for b in range(nbuf):
        d, out, lse = views[b]
        calls_gb.append([B.prepare_append_decode(d["k_new"], d["v_new"], d["slot_new"], d["q"],
                                                 kc, vc, d["block_tables"], d["context_lens"],
                                                 w.scale, out, lse,
                                                 workspace=bench.workspace(0), stream=None)
                         for kc, vc in bench.pools])
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_done = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    fwd = torch.cuda.CUDAGraph()
    with torch.cuda.graph(fwd):
        cap = torch.cuda.current_stream()
        up.wait_stream(cap)
        down.wait_stream(cap)
        for i in range(n):
            b = i % nbuf
            with torch.cuda.stream(up):
                if i >= nbuf:
                    up.wait_event(ev_done[i - nbuf])  # step i-2 is done with dev_in[b]
                dev_in[b].copy_(host_in[b], non_blocking=True)
                ev_in[i].record(up)
            cap.wait_event(ev_in[i])
            if i >= nbuf:
                cap.wait_event(ev_out[i - nbuf])  # step i-2's result has left dev_out[b]
            calls_gb[b][i]()
            ev_done[i].record(cap)
            with torch.cuda.stream(down):
                down.wait_event(ev_done[i])
                host_outs[i].copy_(dev_out[b], non_blocking=True)
                ev_out[i].record(down)
        cap.wait_stream(up)
        cap.wait_stream(down)

    def forward():
        fwd.replay()
        stream.synchronize()
        for i in range(n):
            sink[0] += float(host_outs[i][0])  # every step's result is read on the host

    reps = max(1, -(-steps // n))
    for _ in range(max(2, -(-min(args.warmup, 56) // n))):
        forward()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(reps):
        forward()
    ms = (time.perf_counter() - t0) * 1e3
    res = {"value": w.num_q_tokens * reps * n / (ms / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": host_in[0].numel(), "d2h_bytes_per_step": host_outs[0].numel(),
           "steps": reps * n, "ms_per_step": ms / (reps * n),
           "path": "prepared pa_append_decode call through the Python binding; every step "
                   "copies its inputs in (one H2D copy from pinned memory) and its out + lse "
                   "back (one D2H copy), and the host reads every result; the n layer steps of "
                   "a forward are captured in one CUDA graph with the uploads and downloads on "
                   "side streams overlapping the calls; host-timed over whole forwards"}

    # serial: copy in, call, copy back, sync, every step
    hb, db, ho, do, calls = host_in[0], dev_in[0], host_out[0], dev_out[0], calls_b[0]

    def step(i):
        db.copy_(hb, non_blocking=True)
        calls[i % n]()
        ho.copy_(do, non_blocking=True)
        stream.synchronize()  # the result is read on the host

    for i in range(max(3, min(args.warmup, 50))):
        step(i)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for i in range(steps):
        step(i)
    e.record()
    torch.cuda.synchronize()
    res["serial_value"] = w.num_q_tokens * steps / (s.elapsed_time(e) / 1e3)

    # the serial step as an engine captures it: the two copies and the call in
    # a CUDA graph per layer, replayed and read back every step
    d, out, lse = views[0]
    calls_graph = [B.prepare_append_decode(d["k_new"], d["v_new"], d["slot_new"], d["q"], kc, vc,
                                           d["block_tables"], d["context_lens"], w.scale, out,
                                           lse, workspace=bench.workspace(0), stream=None)
                   for kc, vc in bench.pools]  # the capture stream at capture time
    graphs = []
    for i in range(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            db.copy_(hb, non_blocking=True)
            calls_graph[i]()
            ho.copy_(do, non_blocking=True)
        graphs.append(g)
    for i in range(max(3, min(args.warmup, 50))):
        graphs[i % n].replay()
        stream.synchronize()
    torch.cuda.synchronize()
    s.record()
    for i in range(steps):
        graphs[i % n].replay()
        stream.synchronize()  # the result is read on the host
    e.record()
    torch.cuda.synchronize()
    res["graph_value"] = w.num_q_tokens * steps / (s.elapsed_time(e) / 1e3)
    return res


# ---------------------------------------------------------------------------
# the other rows: verify + chunked prefill, int8 pool, cascade
# ---------------------------------------------------------------------------

def time_graph_calls(fn, per_replay=2, reps=30):
    """Mean ms of one call, `per_replay` calls per graph replay."""
    fn()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_replay):
            fn()
    for _ in range(5):
        g.replay()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(1_000_000)
    for a, b in evs:
        a.record()
        g.replay()
        b.record()
    torch.cuda.synchronize()
    return statistics.fmean(a.elapsed_time(b) for a, b in evs) / per_replay


def unique_kv_bytes(w) -> int:
    """KV bytes of the distinct physical rows a batch attends (a shared prefix
    counted once), plus q / out / lse: the bytes a cascade decode must move."""
    ctx = w.context_lens.to(torch.int64)
    tokens = int(ctx.sum())
    for seqs, t in w.meta.get("prefix_groups", []):
        tokens -= t * (len(seqs) - 1)
    rows = w.num_q_tokens
    return (tokens * w.num_kv_heads * w.head_dim * 2 * 2 +
            rows * w.num_q_heads * w.head_dim * 2 * 2 + rows * w.num_q_heads * 4)


def device_pool(w, dev, B):
    kc, vc = w.empty_pool(dev)
    B.pa_reshape_and_cache(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev), kc, vc)
    B.pa_reshape_and_cache(w.k_new.to(dev), w.v_new.to(dev), w.slot_new.to(dev), kc, vc)
    return kc, vc


def run_secondary_varlen(w, dev, B, peak):
    """Verify + chunked-prefill call (tensor cores) on the mixed workload."""
    kc, vc = device_pool(w, dev, B)
    q = w.q.to(dev)
    bt, cl, cu = w.block_tables.to(dev), w.context_lens.to(dev), w.cu_seqlens_q.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    sh = B.shape_of(q, kc, bt)
    ws = B.workspace(B.pa_decode_varlen_workspace_size(sh, q.shape[0], w.max_q_len), dev)
    ms = time_graph_calls(lambda: B.pa_decode_varlen(q, kc, vc, bt, cl, cu, w.max_q_len, w.scale,
                                                     out, lse, causal=True, workspace=ws))
    alg = decode_algorithmic_bytes(w)
    fl = attention_flops(w)
    gbs = alg / (ms / 1e3) / 1e9
    return {"workload": WORKLOADS["mixed"], "call_ms": round(ms, 5), "alg_bytes": alg,
            "achieved_gbs": round(gbs, 1), "frac_of_measured_peak": round(gbs / peak, 4),
            "useful_gflop": round(fl / 1e9, 3),
            "achieved_tflops": round(fl / (ms / 1e3) / 1e12, 1),
            "value": w.num_q_tokens / (ms / 1e3), "unit": "query tokens/s"}


def run_secondary_int8(ws_by_name, dev, B, peak):
    """Decode over the 8-bit pools (quantised cache write, fused dequant),
    int8 and FP8 E4M3: the engine and ragged batches rotated over the layer
    pools (as their bf16 lines are), and the long batch (one pool, larger
    than L2)."""
    fmts = {
        "int8": (lambda w: w.empty_pool_i8(dev), B.pa_reshape_and_cache_int8,
                 B.pa_decode_int8_workspace_size, B.pa_decode_int8,
                 "int8 codes + fp32 row scales, one 2112-byte tile"),
        "fp8": (lambda w: w.empty_pool_f8(dev), B.pa_reshape_and_cache_fp8,
                B.pa_decode_fp8_workspace_size, B.pa_decode_fp8,
                "FP8 E4M3 codes + fp32 row scales, one 2112-byte tile"),
    }
    res = {}
    for fmt, (empty, write, ws_size, decode, desc) in fmts.items():
        for name, nlayers in (("engine", LAYERS), ("ragged", LAYERS), ("long", 1)):
            w = ws_by_name[name]
            pools = []
            kh, vh, sh_ = w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev)
            kn, vn, sn = w.k_new.to(dev), w.v_new.to(dev), w.slot_new.to(dev)
            for _ in range(nlayers):
                kc, vc = empty(w)
                write(kh, vh, sh_, kc, vc)
                write(kn, vn, sn, kc, vc)
                pools.append((kc, vc))
            del kh, vh, sh_
            q = w.q.to(dev)
            bt, cl = w.block_tables.to(dev), w.context_lens.to(dev)
            out = torch.empty_like(q)
            lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
            sh = B.shape_of(q, pools[0][0], bt)
            ws = B.workspace(ws_size(sh, 0), dev)
            ctr = [0]

            def call():
                kc, vc = pools[ctr[0] % nlayers]
                ctr[0] += 1
                decode(q, kc, vc, bt, cl, w.scale, out, lse, num_splits=0, workspace=ws)
            ms = time_graph_calls(call, per_replay=4 if nlayers > 1 else 2)
            alg = decode_algorithmic_bytes(w, unique=True,
                                           kv_bytes_per_token=int8_bytes_per_token(w))
            gbs = alg / (ms / 1e3) / 1e9
            res[f"{name}_{fmt}"] = {"decode_ms": round(ms, 5), "alg_bytes": alg,
                                    "achieved_gbs": round(gbs, 1),
                                    "frac_of_measured_peak": round(gbs / peak, 4),
                                    "value": w.num_q_tokens / (ms / 1e3), "unit": UNIT,
                                    "kv_format": desc}
            del pools
            torch.cuda.empty_cache()
    return res


def run_secondary_cascade(ws_by_name, dev, B):
    """Cascade (shared-prefix) decode against plain balanced decode on the
    ragged batch (30% share a 512-token prefix) and on a shared-prompt batch
    (128 sequences behind one 4096-token prompt)."""
    from paged_kv_decode_18_gb300 import workloads as W

    res = {}
    for name in ("ragged", "shared_prompt"):
        w = ws_by_name[name]
        kc, vc = device_pool(w, dev, B)
        q = w.q.to(dev)
        bt, cl = w.block_tables.to(dev), w.context_lens.to(dev)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        sh = B.shape_of(q, kc, bt)
        sg, cu, mem, pl, mg, mp = W.cascade_groups(w)
        sg, cu, mem, pl = sg.to(dev), cu.to(dev), mem.to(dev), pl.to(dev)
        wsd = B.workspace(B.pa_decode_workspace_size(sh, 0), dev)
        wsc = B.workspace(B.pa_decode_cascade_workspace_size(sh, pl.shape[0], mem.numel(), mg,
                                                             mp), dev)
        calls = {
            "decode": lambda: B.pa_decode(q, kc, vc, bt, cl, w.scale, out, lse,  # noqa
                                          num_splits=0, workspace=wsd),
            # the library's choice (PA_CASCADE_AUTO), and the cascade's phases forced
            "cascade": lambda: B.pa_decode_cascade(q, kc, vc, bt, cl, sg, cu, mem, pl, mg,  # noqa
                                                   mp, w.scale, out, lse, workspace=wsc),
            "cascade_forced": lambda: B.pa_decode_cascade(  # noqa
                q, kc, vc, bt, cl, sg, cu, mem, pl, mg, mp, w.scale, out, lse, workspace=wsc,
                policy=B.PA_CASCADE_ALWAYS),
        }
        ub = unique_kv_bytes(w)
        for kind, fn in calls.items():
            ms = time_graph_calls(fn)
            res[f"{name}_{kind}"] = {"call_ms": round(ms, 5), "unique_kv_bytes": ub,
                                     "unique_gbs": round(ub / (ms / 1e3) / 1e9, 1),
                                     "value": w.num_q_tokens / (ms / 1e3), "unit": UNIT}
        del kc, vc
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline legs and --impl reference)
# ---------------------------------------------------------------------------

def subset_workload(w, seqs):
    """The sequences `seqs` of a workload with their rows of q / new K/V:
    index bookkeeping only."""
    import copy

    idx = torch.tensor(seqs, dtype=torch.int64)
    cu = w.cu_seqlens_q.to(torch.int64)
    rows = torch.cat([torch.arange(int(cu[s]), int(cu[s + 1])) for s in seqs])
    sub = copy.copy(w)
    sub.context_lens = w.context_lens[idx]
    sub.q_lens = w.q_lens[idx]
    sub.block_tables = w.block_tables[idx]
    sub.q, sub.k_new, sub.v_new, sub.slot_new = (w.q[rows], w.k_new[rows], w.v_new[rows],
                                                 w.slot_new[rows])
    c = torch.zeros(len(seqs) + 1, dtype=torch.int32)
    c[1:] = torch.cumsum(sub.q_lens, 0)
    sub.cu_seqlens_q = c
    return sub


def oracle_rate(w, budget_s: float, num_threads: int = 0, max_steps: int | None = None,
                name: str = ""):
    """Time the fp64 oracle on a workload: each step is the oracle's cache
    write of the new tokens plus paged attention over a sample of the
    sequences (the whole batch when one step fits a third of the budget,
    else evenly spaced sequences sized to that). num_threads 0 = all host
    cores. Returns (query tokens/s, threads, description, steps, tokens per step)."""
    import numpy as np

    from oracle import oracle
    from paged_kv_decode_18_gb300 import workloads as W

    kp = np.full(w.pool_shape(), W.POOL_SENTINEL_BITS, np.uint16)
    vp = kp.copy()
    if w.k_hist.shape[0]:
        oracle.reshape_and_cache(w.k_hist, w.v_hist, w.slot_hist, kp, vp, w.block_size)
    threads = oracle.max_threads() if num_threads <= 0 else num_threads

    def one(x):
        oracle.reshape_and_cache(x.k_new, x.v_new, x.slot_new, kp, vp, x.block_size)
        oracle.paged_attention(x.q, kp, vp, x.block_tables, x.context_lens, x.cu_seqlens_q,
                               x.scale, causal=x.causal, num_threads=threads)

    t = time.perf_counter()
    one(w)
    full = time.perf_counter() - t
    per_step = budget_s / 3 if max_steps is None else budget_s / max(1, max_steps)
    x = w
    if full > per_step and w.num_seqs > 1:
        n = max(1, min(w.num_seqs, int(w.num_seqs * per_step / max(full, 1e-6))))
        seqs = sorted(set(np.linspace(0, w.num_seqs - 1, n).round().astype(int).tolist()))
        x = subset_workload(w, seqs)
    steps = 0
    t0 = time.perf_counter()
    while True:
        one(x)
        steps += 1
        el = time.perf_counter() - t0
        if max_steps is not None and steps >= max_steps:
            break
        if max_steps is None and el >= budget_s and steps >= 3:
            break
    el = time.perf_counter() - t0
    what = "all" if x is w else "an evenly spaced sample"
    desc = (f"fp64 oracle, {name or w.name} workload: {steps} steps of cache write + paged "
            f"attention over {what} {x.num_seqs} of {w.num_seqs} sequences "
            f"({x.num_q_tokens} query tokens per step), {threads} threads")
    return x.num_q_tokens * steps / el, threads, desc, steps, x.num_q_tokens


def cpu_baseline(w, name, budget_all=6.0, budget_one=2.0):
    rate, threads, desc, _, _ = oracle_rate(w, budget_all, name=name)
    rate1, _, desc1, _, _ = oracle_rate(w, budget_one, num_threads=1, name=name)
    return {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
            "value_1_thread": rate1, "sample_1_thread": desc1}


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from paged_kv_decode_18_gb300 import workloads as W

    w = W.make(HEADLINE, seed=args.seed)
    budget = 100.0
    per = budget / (args.steps + max(3, args.warmup))
    oracle_rate(w, per * max(3, args.warmup), max_steps=max(3, args.warmup), name=HEADLINE)
    rate, threads, desc, steps, n = oracle_rate(w, per * args.steps, max_steps=args.steps,
                                                name=HEADLINE)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * n / rate,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOADS[HEADLINE], "num_seqs": w.num_seqs,
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# single-case runs (eager calls; used for ncu captures of one kernel)
# ---------------------------------------------------------------------------

def run_case(args, dev):
    from paged_kv_decode_18_gb300 import binding as B
    from paged_kv_decode_18_gb300 import build as libbuild
    from paged_kv_decode_18_gb300 import workloads as W

    libbuild.build()
    B.load()
    if args.case == "prefill":  # the chunked-prefill part of the mixed batch
        w = W.mixed(seed=args.seed, num_verify=0)
    elif args.case == "prefill_long":  # two 2048-token chunks (contexts 2048 and 8192)
        w = W.mixed(seed=args.seed, num_verify=0, prefill_chunk=2048, prefill_offsets=(0, 6144))
    elif args.case.endswith(("_int8", "_fp8")):
        w = W.make(args.case.rsplit("_", 1)[0], seed=args.seed)
    elif args.case == "shared_prompt":
        w = W.shared_prompt(seed=args.seed)
    else:
        w = W.make(args.case, seed=args.seed)
    int8 = args.case.endswith(("_int8", "_fp8"))
    fp8 = args.case.endswith("_fp8")
    q8_write = B.pa_reshape_and_cache_fp8 if fp8 else B.pa_reshape_and_cache_int8
    q8_decode = B.pa_decode_fp8 if fp8 else B.pa_decode_int8
    q8_ws = B.pa_decode_fp8_workspace_size if fp8 else B.pa_decode_int8_workspace_size
    if int8:
        kc, vc = w.empty_pool_f8(dev) if fp8 else w.empty_pool_i8(dev)
        q8_write(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev), kc, vc)
    else:
        kc, vc = w.empty_pool(dev)
        B.pa_reshape_and_cache(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev), kc, vc)
    k_new, v_new, slot_new = w.k_new.to(dev), w.v_new.to(dev), w.slot_new.to(dev)
    q = w.q.to(dev)
    bt, cl, cu = w.block_tables.to(dev), w.context_lens.to(dev), w.cu_seqlens_q.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    sh = B.shape_of(q, kc, bt)
    varlen = args.case in ("mixed", "prefill", "prefill_long")
    cascade = args.case == "shared_prompt"
    if varlen:
        ws = B.workspace(B.pa_decode_varlen_workspace_size(sh, q.shape[0], w.max_q_len), dev)
    elif int8:
        ws = B.workspace(q8_ws(sh, args.splits), dev)
    elif cascade:
        sg, cg, mem, pl, mg, mp = W.cascade_groups(w)
        sg, cg, mem, pl = sg.to(dev), cg.to(dev), mem.to(dev), pl.to(dev)
        ws = B.workspace(B.pa_decode_cascade_workspace_size(sh, pl.shape[0], mem.numel(), mg,
                                                            mp), dev)
    else:
        ws = B.workspace(B.pa_decode_workspace_size(sh, args.splits), dev)

    def step():
        if int8:
            q8_write(k_new, v_new, slot_new, kc, vc)
            q8_decode(q, kc, vc, bt, cl, w.scale, out, lse, num_splits=args.splits,
                      workspace=ws)
            return
        B.pa_reshape_and_cache(k_new, v_new, slot_new, kc, vc)
        if varlen:
            B.pa_decode_varlen(q, kc, vc, bt, cl, cu, w.max_q_len, w.scale, out, lse,
                               causal=True, workspace=ws)
        elif cascade:
            B.pa_decode_cascade(q, kc, vc, bt, cl, sg, cg, mem, pl, mg, mp, w.scale, out, lse,
                                workspace=ws)
        else:
            B.pa_decode(q, kc, vc, bt, cl, w.scale, out, lse, num_splits=args.splits,
                        workspace=ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    err = B.pa_debug_read_error()
    ms = statistics.fmean(a.elapsed_time(b) for a, b in evs)
    print(json.dumps({"case": args.case, "splits": args.splits, "step_ms": ms,
                      "alg_bytes": decode_algorithmic_bytes(w),
                      "alg_bytes_unique": decode_algorithmic_bytes(w, unique=True),
                      "device_error": err}))
    return 1 if err else 0


# ---------------------------------------------------------------------------

def run_ours(args, rank, world, dev):
    from paged_kv_decode_18_gb300 import binding as B
    from paged_kv_decode_18_gb300 import workloads as W

    B.load()
    peak, _ = peaks()
    clocks = ClockSampler(torch.cuda.current_device() if dev.index is None else dev.index)
    clocks.start()
    w = W.make(HEADLINE, seed=replica_seed(args.seed, rank))
    head = measure_decode(HEADLINE, w, dev, B, args, LAYERS, world=world, clocks=clocks)
    clk = clocks.stop()
    head["clocks"] = clk
    if rank != 0 or args.no_secondary:
        return head, None, {HEADLINE: w}
    sec = {}
    ws_by_name = {HEADLINE: w}
    for name, layers, splits in (("engine", LAYERS, (0,)), ("long", 2, (0, 16, 32, 64))):
        wx = W.make(name, seed=args.seed)
        ws_by_name[name] = wx
        sec[name] = measure_decode(name, wx, dev, B, args, layers, splits=splits)
    wm = W.mixed(seed=args.seed)
    ws_by_name["mixed"] = wm
    sec["mixed_varlen"] = run_secondary_varlen(wm, dev, B, peak)
    sec.update(run_secondary_int8(ws_by_name, dev, B, peak))
    ws_by_name["shared_prompt"] = W.shared_prompt(seed=args.seed)
    sec.update(run_secondary_cascade(ws_by_name, dev, B))
    return head, sec, ws_by_name


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=280)
    ap.add_argument("--warmup", type=int, default=28)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=["tiny", "engine", "ragged", "long", "mixed", "prefill", "prefill_long",
                                       "ragged_int8", "engine_int8", "long_int8",
                                       "ragged_fp8", "engine_fp8", "long_fp8",
                                       "shared_prompt"],
                    help="time one workload with eager calls (for profiling), nothing else")
    ap.add_argument("--splits", type=int, default=0, help="num_splits for --case decode runs")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.case:
        return run_case(args, dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    from paged_kv_decode_18_gb300 import build as libbuild
    if rank == 0:
        libbuild.build()
    if world > 1:
        torch.distributed.barrier()

    head, sec, ws_by_name = run_ours(args, rank, world, dev)
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            cpu = cpu_baseline(ws_by_name[HEADLINE], HEADLINE)
            if sec is not None:
                for name in ("engine", "long"):
                    sec[name]["cpu_baseline"] = cpu_baseline(ws_by_name[name], name)
                sec["mixed_varlen"]["cpu_baseline"] = cpu_baseline(ws_by_name["mixed"], "mixed")
        w = ws_by_name[HEADLINE]
        line = {
            "metric": METRIC,
            "value": head["value"],
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": head["ms_per_step"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOADS[HEADLINE], "num_seqs": w.num_seqs,
                       "context_tokens": int(w.context_lens.sum()),
                       "global_batch": w.num_seqs * world, "parallelism": f"replicas x{world}",
                       "num_splits": 0, "l2": head["l2"],
                       "graph_steps": graph_plan(args.steps)[0]},
            "roofline": head["roofline"],
            "cpu_baseline": cpu,
            "e2e": head["e2e"],
            "gpu_launches": head["launches"],
            "clocks": head["clocks"],
        }
        if sec is not None:
            line["secondary"] = sec
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
