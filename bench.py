"""Benchmark: paged decode attention on GB300 (tokens/s and HBM GB/s).

One step = one attention layer's decode step of the engine-shaped batch
(64 sequences, context 384, q_len 1, 16 query / 8 KV heads, head_dim 128,
block 16, bf16): the slot-mapped write of the 64 new tokens' K/V into the
block pool, then paged decode attention over the pool (balanced split with
its merge) -- one ``pa_append_decode`` call (three kernels). Inputs are device resident when the timed region starts; the
e2e figure instead moves each step's inputs from pinned host memory and
reads the result back, through the library's public calls.

The KV pool of the engine batch (100.7 MB) is smaller than the 129 MB L2, so
the benchmark keeps several layers' caches (as a model has) and rotates
through them step by step: each step reads a pool that the previous steps
have pushed out of L2.

Launch: ``python bench.py [--gpus N --steps K --warmup W]``; for N > 1 under
torchrun, each rank runs its own replica batch (the path shards by sequence
with no exchange) and rank 0 prints one JSON line. ``--impl reference`` times
the fp64 CPU oracle on the same workload instead.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = ("paged decode attention tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU")
UNIT = "tokens/s"
WORKLOAD = ("engine-shaped decode: batch 64, q_len 1, every context 384, 16 Q / 8 KV heads, "
            "head_dim 128, block 16, bf16, shuffled pool; step = cache write of 64 new "
            "tokens + paged decode attention")
LAYERS = 28                     # one KV cache per layer of the Qwen3-0.6B shape (28 x 100.7 MB)
FALLBACK_HBM_GBS = 6800.0       # only if MEASURED_PEAKS.json is missing
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def decode_algorithmic_bytes(w) -> int:
    """Bytes one decode call must move at least: every context token's K and V
    for all KV heads (4096 B per token at 8 x 128 bf16), q in, out and lse
    out, context lengths and the block-table entries it reads."""
    ctx = w.context_lens.to(torch.int64)
    kv = int(ctx.sum()) * w.num_kv_heads * w.head_dim * 2 * 2
    S, Hq, D = w.num_seqs, w.num_q_heads, w.head_dim
    rows = w.num_q_tokens
    q_out = rows * Hq * D * 2 * 2 + rows * Hq * 4
    tables = int(((ctx + w.block_size - 1) // w.block_size).sum()) * 4 + S * 4
    return kv + q_out + tables


def decode_algorithmic_bytes_int8(w) -> int:
    """As decode_algorithmic_bytes for the int8 pool: 1-byte K and V codes plus
    one fp32 scale per (token, KV head) row each (2112 B per token)."""
    ctx = w.context_lens.to(torch.int64)
    kv = int(ctx.sum()) * w.num_kv_heads * (w.head_dim + 4) * 2
    S, Hq, D = w.num_seqs, w.num_q_heads, w.head_dim
    rows = w.num_q_tokens
    q_out = rows * Hq * D * 2 * 2 + rows * Hq * 4
    tables = int(((ctx + w.block_size - 1) // w.block_size).sum()) * 4 + S * 4
    return kv + q_out + tables


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
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current decode kernel source; else None."""
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
# our arm
# ---------------------------------------------------------------------------

class Layer:
    """One layer's KV pool (filled by the CUDA cache write) and its graphs."""

    def __init__(self, w, dev, B, bufs):
        self.kc, self.vc = w.empty_pool(dev)
        if w.k_hist.shape[0]:
            B.pa_reshape_and_cache(bufs["k_hist"], bufs["v_hist"], bufs["slot_hist"],
                                   self.kc, self.vc)
        B.pa_reshape_and_cache(bufs["k_new"], bufs["v_new"], bufs["slot_new"], self.kc,
                               self.vc)


def run_ours(args, rank, world, dev):
    from paged_kv_decode_18_gb300 import binding as B
    from paged_kv_decode_18_gb300 import workloads as W

    B.load()
    w = W.engine(seed=replica_seed(args.seed, rank))
    stream = torch.cuda.current_stream()
    bufs = {k: getattr(w, k).to(dev) for k in
            ("q", "k_new", "v_new", "slot_new", "k_hist", "v_hist", "slot_hist",
             "block_tables", "context_lens")}
    layers = [Layer(w, dev, B, bufs) for _ in range(LAYERS)]
    out = torch.empty_like(bufs["q"])
    lse = torch.empty(bufs["q"].shape[:2], dtype=torch.float32, device=dev)
    sh = B.shape_of(bufs["q"], layers[0].kc, bufs["block_tables"])
    ws = B.workspace(B.pa_decode_workspace_size(sh, 0), dev)
    torch.cuda.synchronize()
    if B.pa_debug_read_error() != 0:
        raise RuntimeError("device error while filling the pools")

    def step(l):
        # the whole step in one call: cache write of the new tokens, then decode
        B.pa_append_decode(bufs["k_new"], bufs["v_new"], bufs["slot_new"], bufs["q"], l.kc, l.vc,
                           bufs["block_tables"], bufs["context_lens"], w.scale, out, lse,
                           workspace=ws)

    def decode(l):
        B.pa_decode(bufs["q"], l.kc, l.vc, bufs["block_tables"], bufs["context_lens"],
                    w.scale, out, lse, num_splits=0, workspace=ws)

    # CUDA graphs, as an engine captures its decode step: one graph runs the
    # attention step of every layer of the model back to back, each layer on
    # its own KV cache (graph launch cost is paid once per replay, not per
    # layer); single-layer graphs cover a remainder.
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for l in layers:
            step(l)
            decode(l)
    stream.wait_stream(side)

    def capture(fn, ls):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for l in ls:
                fn(l)
        return g

    g_steps = capture(step, layers)
    g_decs = capture(decode, layers)
    g_step1 = [capture(step, [l]) for l in layers]
    torch.cuda.synchronize()

    clocks = ClockSampler(torch.cuda.current_device() if dev.index is None else dev.index)
    clocks.start()
    for _ in range(max(1, args.warmup // LAYERS)):
        g_steps.replay()
        g_decs.replay()
    torch.cuda.synchronize()

    def timed(graphs):
        """CUDA-event time (ms) of each graph replay, in order."""
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

    K = args.steps
    plan = [g_steps] * (K // LAYERS) + g_step1[:K % LAYERS]   # exactly K steps
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.mark()
    step_ms = timed(plan)
    clocks.mark()
    if world > 1:
        torch.distributed.barrier()
    # the dominant call on its own, for the roofline: mean time per call of
    # LAYERS back-to-back decode calls in one graph
    dec_rep = timed([g_decs] * max(1, min(K, 2000) // LAYERS))
    dec_ms = [t / LAYERS for t in dec_rep]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    clk = clocks.stop()
    err = B.pa_debug_read_error()
    if err != 0:
        raise RuntimeError(f"device error word {err:#x} after the timed region")

    tokens_per_step = w.num_q_tokens
    value = whole_job_rate(tokens_per_step, K, world, total_ms)
    dec_mean_ms = statistics.fmean(dec_ms)
    alg = decode_algorithmic_bytes(w)
    peak, peak_kind = peaks()
    achieved = alg / (dec_mean_ms / 1e3) / 1e9
    res = {
        "value": value,
        "ms_per_step": total_ms / K,
        "decode_ms": dec_mean_ms,
        "decode_ms_median": statistics.median(dec_ms),
        "alg_bytes": alg,
        "achieved": achieved,
        "peak": peak,
        "peak_kind": peak_kind,
        "clocks": clk,
        "launches": 3 * K,   # cache write, decode, merge per step
    }
    res["e2e"] = run_e2e(args, w, dev, B, layers, ws)
    if rank == 0 and not args.no_secondary:
        res["secondary"] = run_secondary(args, dev, B)
    return res


def run_e2e(args, w, dev, B, layers, ws):
    """Same step through the public calls with host buffers: the step's inputs
    (q, new K/V, slots, block tables, context lengths) staged in one pinned
    buffer and copied host-to-device in one copy, the library call, and out +
    lse (views of one device buffer) copied back in one copy and read on the
    host, every step."""
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
    host_in, host_views = packed(src, "cpu", True)
    for v, t in zip(host_views, src):
        v.copy_(t)
    dev_in, dv = packed(src, dev, False)
    devb = dict(zip(names, dv))
    outs = [torch.empty(w.q.shape, dtype=torch.bfloat16),
            torch.empty(w.q.shape[:2], dtype=torch.float32)]
    dev_out, (out, lse) = packed(outs, dev, False)
    host_out, (out_h, lse_h) = packed(outs, "cpu", True)
    h2d = host_in.numel()
    d2h = host_out.numel()
    steps = max(1, min(args.steps, 2000))

    def step(l):
        dev_in.copy_(host_in, non_blocking=True)
        B.pa_append_decode(devb["k_new"], devb["v_new"], devb["slot_new"], devb["q"], l.kc, l.vc,
                           devb["block_tables"], devb["context_lens"], w.scale, out, lse,
                           workspace=ws)
        host_out.copy_(dev_out, non_blocking=True)
        torch.cuda.current_stream().synchronize()  # the result is read on the host

    for i in range(max(3, min(args.warmup, 50))):
        step(layers[i % LAYERS])
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for i in range(steps):
        step(layers[i % LAYERS])
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e)
    res = {"value": w.num_q_tokens * steps / (ms / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps}

    # the same step as an engine runs it: the two copies and the call captured
    # once in a CUDA graph per layer, replayed and read back every step
    graphs = []
    for l in layers:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            dev_in.copy_(host_in, non_blocking=True)
            B.pa_append_decode(devb["k_new"], devb["v_new"], devb["slot_new"], devb["q"], l.kc,
                               l.vc, devb["block_tables"], devb["context_lens"], w.scale, out,
                               lse, workspace=ws)
            host_out.copy_(dev_out, non_blocking=True)
        graphs.append(g)
    for i in range(max(3, min(args.warmup, 50))):
        graphs[i % LAYERS].replay()
        torch.cuda.current_stream().synchronize()
    torch.cuda.synchronize()
    s.record()
    for i in range(steps):
        graphs[i % LAYERS].replay()
        torch.cuda.current_stream().synchronize()  # the result is read on the host
    e.record()
    torch.cuda.synchronize()
    res["graph_value"] = w.num_q_tokens * steps / (s.elapsed_time(e) / 1e3)
    return res


def run_secondary(args, dev, B):
    """Decode-kernel bandwidth on the other decode workloads (inputs > L2)."""
    from paged_kv_decode_18_gb300 import workloads as W

    peak, _ = peaks()
    res = {}
    cases = [("ragged", W.ragged, [0]), ("long", W.long, [0, 16, 32, 64])]
    for name, make, splits in cases:
        w = make(seed=args.seed)
        kc, vc = w.empty_pool(dev)
        B.pa_reshape_and_cache(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev), kc, vc)
        B.pa_reshape_and_cache(w.k_new.to(dev), w.v_new.to(dev), w.slot_new.to(dev), kc, vc)
        q = w.q.to(dev)
        bt, cl = w.block_tables.to(dev), w.context_lens.to(dev)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        alg = decode_algorithmic_bytes(w)
        for P in splits:
            sh = B.shape_of(q, kc, bt)
            ws = B.workspace(B.pa_decode_workspace_size(sh, P), dev)
            fn = lambda: B.pa_decode(q, kc, vc, bt, cl, w.scale, out, lse, num_splits=P,  # noqa
                                     workspace=ws)
            fn()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):  # two calls per replay: graph launch cost halved
                fn()
                fn()
            for _ in range(5):
                g.replay()
            n = 30
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(n)]
            torch.cuda.synchronize()
            torch.cuda._sleep(1_000_000)
            for a, b in evs:
                a.record()
                g.replay()
                b.record()
            torch.cuda.synchronize()
            ms = statistics.fmean(a.elapsed_time(b) for a, b in evs) / 2
            gbs = alg / (ms / 1e3) / 1e9
            res[f"{name}_splits{P}"] = {"decode_ms": round(ms, 5), "alg_bytes": alg,
                                        "achieved_gbs": round(gbs, 1),
                                        "frac_of_measured_peak": round(gbs / peak, 4),
                                        "tokens_per_s": w.num_q_tokens / (ms / 1e3)}
        del kc, vc
        torch.cuda.empty_cache()
    res.update(run_secondary_varlen(args, dev, B, peak))
    res.update(run_secondary_int8(args, dev, B, peak))
    res.update(run_secondary_cascade(args, dev, B, peak))
    return res


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


def run_secondary_cascade(args, dev, B, peak):
    """Cascade (shared-prefix) decode against plain balanced decode on the
    ragged batch (30% share a 512-token prefix) and on a shared-prompt batch
    (128 sequences behind one 4096-token prompt)."""
    from paged_kv_decode_18_gb300 import workloads as W

    res = {}
    for name, make in (("ragged", W.ragged), ("shared_prompt", W.shared_prompt)):
        w = make(seed=args.seed)
        kc, vc = w.empty_pool(dev)
        B.pa_reshape_and_cache(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev), kc, vc)
        B.pa_reshape_and_cache(w.k_new.to(dev), w.v_new.to(dev), w.slot_new.to(dev), kc, vc)
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
            "cascade": lambda: B.pa_decode_cascade(q, kc, vc, bt, cl, sg, cu, mem, pl, mg,  # noqa
                                                   mp, w.scale, out, lse, workspace=wsc),
        }
        ub = unique_kv_bytes(w)
        for kind, fn in calls.items():
            fn()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
                fn()
            for _ in range(5):
                g.replay()
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(30)]
            torch.cuda.synchronize()
            torch.cuda._sleep(1_000_000)
            for a, b in evs:
                a.record()
                g.replay()
                b.record()
            torch.cuda.synchronize()
            ms = statistics.fmean(a.elapsed_time(b) for a, b in evs) / 2
            res[f"{name}_{kind}"] = {"call_ms": round(ms, 5), "unique_kv_bytes": ub,
                                     "unique_gbs": round(ub / (ms / 1e3) / 1e9, 1),
                                     "tokens_per_s": w.num_q_tokens / (ms / 1e3)}
        del kc, vc
        torch.cuda.empty_cache()
    return res


def run_secondary_int8(args, dev, B, peak):
    """Decode over the INT8 pool (quantised cache write, fused dequant): the
    engine batch rotated over the layer pools, the ragged and the long batch."""
    from paged_kv_decode_18_gb300 import workloads as W

    res = {}
    for name, make, nlayers in (("engine", W.engine, LAYERS), ("ragged", W.ragged, 1),
                                ("long", W.long, 1)):
        w = make(seed=args.seed)
        pools = []
        for _ in range(nlayers):
            kc, vc, ks, vs = w.empty_pool_i8(dev)
            B.pa_reshape_and_cache_int8(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev),
                                        kc, vc, ks, vs)
            B.pa_reshape_and_cache_int8(w.k_new.to(dev), w.v_new.to(dev), w.slot_new.to(dev),
                                        kc, vc, ks, vs)
            pools.append((kc, vc, ks, vs))
        q = w.q.to(dev)
        bt, cl = w.block_tables.to(dev), w.context_lens.to(dev)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        sh = B.shape_of(q, pools[0][0], bt)
        ws = B.workspace(B.pa_decode_int8_workspace_size(sh, 0), dev)

        def call(l):
            kc, vc, ks, vs = pools[l]
            B.pa_decode_int8(q, kc, vc, ks, vs, bt, cl, w.scale, out, lse, num_splits=0,
                             workspace=ws)
        per_replay = 4 if nlayers > 1 else 2
        call(0)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(per_replay):
                call(i % nlayers)
        for _ in range(5):
            g.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(30)]
        torch.cuda.synchronize()
        torch.cuda._sleep(1_000_000)
        for a, b in evs:
            a.record()
            g.replay()
            b.record()
        torch.cuda.synchronize()
        ms = statistics.fmean(a.elapsed_time(b) for a, b in evs) / per_replay
        alg = decode_algorithmic_bytes_int8(w)
        gbs = alg / (ms / 1e3) / 1e9
        res[f"{name}_int8"] = {"decode_ms": round(ms, 5), "alg_bytes": alg,
                               "achieved_gbs": round(gbs, 1),
                               "frac_of_measured_peak": round(gbs / peak, 4),
                               "tokens_per_s": w.num_q_tokens / (ms / 1e3),
                               "kv_format": "int8 + fp32 row scales"}
        del pools
        torch.cuda.empty_cache()
    return res


def attention_flops(w) -> int:
    """Useful flops of one call: 4 * D per (query row, head, visible key)."""
    n = 0
    for c, l in zip(w.context_lens.tolist(), w.q_lens.tolist()):
        n += sum(c - l + j + 1 for j in range(l)) if w.causal else l * c
    return n * 4 * w.head_dim * w.num_q_heads


def run_secondary_varlen(args, dev, B, peak):
    """Verify + chunked-prefill call (tensor cores) on the mixed workload."""
    from paged_kv_decode_18_gb300 import workloads as W

    w = W.mixed(seed=args.seed)
    kc, vc = w.empty_pool(dev)
    B.pa_reshape_and_cache(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev), kc, vc)
    B.pa_reshape_and_cache(w.k_new.to(dev), w.v_new.to(dev), w.slot_new.to(dev), kc, vc)
    q = w.q.to(dev)
    bt, cl, cu = w.block_tables.to(dev), w.context_lens.to(dev), w.cu_seqlens_q.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    sh = B.shape_of(q, kc, bt)
    ws = B.workspace(B.pa_decode_varlen_workspace_size(sh, q.shape[0], w.max_q_len), dev)
    fn = lambda: B.pa_decode_varlen(q, kc, vc, bt, cl, cu, w.max_q_len, w.scale, out, lse,  # noqa
                                    causal=True, workspace=ws)
    fn()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
        fn()
    for _ in range(5):
        g.replay()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(20)]
    torch.cuda.synchronize()
    torch.cuda._sleep(1_000_000)
    for a, b in evs:
        a.record()
        g.replay()
        b.record()
    torch.cuda.synchronize()
    ms = statistics.fmean(a.elapsed_time(b) for a, b in evs) / 2
    alg = decode_algorithmic_bytes(w)
    fl = attention_flops(w)
    gbs = alg / (ms / 1e3) / 1e9
    return {"mixed_varlen": {"call_ms": round(ms, 5), "alg_bytes": alg, "achieved_gbs": round(gbs, 1),
                             "frac_of_measured_peak": round(gbs / peak, 4), "useful_gflop": round(fl / 1e9, 3),
                             "achieved_tflops": round(fl / (ms / 1e3) / 1e12, 1),
                             "query_tokens_per_s": w.num_q_tokens / (ms / 1e3)}}


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------

def oracle_rate(seed: int, budget_s: float, max_steps: int | None = None,
                num_threads: int = 0):
    """Time the fp64 oracle on the engine workload: each step is the oracle's
    cache write of the new tokens plus paged attention over a sample of the
    sequences (num_threads 0 = all host cores). Returns (tokens/s, threads,
    description, steps, seqs/step)."""
    import numpy as np

    from oracle import oracle
    from paged_kv_decode_18_gb300 import workloads as W

    w = W.engine(seed=seed)
    kp = np.full(w.pool_shape(), W.POOL_SENTINEL_BITS, np.uint16)
    vp = kp.copy()
    oracle.reshape_and_cache(w.k_hist, w.v_hist, w.slot_hist, kp, vp, w.block_size)
    threads = oracle.max_threads() if num_threads <= 0 else num_threads

    def one(n_seqs):
        oracle.reshape_and_cache(w.k_new[:n_seqs], w.v_new[:n_seqs], w.slot_new[:n_seqs], kp, vp,
                                 w.block_size)
        oracle.paged_attention(w.q[:n_seqs], kp, vp, w.block_tables[:n_seqs],
                               w.context_lens[:n_seqs], w.cu_seqlens_q[:n_seqs + 1], w.scale,
                               num_threads=threads)

    t = time.perf_counter()
    one(w.num_seqs)
    full = time.perf_counter() - t
    n_seqs = w.num_seqs
    if max_steps is not None:
        per_step = budget_s / max(1, max_steps)
        n_seqs = max(1, min(w.num_seqs, int(w.num_seqs * per_step / max(full, 1e-6))))
    steps = 0
    tokens = 0
    t0 = time.perf_counter()
    while True:
        one(n_seqs)
        steps += 1
        tokens += n_seqs
        el = time.perf_counter() - t0
        if max_steps is not None and steps >= max_steps:
            break
        if max_steps is None and el >= budget_s and steps >= 3:
            break
    el = time.perf_counter() - t0
    desc = (f"fp64 oracle, engine workload: {steps} steps of cache write + paged attention "
            f"over {n_seqs} of 64 sequences (context 384), {threads} threads")
    return tokens / el, threads, desc, steps, n_seqs


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    budget = 120.0
    # warm-up steps, then exactly K timed steps sized to fit the budget
    oracle_rate(args.seed, 5.0, max_steps=max(3, args.warmup))
    rate, threads, desc, steps, n = oracle_rate(args.seed, budget, max_steps=args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * n / rate,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "num_seqs": 64, "context_len": 384,
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
    elif args.case == "ragged_int8":
        w = W.ragged(seed=args.seed)
    elif args.case == "shared_prompt":
        w = W.shared_prompt(seed=args.seed)
    else:
        w = W.make(args.case, seed=args.seed)
    int8 = args.case == "ragged_int8"
    if int8:
        kc, vc, ks, vs = w.empty_pool_i8(dev)
        B.pa_reshape_and_cache_int8(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev),
                                    kc, vc, ks, vs)
    else:
        kc, vc = w.empty_pool(dev)
        B.pa_reshape_and_cache(w.k_hist.to(dev), w.v_hist.to(dev), w.slot_hist.to(dev), kc, vc)
    k_new, v_new, slot_new = w.k_new.to(dev), w.v_new.to(dev), w.slot_new.to(dev)
    q = w.q.to(dev)
    bt, cl, cu = w.block_tables.to(dev), w.context_lens.to(dev), w.cu_seqlens_q.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
    sh = B.shape_of(q, kc, bt)
    varlen = args.case in ("mixed", "prefill")
    cascade = args.case == "shared_prompt"
    if varlen:
        ws = B.workspace(B.pa_decode_varlen_workspace_size(sh, q.shape[0], w.max_q_len), dev)
    elif int8:
        ws = B.workspace(B.pa_decode_int8_workspace_size(sh, args.splits), dev)
    elif cascade:
        sg, cg, mem, pl, mg, mp = W.cascade_groups(w)
        sg, cg, mem, pl = sg.to(dev), cg.to(dev), mem.to(dev), pl.to(dev)
        ws = B.workspace(B.pa_decode_cascade_workspace_size(sh, pl.shape[0], mem.numel(), mg,
                                                            mp), dev)
    else:
        ws = B.workspace(B.pa_decode_workspace_size(sh, args.splits), dev)

    def step():
        if int8:
            B.pa_reshape_and_cache_int8(k_new, v_new, slot_new, kc, vc, ks, vs)
            B.pa_decode_int8(q, kc, vc, ks, vs, bt, cl, w.scale, out, lse,
                             num_splits=args.splits, workspace=ws)
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
                      "alg_bytes": decode_algorithmic_bytes(w), "device_error": err}))
    return 1 if err else 0


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=["tiny", "engine", "ragged", "long", "mixed", "prefill",
                                       "ragged_int8", "shared_prompt"],
                    help="time one workload with eager calls (for profiling), nothing else")
    ap.add_argument("--splits", type=int, default=0, help="num_splits for --case decode runs")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

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

    r = run_ours(args, rank, world, dev)
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            rate, threads, desc, _, _ = oracle_rate(args.seed, 10.0)
            rate1, _, desc1, _, _ = oracle_rate(args.seed, 3.0, num_threads=1)
            cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                   "sample": desc, "value_1_thread": rate1, "sample_1_thread": desc1}
        traffic = traffic_for("engine")
        line = {
            "metric": METRIC,
            "value": r["value"],
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": r["ms_per_step"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "num_seqs": 64, "context_len": 384,
                       "global_batch": 64 * world, "parallelism": f"replicas x{world}",
                       "num_splits": 0,
                       "l2": f"inputs larger than L2: {LAYERS} layer caches of 100.7 MB "
                             "rotated per step"},
            "roofline": {"bound": "hbm", "achieved": round(r["achieved"], 1),
                         "peak": r["peak"], "unit": "GB/s",
                         "frac": round(r["achieved"] / r["peak"], 4), "traffic": traffic,
                         "kernel": "pa_decode (paged_decode_kernel + decode_fixup_kernel)",
                         "alg_bytes_per_launch": r["alg_bytes"],
                         "launch_ms": round(r["decode_ms"], 5),
                         "peak_source": f"{r['peak_kind']} hbm_gbs"},
            "cpu_baseline": cpu,
            "e2e": r["e2e"],
            "gpu_launches": r["launches"],
            "clocks": r["clocks"],
        }
        if "secondary" in r:
            line["secondary"] = r["secondary"]
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
