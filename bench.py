#!/usr/bin/env python3
"""Benchmark of one continuous-batching step of paged GQA attention on GB300.

A step is the whole hot path for every layer of the model: kv_append of all
new tokens (one per decode sequence plus the prefill chunk), paged decode
attention over every decode sequence's cache (split-K main + reduce), and a
chunked-prefill attention of the chunk over itself and its prior cache.

Default workload: the ragged continuous batch -- 32 layers, 32 query / 8 KV
heads, head_dim 128, bf16 cache in 16-token blocks, 128 decode sequences at
seeded log-uniform context in [128, 32768], plus one 2,048-token prefill chunk
over 4,096 cached tokens.  Every layer has its own pools (about 3.1 GB per
layer, far larger than L2), so no L2 flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Per layer the decode and the prefill run side by side on disjoint SMs (the
prefill's SM count picked by a short trial before warm-up; --side-by-side 0
runs them one after the other).

Prints one JSON line (rank 0).  `value` is achieved algorithmic HBM GB/s of
the whole step; decode tokens/s and prefill TFLOP/s ride along, with:
  roofline / prefill_roofline  the decode's and the prefill's own rates
                               against the measured peaks;
  side_by_side                 the split and each half's time alone;
  e2e                          the same step through the C ABI from pinned
                               host buffers, copies included;
  fp8_decode, mla_decode       the decode over an fp8 cache and over a
                               latent cache, each with its own roofline;
  decode_configs               the decode step of the 2,301-token and
                               32,001-token batches, and of the 16-sequence
                               65-token batch with the L2 flushed before
                               every timed step;
  cpu_baseline                 the oracle on a bounded sample, on all host
                               cores and (single_core) on one.
The `reference` arm times the fp64 CPU oracle on a bounded sample of the same
workload (the pages ship no runnable implementation of this path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_cache_104_gb300 import workloads as W  # noqa: E402

METRIC = "paged GQA decode attn: achieved HBM GB/s (% of GB300 peak); decode tokens/s"
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------- accounting
def step_accounting(w: W.Workload, lay: W.Layout):
    """Algorithmic bytes and flops of one step (all layers).

    decode: every stored K and V row of every decode sequence read once (the
            GQA group is resident), plus q read and out written;
    append: new K/V rows read and written once;
    prefill: the chunk's q read and out written, and the K/V of the sequence
            (prior + chunk tokens) read once; flops count causal pairs only:
            4 * D * Hq per visible (query, key) pair."""
    e, hq, hkv, d, L = w.elem_bytes, w.num_q_heads, w.num_kv_heads, w.head_dim, w.layers
    tokens = int(lay.seq_lens.to(torch.int64).sum())
    b = lay.num_decode_tokens
    dec = tokens * hkv * d * 2 * e + 2 * b * hq * d * e
    t = lay.slot_mapping.shape[0]
    app = 2 * t * hkv * d * 2 * e
    c, p = w.prefill_chunk, w.prefill_prior
    pre = 2 * c * hq * d * e + (p + c) * hkv * d * 2 * e if c else 0
    pairs = c * p + c * (c + 1) // 2
    flops = 4 * d * hq * pairs
    return {"decode_bytes_layer": dec, "append_bytes_layer": app, "prefill_bytes_layer": pre,
            "prefill_flops_layer": flops, "bytes_step": L * (dec + app + pre),
            "decode_tokens_step": b}


def measured_peaks():
    """(HBM GB/s, bf16 TFLOP/s sustained, source).  The sustained bf16 figure is
    the one for a kernel timed inside a long step, like the prefill here."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            bf16 = float(d.get("bf16_tflops_sustained") or d.get("bf16_tflops") or 0)
            return float(d["hbm_gbs"]), bf16, "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, 1700.0, "fallback"


def profiled_traffic(kernel: str, source: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel source as it is now (else None)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path)).get(kernel)
        src = open(os.path.join(ROOT, "paged_kv_cache_104_gb300", "csrc", source), "rb").read()
        if rec and rec.get("source_sha256") == hashlib.sha256(src).hexdigest():
            return rec.get("dram_bytes_per_launch_full_size")
    except Exception:
        return None
    return None


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling every 50 ms while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 9:
                self.samples.append(f)
        return False

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4)
                          if s[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


# --------------------------------------------------------------------------- oracle timing
def oracle_prepare(w, lay, n_dec_seqs: int, device="cpu"):
    """Inputs for the oracle sample: a layout holding the first n_dec_seqs
    decode sequences (same lengths as the full batch) and the prefill chunk,
    drawn from the seeded generator (on `device`, then copied to the host) and
    appended by the oracle's own scatter."""
    import oracle
    oracle.build()
    sub = W.make_layout(w, seq_lens_after=lay.seq_lens[:n_dec_seqs],
                        prefill=(w.prefill_prior, w.prefill_chunk))
    x = W.draw_layer(w, sub, 0, device=device)
    x = W.LayerInputs(*(t.to("cpu") for t in (x.q_decode, x.q_prefill, x.k_new, x.v_new,
                                               x.k_cache, x.v_cache)))
    oracle.kv_append(x.k_new, x.v_new, x.k_cache, x.v_cache, sub.slot_mapping)
    return sub, x


def oracle_sample_rates(w, sub, x, n_pre_rows: int):
    """Time the fp64 CPU oracle: decode of every sequence of `sub` (every head)
    and prefill of n_pre_rows evenly spaced chunk rows (every head).
    Returns (decode algorithmic bytes/s, prefill rows/s, description, seconds)."""
    import oracle
    e, hq, hkv, d = w.elem_bytes, w.num_q_heads, w.num_kv_heads, w.head_dim
    n_dec = sub.num_decode_tokens
    t0 = time.perf_counter()
    oracle.paged_decode(x.q_decode, x.k_cache, x.v_cache, sub.decode_block_table, sub.seq_lens,
                        w.scale)
    t_dec = time.perf_counter() - t0
    sample_tokens = int(sub.seq_lens.to(torch.int64).sum())
    dec_bytes = sample_tokens * hkv * d * 2 * e + 2 * n_dec * hq * d * e
    pre_rate, t_pre = None, 0.0
    if w.prefill_chunk and n_pre_rows:
        stride = max(1, w.prefill_chunk // n_pre_rows)
        rows = [(i, h) for i in list(range(0, w.prefill_chunk, stride))[:n_pre_rows]
                for h in range(hq)]
        bt = sub.block_table[sub.prefill_row]
        t0 = time.perf_counter()
        oracle.chunked_prefill(x.q_prefill, x.k_cache, x.v_cache, bt, w.prefill_prior, w.scale,
                               rows=rows)
        t_pre = time.perf_counter() - t0
        pre_rate = (len(rows) / hq) / t_pre
    desc = (f"one layer: decode of {n_dec} of the batch's sequences ({sample_tokens} cached "
            f"tokens, all {hq} heads) in {t_dec:.2f} s"
            + (f"; prefill of {n_pre_rows} evenly spaced chunk rows (all heads) in {t_pre:.2f} s"
               if pre_rate else "")
            + "; the full step (all layers, sequences and chunk rows) is extrapolated from "
              "these rates")
    return dec_bytes / t_dec, pre_rate, desc, t_dec + t_pre


def oracle_step_estimate(w, lay, acct, dec_rate, pre_rate):
    """Seconds the oracle would take for one full step, from sample rates."""
    t = w.layers * acct["decode_bytes_layer"] / dec_rate
    if w.prefill_chunk and pre_rate:
        t += w.layers * w.prefill_chunk / pre_rate
    return t


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# --------------------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws):
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
        return dist
    return None


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# --------------------------------------------------------------------------- reference arm
def run_reference(args, w, lay, acct):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    os.environ.setdefault("OMP_NUM_THREADS", str(cpu_cores()))
    import oracle
    oracle.build()
    threads = oracle.num_threads()
    times = []
    desc = ""
    sub, x = oracle_prepare(w, lay, args.ref_decode_seqs, device="cpu")
    for i in range(args.warmup + args.steps):
        dec_rate, pre_rate, desc, _ = oracle_sample_rates(w, sub, x, args.ref_prefill_rows)
        if i >= args.warmup:
            times.append(oracle_step_estimate(w, lay, acct, dec_rate, pre_rate))
    t = statistics.median(times)
    value = acct["bytes_step"] / t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description, "layers": w.layers},
        "decode_tokens_per_s": acct["decode_tokens_step"] / t,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": desc + " (per step; median over the timed steps)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- our arm
def graphs_of(step, L, nev, dev, stream):
    """Capture the step twice: a clean CUDA graph for the timed region, and one
    with event-record nodes around each layer's calls (nev per layer), replayed
    only after the timed region for the per-call breakdown.  Event nodes inside
    a graph break the kernel-to-kernel edges between layers and add a few
    microseconds per node, so the timed graph holds none.  Returns (clean,
    instrumented or None, its events)."""
    try:
        gev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(nev)]
               for _ in range(L)]
    except TypeError:
        gev = None
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graphs = []
    for ev in (None, gev) if gev is not None else (None,):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                step(ev, s=cap)
        graphs.append(g)
    stream.wait_stream(cap)
    for g in graphs:
        g.replay()
    torch.cuda.synchronize(dev)
    return graphs[0], (graphs[1] if len(graphs) > 1 else None), gev


def breakdown_events(g_ev, gev, step, L, nev, dev):
    """Replay the instrumented graph once (or run one eager step when this
    torch has no graph event nodes) and return its per-layer events."""
    if g_ev is not None:
        g_ev.replay()
        torch.cuda.synchronize(dev)
        return gev
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(L)]
    step(ev)
    torch.cuda.synchronize(dev)
    return ev


def run_fp8_decode(args, w, lay, inputs, dev, stream, dist, n):
    """Time the decode path over an fp8 (E4M3, per-KV-head scales) cache:
    per layer kv_append_fp8 of the decode tokens, then decode attention
    (split-K main + reduce), every layer with its own pools, as one CUDA
    graph per step.  Algorithmic bytes: the codes of every stored K and V row
    once, q read and out written (bf16), and the append (bf16 in, codes out)."""
    from paged_kv_cache_104_gb300 import binding as B

    L, hq, hkv, d = w.layers, w.num_q_heads, w.num_kv_heads, w.head_dim
    nd = lay.num_decode_tokens
    tokens = int(lay.seq_lens.to(torch.int64).sum())
    dec_bytes = tokens * hkv * d * 2 + 2 * nd * hq * d * 2
    app_bytes = nd * hkv * d * 2 * (2 + 1)
    pool_bytes = 2 * lay.num_blocks * hkv * w.block_size * d
    free, _ = torch.cuda.mem_get_info(dev)
    n_pools = min(L, max(2, int((free - 8 * 2 ** 30) // max(pool_bytes, 1))))
    if args.layer_pools > 0:
        n_pools = min(n_pools, args.layer_pools)
    scales = [tuple(t.to(dev) for t in W.fp8_scales(w, li)) for li in range(L)]
    pools = [(W.draw_fp8_pool(w, lay, scales[li][0], li, 0, device=dev),
              W.draw_fp8_pool(w, lay, scales[li][1], li, 1, device=dev)) for li in range(n_pools)]
    slot_dec = lay.slot_mapping[:nd].to(dev)
    bt = lay.decode_block_table.to(dev).contiguous()
    sl = lay.seq_lens.to(dev)
    msl = int(lay.seq_lens.max())
    wsp = B.decode_workspace(nd, hq, d, msl, device=dev)
    outs = [torch.empty_like(inputs[li].q_decode) for li in range(L)]

    def step(ev=None, s=None):
        s = stream if s is None else s
        for li in range(L):
            x = inputs[li]
            kc, vc = pools[li % n_pools]
            ks, vs = scales[li]
            B.kv_append_fp8(x.k_new[:nd], x.v_new[:nd], kc, vc, ks, vs, slot_dec, stream=s)
            if ev is not None:
                ev[li][0].record(s)
            B.paged_decode_attention_fp8(outs[li], x.q_decode, kc, vc, ks, vs, bt, sl, msl,
                                         w.scale, wsp, stream=s)
            if ev is not None:
                ev[li][1].record(s)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert B.get_device_error() == 0, "device error word set during the fp8 warm-up"
    graph, g_ev, gev = graphs_of(step, L, 2, dev, stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(dev)
    t0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    ms_step = max_over_ranks(dist, t0.elapsed_time(t1)) / args.steps
    assert B.get_device_error() == 0, "device error word set during the fp8 steps"
    gev = breakdown_events(g_ev, gev, step, L, 2, dev)
    dec_ms = sum(gev[li][0].elapsed_time(gev[li][1]) for li in range(L)) / L
    hbm_peak, _, peak_src = measured_peaks()
    # the timed step is L x (append + decode call) and nothing else: one
    # layer's time is the step's time over L
    layer_ms = ms_step / L
    leg_gbs = (dec_bytes + app_bytes) / (layer_ms / 1e3) / 1e9
    return {
        "what": "decode path over an fp8 E4M3 cache with per-KV-head scales: kv_append_fp8 of "
                "the decode tokens + decode attention (main + reduce), all layers, one CUDA graph",
        "ms_per_step": ms_step,
        "value": n * L * (dec_bytes + app_bytes) / (ms_step / 1e3) / 1e9, "unit": "GB/s",
        "decode_tokens_per_s": n * nd / (ms_step / 1e3),
        "layer_ms": layer_ms,
        "decode_ms_per_layer_events": dec_ms,
        "distinct_layer_pools": n_pools, "pool_gb_per_layer": pool_bytes / 1e9,
        "gpu_launches": args.steps * L * (2 + (1 if msl > 512 else 0)),
        "roofline": {
            "kernel": "kv_append_fp8 + paged_decode_attention_fp8 (split-K main + reduce), one "
                      "layer", "bound": "hbm",
            "achieved": leg_gbs, "peak": hbm_peak, "unit": "GB/s", "frac": leg_gbs / hbm_peak,
            "traffic": profiled_traffic("decode_fp8_kernel", "decode_fp8.cu"),
            "algorithmic_bytes_per_launch": dec_bytes + app_bytes,
            "timing": "one layer's append + decode call = the timed step over L (CUDA events "
                      "around the replays of a graph with no other work); "
                      "decode_ms_per_layer_events brackets the decode call alone in a separately "
                      "replayed graph with event nodes",
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback 6.8 TB/s",
        },
    }


def run_decode_config(args, name, dev, stream, dist, n):
    """Time the bf16 decode step of another configuration (no prefill chunk):
    per layer the fused append + paged decode (main + reduce), every layer
    with its own pools (as many as fit), one CUDA graph per step, inputs far
    larger than L2."""
    from paged_kv_cache_104_gb300 import binding as B

    w = W.WORKLOADS[name]
    lay = W.make_layout(w)
    acct = step_accounting(w, lay)
    L, hq, hkv, d = w.layers, w.num_q_heads, w.num_kv_heads, w.head_dim
    nd = lay.num_decode_tokens
    pool_bytes = 2 * lay.num_blocks * hkv * w.block_size * d * w.elem_bytes
    free, _ = torch.cuda.mem_get_info(dev)
    n_pools = min(L, max(2, int((free - 8 * 2 ** 30) // max(pool_bytes, 1))))
    if args.layer_pools > 0:
        n_pools = min(n_pools, args.layer_pools)
    xs = [W.draw_layer(w, lay, li + 1000 * dist_env()[1], device=dev, with_pool=li < n_pools)
          for li in range(L)]
    pools = [(xs[li].k_cache, xs[li].v_cache) for li in range(n_pools)]
    bt = lay.decode_block_table.to(dev).contiguous()
    sl = lay.seq_lens.to(dev)
    msl = int(lay.seq_lens.max())
    wsp = B.decode_workspace(nd, hq, d, msl, device=dev)
    outs = [torch.empty_like(xs[li].q_decode) for li in range(L)]

    def step(ev=None, s=None):
        s = stream if s is None else s
        for li in range(L):
            x = xs[li]
            kc, vc = pools[li % n_pools]
            if ev is not None:
                ev[li][0].record(s)
            B.paged_decode_attention_append(outs[li], x.q_decode, x.k_new, x.v_new, kc, vc, bt, sl,
                                            msl, w.scale, wsp, stream=s)
            if ev is not None:
                ev[li][1].record(s)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert B.get_device_error() == 0, f"device error word set during the {name} warm-up"
    graph, g_ev, gev = graphs_of(step, L, 2, dev, stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(dev)
    t0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    ms_step = max_over_ranks(dist, t0.elapsed_time(t1)) / args.steps
    assert B.get_device_error() == 0, f"device error word set during the {name} steps"
    gev = breakdown_events(g_ev, gev, step, L, 2, dev)
    ev_ms = sum(gev[li][0].elapsed_time(gev[li][1]) for li in range(L)) / L
    hbm_peak, _, peak_src = measured_peaks()
    # the timed step is L decode calls and nothing else: one call's average
    # duration is the step's time over L
    dec_ms = ms_step / L
    dec_gbs = acct["decode_bytes_layer"] / (dec_ms / 1e3) / 1e9
    return {
        "what": w.description + "; per layer the fused append + paged decode (main + reduce), "
                "all layers, one CUDA graph",
        "ms_per_step": ms_step,
        "value": n * acct["bytes_step"] / (ms_step / 1e3) / 1e9, "unit": "GB/s",
        "decode_tokens_per_s": n * nd / (ms_step / 1e3),
        "decode_ms_per_layer": dec_ms,
        "decode_ms_per_layer_events": ev_ms,
        "timing": "decode_ms_per_layer = the timed step over L (the step is L decode calls, one "
                  "CUDA graph with no other nodes); decode_ms_per_layer_events brackets each call "
                  "in a separately replayed graph with event nodes",
        "cached_tokens": int(lay.seq_lens.sum()),
        "distinct_layer_pools": n_pools, "pool_gb_per_layer": pool_bytes / 1e9,
        "gpu_launches": args.steps * L * (2 if msl > 512 else 1),
        "roofline": {
            "kernel": "paged_decode_attention (split-K main + reduce)", "bound": "hbm",
            "achieved": dec_gbs, "peak": hbm_peak, "unit": "GB/s", "frac": dec_gbs / hbm_peak,
            "algorithmic_bytes_per_launch": acct["decode_bytes_layer"],
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback 6.8 TB/s",
        },
    }


def run_flushed_decode(args, name, dev, stream, dist, n):
    """Time the bf16 decode step of a configuration whose cache fits in L2
    (the 16-sequence batch at 65 tokens holds 4.3 MB of keys and values, the
    L2 129 MB): per layer the fused append + paged decode, every timed step
    preceded by pkv_l2_flush, which reads a buffer four times the L2's size,
    so the step reads its cache from HBM.  Only the step is timed (CUDA events
    right around it); the median over the timed steps is reported."""
    from paged_kv_cache_104_gb300 import binding as B

    w = W.WORKLOADS[name]
    lay = W.make_layout(w)
    acct = step_accounting(w, lay)
    L, hq, d = w.layers, w.num_q_heads, w.head_dim
    nd = lay.num_decode_tokens
    xs = [W.draw_layer(w, lay, li + 1000 * dist_env()[1], device=dev) for li in range(L)]
    bt = lay.decode_block_table.to(dev).contiguous()
    sl = lay.seq_lens.to(dev)
    msl = int(lay.seq_lens.max())
    wsp = B.decode_workspace(nd, hq, d, msl, device=dev)
    outs = [torch.empty_like(xs[li].q_decode) for li in range(L)]
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2 ** 20)
    flush = torch.empty((4 * l2 + 15) // 16 * 16, dtype=torch.uint8, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)

    def step():
        for li in range(L):
            x = xs[li]
            B.paged_decode_attention_append(outs[li], x.q_decode, x.k_new, x.v_new, x.k_cache,
                                            x.v_cache, bt, sl, msl, w.scale, wsp, stream=stream)

    iters = max(args.steps, 50)
    for _ in range(max(args.warmup, 3)):
        B.l2_flush(flush, sink, stream=stream)
        step()
    torch.cuda.synchronize(dev)
    assert B.get_device_error() == 0, f"device error word set during the {name} warm-up"
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters)]
    barrier(dist)
    torch.cuda.synchronize(dev)
    for e0, e1 in ev:
        B.l2_flush(flush, sink, stream=stream)
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    assert B.get_device_error() == 0, f"device error word set during the {name} steps"
    ms_step = max_over_ranks(dist, statistics.median(e0.elapsed_time(e1) for e0, e1 in ev))
    hbm_peak, _, peak_src = measured_peaks()
    dec_gbs = L * acct["decode_bytes_layer"] / (ms_step / 1e3) / 1e9
    return {
        "what": w.description + "; per layer the fused append + paged decode, the L2 flushed "
                "before every timed step",
        "ms_per_step": ms_step, "timing": f"median of {iters} steps, CUDA events around each",
        "value": n * acct["bytes_step"] / (ms_step / 1e3) / 1e9, "unit": "GB/s",
        "decode_tokens_per_s": n * nd / (ms_step / 1e3),
        "cached_tokens": int(lay.seq_lens.sum()),
        "l2": f"flushed before every timed step: pkv_l2_flush reads {flush.numel() / 1e6:.0f} MB "
              f"(4x the {l2 / 1e6:.0f} MB L2), outside the events",
        "gpu_launches": iters * L * (2 if msl > 512 else 1),
        "roofline": {
            "kernel": "paged_decode_attention (fused append; one launch at this length)",
            "bound": "hbm", "achieved": dec_gbs, "peak": hbm_peak, "unit": "GB/s",
            "frac": dec_gbs / hbm_peak,
            "algorithmic_bytes_per_launch": acct["decode_bytes_layer"],
            "note": "a 4.3 MB launch is latency-bound: launch, the walk's prologue and one "
                    "stage of HBM latency dominate; reported, not a bandwidth target",
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback 6.8 TB/s",
        },
    }


def run_mla_decode(args, w, lay, dev, stream, dist, n):
    """Time decode over a latent (MLA-style) cache on the decode batch of the
    workload: per layer one decode call that appends the decode tokens'
    latents (in the query absorption's launch), then attends over the
    latents, merges the split partials and up-projects, every layer with its
    own pool, as one CUDA graph.
    Algorithmic bytes: every stored latent once, the two projections, q read
    and out written, and the append."""
    from paged_kv_cache_104_gb300 import binding as B

    L, hq, d, r = w.layers, w.num_q_heads, w.head_dim, 128
    lw = W.Workload("latent_" + w.name, torch.bfloat16, L, hq, 1, d, w.block_size, w.num_seqs,
                    seed=w.seed, context=w.context, context_loguniform=w.context_loguniform)
    llay = W.make_layout(lw, prefill=(0, 0))
    nd = llay.num_decode_tokens
    tokens = int(llay.seq_lens.to(torch.int64).sum())
    dec_bytes = tokens * r * 2 + 2 * hq * d * r * 2 + 2 * nd * hq * d * 2
    app_bytes = nd * r * 2 * 2
    pool_bytes = llay.num_blocks * w.block_size * r * 2
    free, _ = torch.cuda.mem_get_info(dev)
    n_pools = min(L, max(2, int((free - 8 * 2 ** 30) // max(pool_bytes, 1))))
    if args.layer_pools > 0:
        n_pools = min(n_pools, args.layer_pools)
    xs = [W.draw_latent(lw, llay, r, layer=li, device=dev) for li in range(L)]
    pools = [xs[li].pool for li in range(n_pools)]
    for li in range(L):
        xs[li].pool = None
    bt = llay.decode_block_table.to(dev).contiguous()
    sl = llay.seq_lens.to(dev)
    msl = int(llay.seq_lens.max())
    wsp = B.mla_workspace(nd, hq, r, msl, device=dev)
    outs = [torch.empty_like(xs[li].q) for li in range(L)]

    def step(ev=None, s=None):
        s = stream if s is None else s
        for li in range(L):
            x = xs[li]
            c = pools[li % n_pools]
            if ev is not None:
                ev[li][0].record(s)
            # one call: the decode tokens' latents appended, then the decode
            B.mla_decode_attention(outs[li], x.q, x.w_k, x.w_v, c, bt, sl, msl, lw.scale, wsp,
                                   stream=s, c_new=x.c_new)
            if ev is not None:
                ev[li][1].record(s)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert B.get_device_error() == 0, "device error word set during the latent warm-up"
    graph, g_ev, gev = graphs_of(step, L, 2, dev, stream)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(dev)
    t0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    ms_step = max_over_ranks(dist, t0.elapsed_time(t1)) / args.steps
    assert B.get_device_error() == 0, "device error word set during the latent steps"
    gev = breakdown_events(g_ev, gev, step, L, 2, dev)
    dec_ms = sum(gev[li][0].elapsed_time(gev[li][1]) for li in range(L)) / L
    hbm_peak, _, peak_src = measured_peaks()
    # the timed step is L decode calls (each appending its tokens' latents)
    layer_ms = ms_step / L
    leg_gbs = (dec_bytes + app_bytes) / (layer_ms / 1e3) / 1e9
    return {
        "what": "decode over a latent (MLA-style) cache, rank 128, 32 query heads with per-head "
                "up-projections: per layer one decode call (append the decode tokens' latents "
                "and absorb the queries, attend over the latents, merge + up-project), all "
                "layers, one CUDA graph",
        "ms_per_step": ms_step,
        "value": n * L * (dec_bytes + app_bytes) / (ms_step / 1e3) / 1e9, "unit": "GB/s",
        "decode_tokens_per_s": n * nd / (ms_step / 1e3),
        "layer_ms": layer_ms,
        "decode_ms_per_layer_events": dec_ms,
        "distinct_layer_pools": n_pools, "pool_gb_per_layer": pool_bytes / 1e9,
        # per layer: append + query absorption, attention, merge + up-projection
        "gpu_launches": args.steps * L * 3,
        "roofline": {
            "kernel": "mla_decode_attention_append (latent append + query absorption, tcgen05 "
                      "attention over the latents, fused merge and up-projection), one layer",
            "bound": "hbm",
            "achieved": leg_gbs, "peak": hbm_peak, "unit": "GB/s", "frac": leg_gbs / hbm_peak,
            "traffic": profiled_traffic("decode_mla_kernel", "decode_mla.cu"),
            "algorithmic_bytes_per_launch": dec_bytes + app_bytes,
            "timing": "one layer's call = the timed step over L (CUDA events around the replays "
                      "of a graph with no other work); decode_ms_per_layer_events brackets each "
                      "call in a separately replayed graph with event nodes",
            "traffic_note": "the call is three launches; traffic is the DRAM bytes of its "
                            "attention launch alone, captured at this size (the absorption and "
                            "the merge read W_K, W_V, q and the partials: a few MB more)",
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback 6.8 TB/s",
        },
    }


def run_ours(args, w, lay, acct):
    from paged_kv_cache_104_gb300 import binding as B

    ws, rank, local = dist_env()
    dist = init_dist(ws)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the CUDA path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.load()
    stream = torch.cuda.current_stream(dev)

    L = w.layers
    hq, hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
    # distinct pools per layer if they fit, else cycle as many as fit (>= 2)
    pool_bytes = 2 * lay.num_blocks * hkv * w.block_size * d * w.elem_bytes
    free, _ = torch.cuda.mem_get_info(dev)
    n_pools = L if args.layer_pools <= 0 else min(L, args.layer_pools)
    fit = int((free - 8 * 2 ** 30) // max(pool_bytes, 1))
    if fit < n_pools:
        n_pools = max(2, fit)
    pools, inputs = [], []
    for li in range(L):
        x = W.draw_layer(w, lay, li + 1000 * rank, device=dev, with_pool=li < n_pools)
        if li < n_pools:
            pools.append((x.k_cache, x.v_cache))
            x.k_cache = x.v_cache = None
        inputs.append(x)
    slot = lay.slot_mapping.to(dev)
    bt_dec = lay.decode_block_table.to(dev).contiguous()
    seq_lens = lay.seq_lens.to(dev)
    bt_pre = lay.block_table[lay.prefill_row].to(dev).contiguous() if w.prefill_chunk else None
    max_seq = int(lay.seq_lens.max())
    wsp = B.decode_workspace(lay.num_decode_tokens, hq, d, max_seq, device=dev)
    out_dec = [torch.empty_like(inputs[li].q_decode) for li in range(L)]
    out_pre = [torch.empty_like(inputs[li].q_prefill) for li in range(L)]
    split_launch = 2 if max_seq > 512 else 1  # decode main (+ reduce when any sequence splits)

    nd = lay.num_decode_tokens
    fused = args.fused_append and w.dtype == torch.bfloat16 and w.head_dim == 128
    k_new_dec = [inputs[li].k_new[:nd] for li in range(L)]
    v_new_dec = [inputs[li].v_new[:nd] for li in range(L)]
    k_new_pre = [inputs[li].k_new[nd:] for li in range(L)]
    v_new_pre = [inputs[li].v_new[nd:] for li in range(L)]
    slot_pre = slot[nd:]
    # decode and prefill of a layer side by side on disjoint SMs (the prefill
    # as persistent CTAs on prefill_sms SMs, the decode on the rest)
    side = bool(args.side_by_side and fused and w.prefill_chunk)
    split = {"prefill_sms": int(args.prefill_sms)}

    def step(ev=None, s=None, serial=False):
        for li in range(L):
            layer(li, ev, s, serial)

    def layer(li, ev=None, s=None, serial=False):
        s = stream if s is None else s
        if True:
            x = inputs[li]
            kc, vc = pools[li % n_pools]
            if side and not serial:
                # one call: it appends the chunk's tokens, then runs the decode
                # (appending its tokens) and the prefill side by side
                if ev is not None:
                    ev[li][0].record(s)
                B.decode_prefill_attention(out_dec[li], x.q_decode, k_new_dec[li], v_new_dec[li],
                                           kc, vc, bt_dec, seq_lens, max_seq, out_pre[li],
                                           x.q_prefill, bt_pre, w.prefill_prior, w.scale, wsp,
                                           prefill_sms=split["prefill_sms"], stream=s,
                                           chunk_k_new=k_new_pre[li], chunk_v_new=v_new_pre[li],
                                           chunk_slots=slot_pre)
                if ev is not None:
                    ev[li][1].record(s)
                    ev[li][2].record(s)
                return
            if fused:
                # decode tokens are appended inside the decode launch; the
                # prefill chunk's tokens by kv_append
                if w.prefill_chunk:
                    B.kv_append(k_new_pre[li], v_new_pre[li], kc, vc, slot_pre, stream=s)
                if ev is not None:
                    ev[li][0].record(s)
                B.paged_decode_attention_append(out_dec[li], x.q_decode, k_new_dec[li],
                                                v_new_dec[li], kc, vc, bt_dec, seq_lens, max_seq,
                                                w.scale, wsp, stream=s)
            else:
                B.kv_append(x.k_new, x.v_new, kc, vc, slot, stream=s)
                if ev is not None:
                    ev[li][0].record(s)
                B.paged_decode_attention(out_dec[li], x.q_decode, kc, vc, bt_dec, seq_lens,
                                         max_seq, w.scale, wsp, stream=s)
            if ev is not None:
                ev[li][1].record(s)
            if w.prefill_chunk:
                B.chunked_prefill_attention(out_pre[li], x.q_prefill, kc, vc, bt_pre,
                                            w.prefill_prior, w.scale, stream=s)
                if ev is not None:
                    ev[li][2].record(s)

    if side and split["prefill_sms"] <= 0:
        # pick the split: a short eager run of the whole step per candidate
        # (outside the timed region); the decode needs far fewer SMs than the
        # GPU has to stream the cache, the prefill's time falls with its SMs
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        trials = {}

        def trial(cand):
            if cand in trials or not 1 <= cand < nsm:
                return
            split["prefill_sms"] = cand
            step()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            trials[cand] = e0.elapsed_time(e1)

        # a coarse sweep, then every count within 3 of the best one
        for cand in sorted({max(4, nsm * f // 64) for f in (8, 10, 12, 14, 16, 18, 20, 24)}):
            trial(cand)
        best = min(trials, key=trials.get)
        for cand in range(best - 3, best + 4):
            trial(cand)
        split["prefill_sms"] = min(trials, key=trials.get)
        split["trials_ms"] = {str(k): round(v, 3) for k, v in sorted(trials.items())}
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert B.get_device_error() == 0, "device error word set during warm-up"
    graph = None
    if args.graph:
        # one CUDA graph per step (all layers), with no event nodes; the
        # per-call breakdown comes from a second, instrumented graph replayed
        # after the timed region
        graph, g_ev, graph_events = graphs_of(step, L, 3, dev, stream)
        graph.replay()
        torch.cuda.synchronize(dev)

    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(L)]
           for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for k in range(args.steps):
            if graph is not None:
                graph.replay()
            else:
                step(evs[k])
        t_end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(dist)
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(dist, total_ms)
    assert B.get_device_error() == 0, "device error word set during the timed steps"
    if graph is not None:
        # the per-call breakdown: one replay of the instrumented graph (or,
        # without graph event nodes in this torch, one eager step)
        evs = [breakdown_events(g_ev, graph_events, step, L, 3, dev)]
        assert B.get_device_error() == 0, "device error word set during the breakdown replay"
    nsteps_ev = len(evs)
    dec_ms = [evs[k][li][0].elapsed_time(evs[k][li][1]) for k in range(nsteps_ev) for li in range(L)]
    pre_ms = ([evs[k][li][1].elapsed_time(evs[k][li][2]) for k in range(nsteps_ev)
               for li in range(L)] if w.prefill_chunk else [])
    ser_dec_ms = None
    if side:
        # in the timed steps the decode and the prefill of a layer overlap,
        # and the decode spans the pair, so the decode's rate over the timed
        # region is its bytes over a layer's time.  Each half's time alone
        # comes from one serial step (decode, then prefill, each on the whole
        # GPU) right after, and each half's span inside the pair from one
        # more step with the span record.
        ev_ser = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(L)]
        step(ev_ser, serial=True)
        torch.cuda.synchronize(dev)
        assert B.get_device_error() == 0, "device error word set during the serial step"
        ser_dec_ms = [ev_ser[li][0].elapsed_time(ev_ser[li][1]) for li in range(L)]
        pre_ms = [ev_ser[li][1].elapsed_time(ev_ser[li][2]) for li in range(L)]
        # each half's span inside the pair: one eager step with the kernels'
        # %globaltimer records (earliest CTA start, latest CTA end per grid)
        spans = torch.tensor([[-1, 0, -1, 0]] * L, dtype=torch.int64, device=dev)
        for li in range(L):
            B.set_span_buffer(spans[li])
            layer(li)
        B.set_span_buffer(None)
        torch.cuda.synchronize(dev)
        assert B.get_device_error() == 0, "device error word set during the span step"
        sp = spans.cpu().tolist()
        in_pair = {
            "prefill_ms": statistics.median((r[1] - r[0]) / 1e6 for r in sp),
            "decode_main_ms": statistics.median((r[3] - r[2]) / 1e6 for r in sp),
            "decode_start_after_prefill_start_us": statistics.median((r[2] - r[0]) / 1e3 for r in sp),
            "prefill_end_before_decode_end_us": statistics.median((r[3] - r[1]) / 1e3 for r in sp),
            "how": "medians over the layers of one eager step after the timed region; each "
                   "kernel records its CTAs' earliest start and latest end (%globaltimer, "
                   "pkv_set_span_buffer); the decode's split merge runs after both",
        }
    ms_step = total_ms / args.steps
    n = ws
    value = n * acct["bytes_step"] / (ms_step / 1e3) / 1e9
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    dec_avg = sum(dec_ms) / len(dec_ms)   # event brackets (the breakdown)
    if side and graph is not None:
        # the timed graph is L side-by-side calls (each appends the chunk's
        # keys and values, then runs the pair) and nothing else: a layer's
        # time is the step's over L
        roof_ms = ms_step / L
    else:
        roof_ms = dec_avg
    dec_gbs = acct["decode_bytes_layer"] / (roof_ms / 1e3) / 1e9
    traffic = profiled_traffic("decode_mma_kernel", "decode_mma.cu")
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
        "data": "synthetic",
        "config": {
            "workload": w.name, "description": w.description, "layers": L,
            "decode_seqs": lay.num_decode_tokens, "cached_tokens": int(lay.seq_lens.sum()),
            "prefill_chunk": w.prefill_chunk, "prefill_prior": w.prefill_prior,
            "distinct_layer_pools": n_pools, "pool_gb_per_layer": pool_bytes / 1e9,
            "l2": "inputs larger than L2: every layer has its own pools, each far larger than L2",
            "parallelism": f"replicas x{n} (independent batches, no collective)",
            "bytes_per_step": acct["bytes_step"],
        },
        "decode_tokens_per_s": n * acct["decode_tokens_step"] / (ms_step / 1e3),
        "decode_gbs": dec_gbs,
        "decode_hbm_frac": dec_gbs / hbm_peak,
        "prefill_tflops": (acct["prefill_flops_layer"] / (sum(pre_ms) / len(pre_ms) / 1e3) / 1e12
                           if pre_ms else None),
        "prefill_ms_per_layer": sum(pre_ms) / len(pre_ms) if pre_ms else None,
        "decode_ms_per_layer": roof_ms,
        "decode_ms_per_layer_events": dec_avg,
        "roofline": {
            "kernel": "paged_decode_attention (split-K main + reduce)",
            "bound": "hbm", "achieved": dec_gbs, "peak": hbm_peak, "unit": "GB/s",
            "frac": dec_gbs / hbm_peak, "traffic": traffic,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
            else "fallback 6.8 TB/s",
        },
        "prefill_roofline": ({
            "kernel": "chunked_prefill_attention (tcgen05, two heads per CTA)",
            "bound": "tensor", "achieved": acct["prefill_flops_layer"] / (sum(pre_ms) / len(pre_ms) / 1e3) / 1e12,
            "peak": bf16_peak, "unit": "TFLOP/s",
            "frac": acct["prefill_flops_layer"] / (sum(pre_ms) / len(pre_ms) / 1e3) / 1e12 / bf16_peak,
            "traffic": profiled_traffic("prefill_pair_kernel", "prefill_pair.cu"),
            "peak_source": ("measured (MEASURED_PEAKS.json bf16_tflops_sustained)" if peak_src == "measured"
                            else "fallback 1.7 PFLOP/s sustained"),
        } if pre_ms else None),
        "clocks": clk.summary(),
        "gpu_launches": args.steps * L * ((0 if fused and not w.prefill_chunk else 1) + split_launch
                                          + (1 if w.prefill_chunk else 0)),
        "mode": {"fused_append": bool(fused), "cuda_graph": graph is not None,
                 "side_by_side": side},
    }
    if side:
        nsm = torch.cuda.get_device_properties(dev).multi_processor_count
        ser_dec = sum(ser_dec_ms) / len(ser_dec_ms)
        line["side_by_side"] = {
            "what": "per layer, the decode (fused append, main + reduce) and the chunk's prefill run "
                    "at the same time on disjoint SMs: the prefill as persistent CTAs on prefill_sms "
                    "SMs, the decode as their programmatic dependent on the rest",
            "prefill_sms": split["prefill_sms"], "decode_sms": nsm - split["prefill_sms"],
            "split_trials_ms_per_step": split.get("trials_ms"),
            "layer_ms": roof_ms,
            "pair_ms_per_layer_events": dec_avg,
            # from the previous layer's end event to this layer's start event
            # (instrumented replay): the gap between calls
            "between_calls_ms_events": (
                sum(evs[0][li - 1][2].elapsed_time(evs[0][li][0]) for li in range(1, L)) / (L - 1)
                if L > 1 else None),
            "decode_ms_per_layer_alone": ser_dec,
            "decode_gbs_alone": acct["decode_bytes_layer"] / (ser_dec / 1e3) / 1e9,
            "prefill_ms_per_layer_alone": line["prefill_ms_per_layer"],
            "in_pair": in_pair,
        }
        line["roofline"]["note"] = (
            "the decode runs side by side with the prefill and spans the pair; achieved = the "
            "decode's bytes / one layer's time, which is the timed step over L (one CUDA graph "
            "with no event nodes: per layer one side-by-side call, which also appends the chunk's "
            "keys and values), a lower bound on the decode's own rate" if graph is not None else
            "the decode runs side by side with the prefill and spans the pair; achieved = the "
            "decode's bytes / the event time of the pair (a lower bound on its own rate)")
        if line["prefill_roofline"]:
            line["prefill_roofline"]["note"] = ("prefill measured alone, on all SMs, in one serial "
                                                "step right after the timed region")

    # ---- end to end through the C ABI with host buffers (pinned), same step
    if args.e2e_steps > 0:
        h_in = []
        h2d = 0
        for li in range(L):
            x = inputs[li]
            hb = [t.to("cpu").pin_memory() for t in (x.q_decode, x.q_prefill, x.k_new, x.v_new)]
            h2d += sum(t.numel() * t.element_size() for t in hb)
            h_in.append(hb)
        h_meta = [lay.slot_mapping.pin_memory(), lay.decode_block_table.contiguous().pin_memory(),
                  lay.seq_lens.pin_memory()]
        if w.prefill_chunk:
            h_meta.append(lay.block_table[lay.prefill_row].contiguous().pin_memory())
        h2d += sum(t.numel() * t.element_size() for t in h_meta)
        d_meta = [slot, bt_dec, seq_lens] + ([bt_pre] if w.prefill_chunk else [])
        h_out = [(torch.empty_like(out_dec[li], device="cpu").pin_memory(),
                  torch.empty_like(out_pre[li], device="cpu").pin_memory()) for li in range(L)]
        d2h = sum(a.numel() * a.element_size() + b.numel() * b.element_size() for a, b in h_out)

        # layer-pipelined: host->device copies of layer l+1's inputs and the
        # device->host copy of layer l-1's outputs run on two copy streams
        # while layer l computes
        h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(L)]
        ev_done = [torch.cuda.Event() for _ in range(L)]

        def e2e_step(s=None):
            # a step's copies start after the previous step's kernels (its
            # input buffers are reused) and after the timer's start event
            s = stream if s is None else s
            h2d_s.wait_stream(s)
            d2h_s.wait_stream(s)
            with torch.cuda.stream(h2d_s):
                for hsrc, dst in zip(h_meta, d_meta):
                    dst.copy_(hsrc, non_blocking=True)
                for li in range(L):
                    x = inputs[li]
                    for hsrc, dst in zip(h_in[li], (x.q_decode, x.q_prefill, x.k_new, x.v_new)):
                        dst.copy_(hsrc, non_blocking=True)
                    ev_in[li].record(h2d_s)
            for li in range(L):
                s.wait_event(ev_in[li])
                layer(li, s=s)
                ev_done[li].record(s)
            with torch.cuda.stream(d2h_s):
                for li in range(L):
                    d2h_s.wait_event(ev_done[li])
                    h_out[li][0].copy_(out_dec[li], non_blocking=True)
                    h_out[li][1].copy_(out_pre[li], non_blocking=True)
            s.wait_stream(d2h_s)
            s.wait_stream(h2d_s)

        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2e_step()
        torch.cuda.synchronize(dev)
        e2e_graph = None
        if graph is not None:
            # the same step (copies, calls, copies back) captured as one CUDA
            # graph, as the timed step is: every replay copies the inputs in
            # from pinned host memory and the outputs back out
            e2e_graph = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):
                with torch.cuda.graph(e2e_graph, stream=cap):
                    e2e_step(cap)
            stream.wait_stream(cap)
            e2e_graph.replay()
            torch.cuda.synchronize(dev)
        barrier(dist)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            if e2e_graph is not None:
                e2e_graph.replay()
            else:
                e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = max_over_ranks(dist, e0.elapsed_time(e1)) / args.e2e_steps
        # the same steps with eager launches (reported beside the graph's)
        eager_ms = None
        if e2e_graph is not None:
            barrier(dist)
            e0.record(stream)
            for _ in range(args.e2e_steps):
                e2e_step()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            eager_ms = max_over_ranks(dist, e0.elapsed_time(e1)) / args.e2e_steps
        line["e2e"] = {"value": n * acct["bytes_step"] / (e_ms / 1e3) / 1e9, "unit": "GB/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e_ms, "steps": args.e2e_steps,
                       "eager_ms_per_step": eager_ms,
                       "how": ("the C ABI calls and the copies captured as one CUDA graph per step "
                               "(replayed like the timed step); " if e2e_graph is not None else
                               "eager launches through the C ABI; ") +
                              "per layer, pinned host->device copies of its inputs and "
                              "device->host copies of its outputs on two copy streams, overlapped "
                              "with the other layers' kernels"}

    # ---- fp8 (E4M3) cache variant of the decode path: append + decode + reduce
    if args.fp8_decode and w.head_dim == 128 and w.dtype == torch.bfloat16:
        del pools
        torch.cuda.empty_cache()
        line["fp8_decode"] = run_fp8_decode(args, w, lay, inputs, dev, stream, dist, n)

    # ---- latent (MLA-style) cache variant of the decode path
    if args.mla_decode and w.head_dim == 128 and w.num_q_heads == 32 and w.dtype == torch.bfloat16:
        torch.cuda.empty_cache()
        line["mla_decode"] = run_mla_decode(args, w, lay, dev, stream, dist, n)

    # ---- the decode step of the other multi-layer configurations
    if args.other_configs and w.name == "ragged_prefill":
        torch.cuda.empty_cache()
        line["decode_configs"] = {}
        for name in ("llama8b_decode", "long_context"):
            line["decode_configs"][name] = run_decode_config(args, name, dev, stream, dist, n)
            torch.cuda.empty_cache()
        line["decode_configs"]["toy_decode"] = run_flushed_decode(args, "toy_decode", dev,
                                                                  stream, dist, n)
        torch.cuda.empty_cache()

    # ---- the oracle on this host's cores, bounded sample, rank 0 at N=1 only
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        pools = None
        del pools, inputs, out_dec, out_pre
        torch.cuda.empty_cache()
        os.environ.setdefault("OMP_NUM_THREADS", str(cpu_cores()))
        import oracle
        sub, xs = oracle_prepare(w, lay, args.cpu_decode_seqs, device=dev)
        dec_rate, pre_rate, desc, spent = oracle_sample_rates(w, sub, xs, args.cpu_prefill_rows)
        t_cpu = oracle_step_estimate(w, lay, acct, dec_rate, pre_rate)
        line["cpu_baseline"] = {"value": acct["bytes_step"] / t_cpu / 1e9, "unit": "GB/s",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": desc, "seconds": spent}
        # the same oracle on one core, on a smaller sample of the same step
        all_threads = oracle.num_threads()
        oracle.set_threads(1)
        sub1, xs1 = oracle_prepare(w, lay, args.cpu_single_decode_seqs, device=dev)
        dec1, pre1, desc1, spent1 = oracle_sample_rates(w, sub1, xs1, args.cpu_single_prefill_rows)
        oracle.set_threads(all_threads)
        t1 = oracle_step_estimate(w, lay, acct, dec1, pre1)
        line["cpu_baseline"]["single_core"] = {
            "value": acct["bytes_step"] / t1 / 1e9, "unit": "GB/s", "cores": 1,
            "sample": desc1, "seconds": spent1}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ragged_prefill", choices=sorted(W.WORKLOADS))
    ap.add_argument("--layer-pools", type=int, default=0,
                    help="distinct layer pools to allocate (0 = one per layer); the step always "
                         "runs every layer, cycling the pools")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--fused-append", type=int, default=1,
                    help="1: decode tokens are appended inside the decode launch")
    ap.add_argument("--side-by-side", type=int, default=1,
                    help="1: each layer's decode and prefill run at the same time on disjoint SMs")
    ap.add_argument("--prefill-sms", type=int, default=0,
                    help="SMs for the prefill when side by side (0: pick by a short trial)")
    ap.add_argument("--graph", type=int, default=1,
                    help="1: replay the whole step as one captured CUDA graph")
    ap.add_argument("--fp8-decode", type=int, default=1,
                    help="1: also time the decode path over an fp8 (E4M3) cache (reported "
                         "under fp8_decode, after the bf16 step)")
    ap.add_argument("--mla-decode", type=int, default=1,
                    help="1: also time decode over a latent (MLA-style) cache (reported under "
                         "mla_decode)")
    ap.add_argument("--other-configs", type=int, default=1,
                    help="also time the decode step of the 2,301-token and 32,001-token "
                         "batches (decode_configs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-decode-seqs", type=int, default=128,
                    help="decode sequences in the oracle sample of cpu_baseline")
    ap.add_argument("--cpu-prefill-rows", type=int, default=256,
                    help="chunk rows in the oracle sample of cpu_baseline")
    ap.add_argument("--cpu-single-decode-seqs", type=int, default=16,
                    help="decode sequences in the one-core oracle sample of cpu_baseline")
    ap.add_argument("--cpu-single-prefill-rows", type=int, default=32,
                    help="chunk rows in the one-core oracle sample of cpu_baseline")
    ap.add_argument("--ref-decode-seqs", type=int, default=16,
                    help="decode sequences per step of the reference (oracle) arm")
    ap.add_argument("--ref-prefill-rows", type=int, default=32,
                    help="chunk rows per step of the reference (oracle) arm")
    args = ap.parse_args()
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    w = W.WORKLOADS[args.workload]
    lay = W.make_layout(w)
    acct = step_accounting(w, lay)
    if args.impl == "reference":
        return run_reference(args, w, lay, acct)
    return run_ours(args, w, lay, acct)


if __name__ == "__main__":
    sys.exit(main())
