"""Benchmark of the per-layer decode KV swap-in on one GB300 (or N replicas).

One step is one layer-call of the whole hot path on one batch, in one kernel:
lookup (token -> slot index), cross-step miss de-duplication and locations,
then the commit (epoch-CLOCK victims, rotation, index update) side by side
with the miss-row copy from the pinned host pool; plus the sparse page table
for the paged workload.  The default workload is the largest configuration,
the 4-step (MTP) swap at batch 64 (C3).

Metric: selected tokens resolved per second per layer-call (B * S * K / step
time).  Inputs (top-k, request slots, sequence lengths) are resident on the
device before the timed region; L2 is flushed (a 256 MiB write) between timed
steps.  Each timed step is bracketed by CUDA events on the launching stream.
`e2e` repeats the measurement through the same C ABI calls with host buffers:
per step the host->device copy of the inputs from pinned memory and the
device->host read of the locations are inside the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config C3]
                       [--impl reference]
Under torchrun each rank drives one GPU with its own copy of the workload
(replicas, weak scaling); rank 0 prints one JSON line.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import hs_workloads as W  # noqa: E402

METRIC = "selected tokens resolved/s per layer-call"
# Per-launch counters of the swap-in kernel from one ncu capture per
# workload of the timed steps (steady state, after an L2 flush), recorded in
# profiles/swapin_kernel_traffic.md: DRAM read + write bytes and host-link
# (system memory) read bytes.  Workloads without a capture of the current
# kernel report null.
NCU_TRAFFIC = {("C3", "dense"): {"dram_bytes": 17851477, "host_link_bytes": 41563722},
               ("C2", "dense"): {"dram_bytes": 7540650, "host_link_bytes": 11197845},
               ("C4", "dense"): {"dram_bytes": 1712640, "host_link_bytes": 22087381},
               ("C5", "dense"): {"dram_bytes": 1957632, "host_link_bytes": 1695200}}
NCU_CAPTURE = "profiles/swapin_kernel_traffic.md"
UNIT = "tokens/s"
PREROLL_CALLS = 8  # calls of the stream run before warm-up so the cache is in steady state
# Untimed steps run right after each gate, before the timed ones.  On GB300
# the first step after the gate always ran about twice as slow as the rest,
# and about one run in five began with a slow stretch of up to ~15 ms (steps
# up to 10x slow, decaying), host enqueue well ahead of the GPU throughout.
# 16 primer steps (2.5 ms of C2 work) absorbed most of it; 64 (10 ms of C2
# work, 20 ms of C3) leave the timed steps clear of the longest stretches seen.
PRIMER_STEPS = 64
FLUSH_BYTES = 256 << 20


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="C3", choices=sorted(W.WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--copy-ctas", type=int, default=0)
    ap.add_argument("--index", default="dense", choices=["hash", "dense"],
                    help="token -> slot index: a dense map (faster on GB300 at these "
                         "sizes) or per-request hash banks")
    ap.add_argument("--launch", default="graph", choices=["graph", "direct"],
                    help="timed steps as one replayed CUDA graph per step, or direct launches")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--compare-sequential", action="store_true",
                    help="multi-step vs sequential per-step swap under CUDA graphs")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.samples = []
        self.proc = None
        self.gpu = self.smi_id(gpu_index)
        self.interval = interval_ms
        self.thread = None

    @staticmethod
    def smi_id(gpu_index: int) -> str:
        """nvidia-smi's name for torch device `gpu_index`: its UUID, which stays
        right when CUDA_VISIBLE_DEVICES renumbers the devices (else the index)."""
        try:
            import torch
            u = str(torch.cuda.get_device_properties(gpu_index).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return str(gpu_index)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def wait_first(self, timeout: float = 5.0):
        """Returns once the first sample has arrived: nvidia-smi's start-up
        (which slowed the GPU's first steps when it overlapped them) is over."""
        t_end = time.time() + timeout
        while self.proc is not None and not self.samples and time.time() < t_end:
            time.sleep(0.01)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        inside = [s for t, s in self.samples if t0 <= t <= t1]
        used = inside
        if not used and self.samples:  # region shorter than the sampling interval
            mid = 0.5 * (t0 + t1)
            used = [min(self.samples, key=lambda ts: abs(ts[0] - mid))[1]]
        out = {"samples_in_region": len(inside), "samples_used": len(used)}
        if not used:
            return out
        try:
            sm = [float(s[1]) for s in used]
            out["sm_mhz"] = statistics.median(sm)
            out["sm_max_mhz"] = max(float(s[2]) for s in used)
            out["power_w_max"] = max(float(s[3]) for s in used)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            out["reasons"] = sorted({n for s in used for n, v in zip(names, s[5:9])
                                     if v.lower().startswith("active")})
        except (ValueError, IndexError):
            out["raw"] = used[:3]
        return out


def measure_h2d_peak(torch, dev, nbytes=256 << 20, reps=20):
    """Pinned host -> device cudaMemcpyAsync bandwidth, best of `reps` (GB/s)."""
    src = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    src.fill_(1)
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = 0.0
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(reps):
        s.record()
        dst.copy_(src, non_blocking=True)
        e.record()
        e.synchronize()
        best = max(best, nbytes / (s.elapsed_time(e) * 1e-3) / 1e9)
    del src, dst
    return best


def max_over_ranks(torch, ms, world, device):
    """The slowest rank's time (every rank holds its own replica)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(entries_per_replica, world, ms):
    """Tokens resolved per second by all replicas together (weak scaling)."""
    return entries_per_replica * world / (ms * 1e-3)


def gate(torch, steps):
    """Hold the stream with a short device-side sleep so that the host can
    queue every step before the first one runs: the per-step events then see
    GPU time only, not host launch latency."""
    torch.cuda._sleep(int(2e6 * (20 + 1.0 * steps)))  # ~2e6 cycles per ms


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


def cpu_baseline_oracle(w, calls, rpi, sl, seconds, pool_np):
    """The CPU oracle on the same stream: pre-roll untimed, then time calls
    until `seconds` of CPU work (at least 2 calls)."""
    from oracle import Oracle
    threads = min(w.batch, os.cpu_count() or 1)
    C = w.steps * w.top_k
    o = Oracle(w.batch, w.seq_len, w.row_bytes, w.hot_buffer, w.top_k, w.steps, 1)
    mirror = np.zeros((w.batch * (w.hot_buffer + C), w.row_bytes), dtype=np.uint8)
    for c in calls[:PREROLL_CALLS]:
        o.swap_in(0, pool_np, mirror, rpi, sl, c, num_threads=threads)
    n = 0
    t_total = 0.0
    for c in calls[PREROLL_CALLS:]:
        t = time.perf_counter()
        o.swap_in(0, pool_np, mirror, rpi, sl, c, num_threads=threads)
        t_total += time.perf_counter() - t
        n += 1
        if t_total >= seconds and n >= 2:
            break
    return {"value": w.entries * n / t_total, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": "%d steady-state calls of %s after %d pre-roll calls (%d request threads, "
                      "row copies included)" % (n, w.name, PREROLL_CALLS, threads)}


def run_reference(args, w):
    """--impl reference: the CPU oracle timed on this workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    from oracle import Oracle
    stream = W.TopkStream(w)
    total_calls = PREROLL_CALLS + args.warmup + args.steps
    calls = stream.calls(total_calls)
    rpi, sl = W.req_pool_indices(w), W.seq_lens(w)
    pool = np.empty((w.batch, w.seq_len, w.row_bytes), dtype=np.uint8)
    W.fill_host_pool(pool, 0)
    threads = min(w.batch, os.cpu_count() or 1)
    C = w.steps * w.top_k
    o = Oracle(w.batch, w.seq_len, w.row_bytes, w.hot_buffer, w.top_k, w.steps, 1)
    mirror = np.zeros((w.batch * (w.hot_buffer + C), w.row_bytes), dtype=np.uint8)
    for c in calls[:PREROLL_CALLS + args.warmup]:
        o.swap_in(0, pool, mirror, rpi, sl, c, num_threads=threads)
    times = []
    for c in calls[PREROLL_CALLS + args.warmup:]:
        t = time.perf_counter()
        o.swap_in(0, pool, mirror, rpi, sl, c, num_threads=threads)
        if w.page_size:
            from oracle import page_table
            page_table(c, sl, w.page_size, max_seq_len=w.seq_len)
        times.append(time.perf_counter() - t)
    ms = 1e3 * sum(times) / len(times)
    value = w.entries / (ms * 1e-3)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic", "impl": "reference",
            "config": config_dict(w, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": "%d timed calls of %s after %d pre-roll + %d warm-up calls"
                                       % (args.steps, w.name, PREROLL_CALLS, args.warmup)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def copy_ceiling(torch, pkg, cache, w, dev, flush, rows_per_request, reps=10):
    """Host-link ceiling of the library's row copy: replays synthetic miss
    plans with hs_copy_planned (16-byte vector copies like the swap-in's) for
    (a) consecutive host rows and (b) random host rows, the latter with as many
    rows per request as a measured step, in random and in ascending order and
    at 128-byte aligned offsets.  Writes device rows, so it runs after
    every other measurement."""
    Bn, C, H, L, Wr = w.batch, w.steps * w.top_k, w.hot_buffer, w.seq_len, w.row_bytes
    rng = np.random.default_rng(5)
    out = {}
    n_step = max(1, int(rows_per_request))
    # rows whose host byte offset is a multiple of 128 (t * W % 128 == 0)
    align = 128 // int(np.gcd(Wr, 128))
    for kind, n in (("consecutive_rows", C), ("random_rows", n_step),
                    ("random_rows_ascending", n_step), ("random_rows_128B_aligned", n_step)):
        n = min(n, C)
        src = np.zeros((Bn, C), np.int64)
        dst = np.zeros((Bn, C), np.int64)
        for b in range(Bn):
            if kind == "consecutive_rows":
                toks = np.arange(n) + rng.integers(0, L - n + 1)
            elif kind == "random_rows":
                toks = rng.choice(L, size=n, replace=False)
            elif kind == "random_rows_ascending":  # the same kind of rows in host order
                toks = np.sort(rng.choice(L, size=n, replace=False))
            else:
                n = min(n, L // align)
                toks = rng.choice(L // align, size=n, replace=False) * align
            src[b, :n] = b * L + toks
            dst[b, :n] = b * (H + C) + H + np.arange(n)
        cnt = torch.full((Bn,), n, dtype=torch.int32, device=dev)
        s_t, d_t = torch.from_numpy(src).to(dev), torch.from_numpy(dst).to(dev)
        times = []
        for r in range(reps + 2):
            flush.fill_(r & 0xFF)
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            pkg.hs_copy_planned(cache.handle, 0, s_t, d_t, cnt)
            b_.record()
            b_.synchronize()
            if r >= 2:
                times.append(a.elapsed_time(b_))
        ms = statistics.median(times)
        nbytes = Bn * n * Wr
        out[kind] = {"rows": Bn * n, "mb": nbytes / 1e6, "ms": ms,
                     "gbs": nbytes / (ms * 1e-3) / 1e9}
    return out


def decode_step_extra_page(torch, pkg, w, dev, flush, calls, pool, dense, E=256, n=20):
    """Decode step with the extra page on: per step, the write-back of one new
    row per request (hs_append_rows: host pool over the host link, extra page
    and hot copy in HBM), then the swap-in with the newest E positions of
    every request served from its extra page.  A fresh cache on the same host
    pool, pre-rolled like the main measurement; the extra page is filled once
    (prefill) before."""
    from sparse_attention_kv_swap_gb300.cache import SwapInCache
    Bn, L, Wr = w.batch, w.seq_len, w.row_bytes
    cfg = pkg.make_config(Bn, L, Wr, w.hot_buffer, w.top_k, w.steps, 1,
                          index_kind=1 if dense else 0, extra_page_size=E)
    cache = SwapInCache(cfg, host_pools=[pool], device=dev)
    rpi = torch.from_numpy(W.req_pool_indices(w)).to(dev)
    sl = torch.from_numpy(W.seq_lens(w)).to(dev)
    q = torch.arange(Bn, dtype=torch.int32, device=dev)
    page = torch.arange((L - 1) // E * E, L, dtype=torch.int32, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)
    pre_rows = torch.randint(0, 256, (Bn * page.numel(), Wr), dtype=torch.uint8, device=dev,
                             generator=gen)
    cache.append_rows(q.repeat_interleave(page.numel()), page.repeat(Bn),
                      torch.full((Bn * page.numel(),), L, dtype=torch.int32, device=dev),
                      pre_rows)
    new_tok = torch.full((Bn,), L - 1, dtype=torch.int32, device=dev)
    new_len = torch.full((Bn,), L, dtype=torch.int32, device=dev)
    lead = PREROLL_CALLS + PRIMER_STEPS  # untimed calls before the timed ones
    rows = torch.randint(0, 256, (n + lead, Bn, Wr), dtype=torch.uint8, device=dev,
                         generator=gen)
    topk_all = torch.from_numpy(np.stack(calls[:lead + n])).to(dev)
    locs = torch.empty((Bn, w.steps, w.top_k), dtype=torch.int32, device=dev)
    stats = torch.zeros((lead + n, Bn, pkg.binding.HS_NUM_STATS), dtype=torch.int32,
                        device=dev)
    s = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for i in range(lead + n):
        k = i - lead
        if k == -PRIMER_STEPS:
            torch.cuda.synchronize()
            gate(torch, n + PRIMER_STEPS)
        if k == 0:
            torch.cuda.nvtx.range_push("decode_steps")  # lets a profiler select these launches
        flush.fill_(i & 0xFF)
        if k >= 0:
            ev[k][0].record(s)
        cache.append_rows(q, new_tok, new_len, rows[i])
        if k >= 0:
            ev[k][1].record(s)
        cache.swap_in(rpi, sl, topk_all[i], 0, out={"device_locs": locs, "stats": stats[i]})
        if k >= 0:
            ev[k][2].record(s)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    rc, flags = cache.status()
    if flags:
        raise RuntimeError("device status flags %#x in the decode-step measurement" % flags)
    app = [e[0].elapsed_time(e[1]) for e in ev]
    swp = [e[1].elapsed_time(e[2]) for e in ev]
    pair = [e[0].elapsed_time(e[2]) for e in ev]
    st = stats[lead:].cpu().numpy()
    ms = statistics.mean(pair)
    cache.close()
    return {"extra_page_size": E, "steps": n, "launch": "direct launches through the C ABI",
            "ms_per_step": ms, "value": w.entries / (ms * 1e-3), "unit": UNIT,
            "append_ms_median": statistics.median(app),
            "swap_in_ms_median": statistics.median(swp),
            "append_rows_per_step": Bn, "append_bytes_per_step": Bn * Wr,
            "extra_entries_fraction": float(st[:, :, 8].sum() / (n * w.entries)),
            "unique_misses_per_step": float(st[:, :, 3].sum(axis=1).mean()),
            "gpu_launches_per_step": 3}


def deferred_copy_pipeline(torch, pkg, w, dev, flush, calls, pool, dense, layers=4, n=10,
                           copy_ctas=32):
    """F2 in use: a `layers`-layer decode step, swap-in after swap-in on one
    stream, against the deferred-copy protocol, where each layer's swap-in only
    resolves and commits and its recorded miss plan is copied on a second
    stream (hs_copy_planned), so that layer l's copy overlaps the resolve of
    layer l + 1.  Every layer sees the same call stream (independent state per
    layer) and shares the host pool."""
    from sparse_attention_kv_swap_gb300.cache import SwapInCache
    Bn, S, Kk, C = w.batch, w.steps, w.top_k, w.steps * w.top_k
    cfg = pkg.make_config(Bn, w.seq_len, w.row_bytes, w.hot_buffer, Kk, S, layers,
                          index_kind=1 if dense else 0)
    seq = SwapInCache(cfg, host_pools=[pool] * layers, device=dev)
    dfr = SwapInCache(cfg, host_pools=[pool] * layers, device=dev)
    pkg.hs_set_defer_copy(dfr.handle, True)
    if copy_ctas:
        pkg.hs_set_copy_ctas(dfr.handle, copy_ctas)
    rpi = torch.from_numpy(W.req_pool_indices(w)).to(dev)
    sl = torch.from_numpy(W.seq_lens(w)).to(dev)
    lead = PREROLL_CALLS + PRIMER_STEPS  # untimed calls before the timed ones
    topk_all = torch.from_numpy(np.stack(calls[:lead + n])).to(dev)
    locs = [torch.empty((Bn, S, Kk), dtype=torch.int32, device=dev) for _ in range(layers)]
    plans = [{"device_locs": locs[l],
              "miss_src": torch.empty((Bn, C), dtype=torch.int64, device=dev),
              "miss_dst": torch.empty((Bn, C), dtype=torch.int64, device=dev),
              "miss_count": torch.empty(Bn, dtype=torch.int32, device=dev)}
             for l in range(layers)]
    s0 = torch.cuda.current_stream()
    # two copy streams, alternating by layer, so that one layer's copy can
    # start while the previous one drains; 32 CTAs per copy keep the link full
    # and leave the SMs that the next layer's lookup needs
    copy_streams = (torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
    done = [torch.cuda.Event() for _ in range(layers)]

    def sequential(i):
        for l in range(layers):
            seq.swap_in(rpi, sl, topk_all[i], l, out={"device_locs": locs[l]})

    def pipelined(i):
        for l in range(layers):
            dfr.swap_in(rpi, sl, topk_all[i], l, plan=True, out=plans[l])
            done[l].record(s0)
            sc = copy_streams[l % 2]
            sc.wait_event(done[l])
            pkg.hs_copy_planned(dfr.handle, l, plans[l]["miss_src"], plans[l]["miss_dst"],
                                plans[l]["miss_count"], stream=sc)
        for sc in copy_streams:  # the step ends when every layer's rows are in
            s0.wait_stream(sc)

    out = {}
    for name, fn in (("sequential", sequential), ("deferred_pipelined", pipelined)):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for i in range(lead + n):
            k = i - lead
            if k == -PRIMER_STEPS:
                torch.cuda.synchronize()
                gate(torch, 2 * (n + PRIMER_STEPS))
            if k == 0:
                torch.cuda.nvtx.range_push(name + "_layers")
            flush.fill_(i & 0xFF)
            if k >= 0:
                ev[k][0].record(s0)
            fn(i)
            if k >= 0:
                ev[k][1].record(s0)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        out[name] = {"ms_per_step": ms, "value": layers * w.entries / (ms * 1e-3)}
    for cache in (seq, dfr):
        rc, flags = cache.status()
        if flags:
            raise RuntimeError("device status flags %#x in the deferred-copy pipeline" % flags)
        cache.close()
    out.update(layers=layers, steps=n, unit=UNIT,
               speedup=out["sequential"]["ms_per_step"] / out["deferred_pipelined"]["ms_per_step"],
               copy_ctas=copy_ctas or "default",
               launch="direct launches through the C ABI; copies on two more streams, "
                      "alternating by layer")
    return out


# Words of the kernel's per-CTA timeline (hs_set_timeline), in phase order.
TIMELINE_WORDS = (("probed", 1), ("barrier_0", 2), ("inserted", 3), ("table_complete", 4),
                  ("flagged", 5), ("words_exchanged", 6), ("rows_loaded", 7),
                  ("lists_written", 8), ("commit_done", 9), ("copy_done", 10))
TL_START, TL_LISTS, TL_COMMIT, TL_COPY, TL_P = 0, 8, 9, 10, 15


def phase_times(tls):
    """Phase spans of each timed launch from the kernel's timeline stamps.

    tls: int64 [launches, batch, 8 ranks, 16 words] as written with
    hs_set_timeline (words 0-10 global-timer ns, word 15 the cluster size).
    Per launch, with t0 the first CTA's start:
      gather_span   = last word 8 (locations and miss lists written) - t0;
      commit_span   = last word 9 of the leader CTAs - their first word 8;
      commit        = each leader CTA's word 9 - word 8;
      copy_span     = last word 10 (a CTA's last warp done) - first word 8.
    The summary gives, in microseconds from t0, the median over launches of
    the median and the last CTA at each stamp."""
    tls = np.asarray(tls, dtype=np.int64)
    out = {"gather_span_us": [], "commit_span_us": [], "commit_us": [], "copy_span_us": []}
    marks = {n: ([], []) for n, _ in TIMELINE_WORDS}
    for t in tls:
        P = int(t[0, 0, TL_P])
        used = t[:, :P, :]
        t0 = used[:, :, TL_START].min()
        out["gather_span_us"].append((used[:, :, TL_LISTS].max() - t0) / 1e3)
        lead = t[:, 0, :]
        out["commit_span_us"].append((lead[:, TL_COMMIT].max() - lead[:, TL_LISTS].min()) / 1e3)
        out["commit_us"].extend(((lead[:, TL_COMMIT] - lead[:, TL_LISTS]) / 1e3).tolist())
        out["copy_span_us"].append((used[:, :, TL_COPY].max() - used[:, :, TL_LISTS].min()) / 1e3)
        for n, k in TIMELINE_WORDS:
            v = (lead[:, k] if k == TL_COMMIT else used[:, :, k].ravel()) - t0
            marks[n][0].append(float(np.median(v)) / 1e3)
            marks[n][1].append(float(v.max()) / 1e3)
    out["summary"] = {n: {"median_cta": statistics.median(m[0]), "last_cta": statistics.median(m[1])}
                      for n, m in marks.items()}
    out["summary"]["cluster_size"] = int(tls[0, 0, 0, TL_P])
    return out


def multi_vs_sequential(torch, pkg, w, dev, flush, calls, pool, dense, n=20, warmup=5):
    """F1: the multi-step swap (one S-step call) against sequential per-step
    swap (S single-step calls) on the same index stream, each captured as a
    CUDA graph and replayed after an L2 flush, as in the multi-step swap
    report's benchmark (section 实现拆解 item 4; its 48.2% figure is for
    batch 64, 4 steps on an H20).  Two fresh caches on the same host pool,
    with the bench's index kind."""
    from sparse_attention_kv_swap_gb300.cache import SwapInCache
    Bn, S, Kk = w.batch, w.steps, w.top_k
    cfg = pkg.make_config(Bn, w.seq_len, w.row_bytes, w.hot_buffer, Kk, S, 1,
                          index_kind=1 if dense else 0)
    multi = SwapInCache(cfg, host_pools=[pool], device=dev)
    seq = SwapInCache(cfg, host_pools=[pool], device=dev)
    rpi = torch.from_numpy(W.req_pool_indices(w)).to(dev)
    sl = torch.from_numpy(W.seq_lens(w)).to(dev)
    buf_m = torch.empty((Bn, S, Kk), dtype=torch.int32, device=dev)
    buf_s = [torch.empty((Bn, 1, Kk), dtype=torch.int32, device=dev) for _ in range(S)]
    out_m = {"device_locs": torch.empty((Bn, S, Kk), dtype=torch.int32, device=dev)}
    out_s = [{"device_locs": torch.empty((Bn, 1, Kk), dtype=torch.int32, device=dev)}
             for _ in range(S)]
    stream = torch.cuda.Stream(device=dev)

    def load(c):
        t = torch.from_numpy(c).to(dev)
        buf_m.copy_(t)
        for k in range(S):
            buf_s[k].copy_(t[:, k:k + 1])

    def run_multi():
        multi.swap_in(rpi, sl, buf_m, 0, out=out_m, stream=stream)

    def run_seq():
        for k in range(S):
            seq.swap_in(rpi, sl, buf_s[k], 0, out=out_s[k], stream=stream)

    load(calls[0])
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):  # first calls set kernel attributes outside capture
        run_multi()
        run_seq()
    torch.cuda.synchronize()
    multi.reset_requests(torch.arange(Bn, dtype=torch.int32, device=dev))
    seq.reset_requests(torch.arange(Bn, dtype=torch.int32, device=dev))
    g_multi, g_seq = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_multi, stream=stream):
        run_multi()
    with torch.cuda.graph(g_seq, stream=stream):
        run_seq()
    torch.cuda.synchronize()
    t_m, t_s = [], []
    for i, c in enumerate(calls[:PREROLL_CALLS + warmup + n]):
        load(c)
        torch.cuda.synchronize()
        timed = i >= PREROLL_CALLS + warmup
        pair = ((g_multi, t_m), (g_seq, t_s))
        for g, acc in (pair if i % 2 == 0 else pair[::-1]):  # alternate which runs first
            flush.fill_(i & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):  # replay runs on the current stream
                # a 1 ms device-side hold so that the graph launch is queued
                # before event `a` runs (too short for the clocks to drop)
                torch.cuda._sleep(int(2e6))
                a.record(stream)
                g.replay()
                b.record(stream)
            b.synchronize()
            if timed:
                acc.append(a.elapsed_time(b))
    for cache in (multi, seq):
        rc, flags = cache.status()
        if flags:
            raise RuntimeError("device status flags %#x in the multi-step comparison" % flags)
        cache.close()
    # medians: a single slow replay (seen on a shared box) would move a mean
    ms_m, ms_s = statistics.median(t_m), statistics.median(t_s)
    return {"latency_reduction": 1.0 - ms_m / ms_s, "multi_step_ms": ms_m,
            "sequential_ms": ms_s, "multi_step_ms_mean": statistics.mean(t_m),
            "sequential_ms_mean": statistics.mean(t_s),
            "multi_step_tokens_per_s": w.entries / (ms_m * 1e-3),
            "sequential_tokens_per_s": w.entries / (ms_s * 1e-3), "steps": n,
            "index": "dense" if dense else "hash", "cuda_graph": True,
            "context": "pages: 48.2% at batch 64, 4 steps, H20 (Hopper)"}


def run_compare_sequential(args, w):
    """--compare-sequential: F1 alone, as its own JSON line."""
    import torch
    import sparse_attention_kv_swap_gb300 as pkg
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    calls = W.TopkStream(w).calls(PREROLL_CALLS + args.warmup + args.steps)
    pool = torch.empty((w.batch, w.seq_len, w.row_bytes), dtype=torch.uint8, pin_memory=True)
    W.fill_host_pool(pool.numpy(), 0)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clocks = ClockSampler(0)
    clocks.start()
    clocks.wait_first()
    t0 = time.time()
    f1 = multi_vs_sequential(torch, pkg, w, dev, flush, calls, pool, args.index == "dense",
                             n=args.steps, warmup=args.warmup)
    t1 = time.time()
    clocks.stop()
    line = {"metric": "multi-step vs sequential per-step swap latency reduction",
            "value": f1["latency_reduction"], "unit": "fraction", "higher_is_better": True,
            **f1, "warmup": args.warmup, "data": "synthetic", "config": config_dict(w, 1),
            "clocks": clocks.summary(t0, t1)}
    print(json.dumps(line), flush=True)
    return 0


def config_dict(w, world):
    return {"workload": "%s (%s)" % (w.name, "C%d" % w.cfg_id), "batch": w.batch,
            "steps": w.steps, "top_k": w.top_k, "seq_len": w.seq_len, "hot_buffer": w.hot_buffer,
            "row_bytes": w.row_bytes, "page_size": w.page_size, "index_mix": w.kind,
            "reuse": w.reuse, "preroll_calls": PREROLL_CALLS,
            "l2": "flushed between timed steps (256 MiB write)",
            "parallelism": "replicas x%d" % world if world > 1 else "single GPU"}


def main():
    args = parse_args()
    w = W.WORKLOADS[args.config]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.compare_sequential:
        return run_compare_sequential(args, w)

    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import sparse_attention_kv_swap_gb300 as pkg
    from sparse_attention_kv_swap_gb300.cache import SwapInCache

    K, Wm = args.steps, args.warmup
    n_e2e = min(K, 20)
    n_phase = min(K, 20)
    n_alt = min(K, 20)
    total_calls = (PREROLL_CALLS + Wm + 1 + K + n_phase + 2 * (n_e2e + PRIMER_STEPS) + n_alt
                   + 3 * PRIMER_STEPS)
    stream_gen = W.TopkStream(w)
    calls = stream_gen.calls(total_calls)
    rpi_np, sl_np = W.req_pool_indices(w), W.seq_lens(w)

    cfg = pkg.make_config(w.batch, w.seq_len, w.row_bytes, w.hot_buffer, w.top_k, w.steps, 1,
                          index_kind=1 if args.index == "dense" else 0)
    pool = torch.empty((w.batch, w.seq_len, w.row_bytes), dtype=torch.uint8, pin_memory=True)
    W.fill_host_pool(pool.numpy(), 0)
    cache = SwapInCache(cfg, host_pools=[pool], device=dev)
    if args.copy_ctas:
        pkg.hs_set_copy_ctas(cache.handle, args.copy_ctas)
    s = torch.cuda.current_stream()

    topk_all = torch.from_numpy(np.stack(calls)).to(dev)  # [calls, B, S, K]
    rpi = torch.from_numpy(rpi_np).to(dev)
    sl = torch.from_numpy(sl_np).to(dev)
    Bn, S, Kk = w.batch, w.steps, w.top_k
    locs = torch.empty((Bn, S, Kk), dtype=torch.int32, device=dev)
    stats = torch.zeros((total_calls, Bn, pkg.binding.HS_NUM_STATS), dtype=torch.int32,
                        device=dev)
    page_out = None
    if w.page_size:
        page_out = {"pages": torch.empty((Bn, S * Kk), dtype=torch.int32, device=dev),
                    "num_pages": torch.empty(Bn, dtype=torch.int32, device=dev),
                    "token_page": torch.empty((Bn, S, Kk), dtype=torch.int32, device=dev)}
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    # The page table depends on the top-k and lengths only, so it runs on a
    # second stream beside the swap-in and joins it at the end of the step.
    pt_stream = torch.cuda.Stream(device=dev)

    def page_table_beside(topk, lens, origin):
        pt_stream.wait_stream(origin)
        cache.page_table(topk, lens, w.page_size, out=page_out, stream=pt_stream)

    def step(i, topk):
        if page_out is not None:
            page_table_beside(topk, sl, s)
        cache.swap_in(rpi, sl, topk, 0, out={"device_locs": locs, "stats": stats[i]})
        if page_out is not None:
            s.wait_stream(pt_stream)

    # the host-link peak first, far from any timed region
    h2d_peak = measure_h2d_peak(torch, dev)

    # pre-roll and warm-up
    for i in range(PREROLL_CALLS + Wm):
        step(i, topk_all[i])
    torch.cuda.synchronize()
    rc, flags = cache.status()
    if flags:
        raise RuntimeError("device status flags %#x after warm-up" % flags)

    # One CUDA graph of a whole step (the way a decode loop replays it): the
    # step's top-k is staged into the graph's input buffer before its events.
    topk_buf = torch.empty((Bn, S, Kk), dtype=torch.int32, device=dev)
    stats_buf = torch.empty((Bn, pkg.binding.HS_NUM_STATS), dtype=torch.int32, device=dev)
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        if page_out is not None:
            page_table_beside(topk_buf, sl, side)
        cache.swap_in(rpi, sl, topk_buf, 0, out={"device_locs": locs, "stats": stats_buf},
                      stream=side)
        if page_out is not None:
            side.wait_stream(pt_stream)

    def run_steps(first, n, mode, events):
        """n steps from call `first` on, each between its own pair of events."""
        for k in range(n):
            i = first + k
            if mode == "graph":
                topk_buf.copy_(topk_all[i])
            flush.fill_(k & 0xFF)
            events[k][0].record(s)
            if mode == "graph":
                graph.replay()
            else:
                step(i, topk_all[i])
            events[k][1].record(s)
            if mode == "graph":
                stats[i].copy_(stats_buf)

    # The graph's first replay uploads it to the device: do that on one more
    # warm-up call, outside any timing.
    warm_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))]
    run_steps(PREROLL_CALLS + Wm, 1, "graph", warm_ev)
    torch.cuda.synchronize()

    peaks = read_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    hbm_src = "MEASURED_PEAKS.json hbm_gbs (measured)" if "hbm_gbs" in peaks else "fallback 6.8 TB/s"

    # ---- timed region: K steps, per-step events, L2 flush between steps ----
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    primer_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(PRIMER_STEPS)]
    clocks = ClockSampler(local)
    clocks.start()
    clocks.wait_first()
    time.sleep(0.05)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    base = PREROLL_CALLS + Wm + 1 + PRIMER_STEPS  # after the graph warm-up and primer calls
    gate(torch, K + PRIMER_STEPS)
    run_steps(base - PRIMER_STEPS, PRIMER_STEPS, args.launch, primer_ev)
    torch.cuda.nvtx.range_push("timed_steps")  # lets a profiler select these launches
    run_steps(base, K, args.launch, ev)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(torch, sum(step_ms) / K, world, dev)
    value = whole_job_rate(w.entries, world, ms)
    st_timed = stats[base:base + K].cpu().numpy()
    # the other launch mode on the next calls of the stream, for comparison
    alt = "direct" if args.launch == "graph" else "graph"
    abase = base + K + PRIMER_STEPS + n_phase + 2 * (n_e2e + PRIMER_STEPS) + PRIMER_STEPS
    ev_alt = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n_alt)]

    # ---- phase split from the kernel's own timeline (separate pass) ----
    # Every CTA stamps the GPU's global timer at its phase boundaries
    # (hs_set_timeline); the launches are direct, each between two events.
    tl = torch.zeros((Bn, 8, 16), dtype=torch.int64, device=dev)
    tls = torch.zeros((n_phase, Bn, 8, 16), dtype=torch.int64, device=dev)
    e_a = [torch.cuda.Event(enable_timing=True) for _ in range(n_phase)]
    e_b = [torch.cuda.Event(enable_timing=True) for _ in range(n_phase)]
    pbase = base + K + PRIMER_STEPS
    pkg.hs_set_timeline(cache.handle, tl)
    torch.cuda.synchronize()
    gate(torch, n_phase + PRIMER_STEPS)
    for i in range(base + K, pbase):
        flush.fill_(i & 0xFF)
        step(i, topk_all[i])
    for k in range(n_phase):
        flush.fill_(k & 0xFF)
        e_a[k].record(s)
        cache.swap_in(rpi, sl, topk_all[pbase + k], 0,
                      out={"device_locs": locs, "stats": stats[pbase + k]})
        e_b[k].record(s)
        tls[k].copy_(tl)
    torch.cuda.synchronize()
    pkg.hs_set_timeline(cache.handle, None)
    t_kernel = [a.elapsed_time(b) for a, b in zip(e_a, e_b)]
    st_phase = stats[pbase:pbase + n_phase].cpu().numpy()
    timeline = phase_times(tls.cpu().numpy())

    # ---- e2e: host buffers through the same C ABI call ----
    # Each step's inputs sit in one pinned host record [top-k | slots | lengths]
    # and go over in one copy; the locations come back into pinned memory.
    # PRIMER_STEPS untimed steps come first (they also touch the host buffers).
    ebase = pbase + n_phase
    n_in = Bn * S * Kk + 2 * Bn
    host_in = torch.empty((n_e2e + PRIMER_STEPS, n_in), dtype=torch.int32).pin_memory()
    for k in range(n_e2e + PRIMER_STEPS):
        host_in[k, :Bn * S * Kk] = torch.from_numpy(calls[ebase + k].reshape(-1))
        host_in[k, Bn * S * Kk:Bn * S * Kk + Bn] = torch.from_numpy(rpi_np)
        host_in[k, Bn * S * Kk + Bn:] = torch.from_numpy(sl_np)
    locs_host = torch.empty((Bn, S, Kk), dtype=torch.int32).pin_memory()
    dev_in = torch.empty(n_in, dtype=torch.int32, device=dev)
    topk_dev = dev_in[:Bn * S * Kk].view(Bn, S, Kk)
    rpi_dev = dev_in[Bn * S * Kk:Bn * S * Kk + Bn]
    sl_dev = dev_in[Bn * S * Kk + Bn:]
    e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_e2e + PRIMER_STEPS)]
    torch.cuda.synchronize()
    gate(torch, n_e2e + PRIMER_STEPS)
    for k in range(n_e2e + PRIMER_STEPS):
        flush.fill_(k & 0xFF)
        e2e_ev[k][0].record(s)
        dev_in.copy_(host_in[k], non_blocking=True)
        e2e_ev[k][1].record(s)
        if page_out is not None:
            page_table_beside(topk_dev, sl_dev, s)
        cache.swap_in(rpi_dev, sl_dev, topk_dev, 0, out={"device_locs": locs})
        if page_out is not None:
            s.wait_stream(pt_stream)
        e2e_ev[k][2].record(s)
        locs_host.copy_(locs, non_blocking=True)
        e2e_ev[k][3].record(s)
    torch.cuda.synchronize()
    e2e_ev = e2e_ev[PRIMER_STEPS:]
    e2e_ms = sum(ev[0].elapsed_time(ev[3]) for ev in e2e_ev) / n_e2e
    e2e_parts = {name: statistics.median(ev[i].elapsed_time(ev[i + 1]) for ev in e2e_ev)
                 for i, name in enumerate(("h2d_ms_median", "swap_in_ms_median",
                                           "d2h_ms_median"))}
    e2e_ms = max_over_ranks(torch, e2e_ms, world, dev)
    h2d_bytes = n_in * 4
    d2h_bytes = locs_host.numel() * 4
    # The same steps with no copy engine: over NVLink-C2C pinned host memory is
    # device-addressable, so the call is given the pinned records and a pinned
    # output, and its kernels read the inputs and write the locations across
    # the link.  Same bytes each way.
    zbase = ebase + n_e2e + PRIMER_STEPS
    host_zc = torch.empty((n_e2e + PRIMER_STEPS, n_in), dtype=torch.int32).pin_memory()
    for k in range(n_e2e + PRIMER_STEPS):
        host_zc[k, :Bn * S * Kk] = torch.from_numpy(calls[zbase + k].reshape(-1))
        host_zc[k, Bn * S * Kk:Bn * S * Kk + Bn] = torch.from_numpy(rpi_np)
        host_zc[k, Bn * S * Kk + Bn:] = torch.from_numpy(sl_np)
    zc_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_e2e + PRIMER_STEPS)]
    torch.cuda.synchronize()
    gate(torch, n_e2e + PRIMER_STEPS)
    for k in range(n_e2e + PRIMER_STEPS):
        flush.fill_(k & 0xFF)
        rec = host_zc[k]
        zc_ev[k][0].record(s)
        if page_out is not None:
            page_table_beside(rec[:Bn * S * Kk].view(Bn, S, Kk), rec[Bn * S * Kk + Bn:], s)
        cache.swap_in(rec[Bn * S * Kk:Bn * S * Kk + Bn], rec[Bn * S * Kk + Bn:],
                      rec[:Bn * S * Kk].view(Bn, S, Kk), 0, out={"device_locs": locs_host})
        if page_out is not None:
            s.wait_stream(pt_stream)
        zc_ev[k][1].record(s)
    torch.cuda.synchronize()
    zc_ms = max_over_ranks(torch, sum(a.elapsed_time(b) for a, b in zc_ev[PRIMER_STEPS:]) / n_e2e, world,
                           dev)
    rc, flags = cache.status()
    if flags:
        raise RuntimeError("device status flags %#x after the timed region" % flags)
    torch.cuda.synchronize()
    gate(torch, n_alt + PRIMER_STEPS)
    run_steps(abase - PRIMER_STEPS, PRIMER_STEPS, alt, primer_ev)
    run_steps(abase, n_alt, alt, ev_alt)
    torch.cuda.synchronize()
    alt_ms = sum(a.elapsed_time(b) for a, b in ev_alt) / n_alt
    # Differential all-hit replay: each of the last calls repeated at once
    # finds its tokens resident (when they fit), so it copies nothing; the
    # step time minus this time is the part of a step the copy adds.
    n_ah = min(n_alt, 10)
    ev_ah = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(n_ah)]
    ah_stats = torch.zeros((n_ah, Bn, pkg.binding.HS_NUM_STATS), dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    gate(torch, 2 * n_ah)
    for k in range(n_ah):
        i = abase + n_alt - n_ah + k
        flush.fill_(k & 0xFF)
        cache.swap_in(rpi, sl, topk_all[i], 0, out={"device_locs": locs})  # untimed: the call
        flush.fill_((k + 1) & 0xFF)
        ev_ah[k][0].record(s)
        cache.swap_in(rpi, sl, topk_all[i], 0, out={"device_locs": locs, "stats": ah_stats[k]})
        ev_ah[k][1].record(s)
    torch.cuda.synchronize()
    ah_ms = statistics.median(a.elapsed_time(b) for a, b in ev_ah)
    ah_misses = float(ah_stats[:, :, 3].sum(dim=1).float().mean())
    ceiling = copy_ceiling(torch, pkg, cache, w, dev, flush,
                           float(stats[base:base + K, :, 3].float().mean()))
    decode = decode_step_extra_page(torch, pkg, w, dev, flush, calls, pool,
                                    args.index == "dense", n=min(K, 20))
    pipeline = deferred_copy_pipeline(torch, pkg, w, dev, flush, calls, pool,
                                      args.index == "dense", n=min(K, 10))

    f1_t0 = time.time()
    f1 = multi_vs_sequential(torch, pkg, w, dev, flush, calls, pool, args.index == "dense",
                             n=min(K, 20), warmup=Wm)
    f1_t1 = time.time()
    clocks.stop()
    f1["clocks"] = clocks.summary(f1_t0, f1_t1)

    # ---- roofline bookkeeping (algorithmic bytes) ----
    U_timed = st_timed[:, :, 3].sum(axis=1).astype(np.float64)
    copy_bytes_timed = U_timed * w.row_bytes  # host-link bytes (same again written to HBM)
    achieved_copy = float(np.mean(copy_bytes_timed) / (np.mean(step_ms) * 1e-3) / 1e9)
    U_phase = st_phase[:, :, 3].sum(axis=1).astype(np.float64)
    m_phase = st_phase[:, :, 4].sum(axis=1).astype(np.float64)
    hs_phase = st_phase[:, :, 1].sum(axis=1).astype(np.float64)
    gather_bytes = 16.0 * w.entries + 16.0 * U_phase
    commit_bytes = 8.0 * w.hot_buffer * w.batch + 32.0 * m_phase + 4.0 * hs_phase
    copy_bytes_phase = U_phase * w.row_bytes

    def hbm_phase(nbytes, span_us):
        achieved = float(np.mean(nbytes / (np.asarray(span_us) * 1e-6)) / 1e9)
        return {"achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "peak_source": hbm_src,
                "algorithmic_bytes_per_launch": float(np.mean(nbytes)),
                "span_us_mean": float(np.mean(span_us))}

    traffic = NCU_TRAFFIC.get((args.config, args.index), {})
    gather_hbm = dict(hbm_phase(gather_bytes, timeline["gather_span_us"]),
                      span="first CTA start to the last CTA's locations and miss lists")
    commit_hbm = dict(hbm_phase(commit_bytes, timeline["commit_span_us"]),
                      span="first leader CTA's commit start to the last one's end "
                           "(each request's commit starts when its own lookup ends)",
                      per_request_commit_us_median=float(np.median(timeline["commit_us"])))
    copy_window = copy_bytes_phase / (np.asarray(timeline["copy_span_us"]) * 1e-6) / 1e9
    clk = clocks.summary(t_wall0, t_wall1)
    n_kernels = 1 + (1 if page_out is not None else 0)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": Wm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "data": "synthetic",
        "config": dict(config_dict(w, world), index=args.index, launch=(
            "one CUDA graph per step (the swap-in kernel%s), replayed; the step's top-k is "
            "staged into the graph's input buffer before the step's events"
            % (" and, on a second stream, the page table" if page_out is not None else "")
            if args.launch == "graph" else "direct launches through the C ABI")),
        "e2e": {"value": whole_job_rate(w.entries, world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(d2h_bytes),
                "ms_per_step": e2e_ms, **e2e_parts,
                "zero_copy": {"value": whole_job_rate(w.entries, world, zc_ms), "unit": UNIT,
                              "ms_per_step": zc_ms, "h2d_bytes_per_step": int(h2d_bytes),
                              "d2h_bytes_per_step": int(d2h_bytes),
                              "how": "pinned host input record and pinned output passed to "
                                     "the call; the kernels read and write them over "
                                     "NVLink-C2C (no copy-engine transfer)"}},
        "gpu_launches": K * n_kernels,
        "roofline": {"kernel": "swapin_kernel (lookup, de-duplication, locations, commit and "
                               "miss-row copy in one launch)",
                     "bound": "host_link", "achieved": achieved_copy, "peak": h2d_peak,
                     "unit": "GB/s", "frac": achieved_copy / h2d_peak,
                     "traffic": traffic.get("dram_bytes"),
                     "host_link_traffic": traffic.get("host_link_bytes"),
                     "traffic_note": ("traffic = DRAM read+write bytes per launch; "
                                      "host_link_traffic = system-memory read bytes per "
                                      "launch, the link this kernel is bound by; both from "
                                      "the ncu capture of this workload in " + NCU_CAPTURE)
                     if traffic else "no ncu capture of the current kernel on this workload",
                     "peak_source": "measured in this run: pinned host->device cudaMemcpyAsync "
                                    "256 MiB, best of 20",
                     "algorithmic_bytes_per_launch": float(np.mean(copy_bytes_timed)),
                     "duration": "mean event-timed step of the timed region (one launch "
                                 "of this kernel per step)"},
        "phases": {
            "kernel_ms_direct": float(np.mean(t_kernel)),
            "timeline_us": timeline["summary"],
            "gather_hbm": gather_hbm,
            "commit_hbm": commit_hbm,
            "dram_traffic": {
                "bytes_per_launch": traffic.get("dram_bytes"),
                "lookup_commit_algorithmic_bytes": float(np.mean(gather_bytes + commit_bytes)),
                "ratio": (traffic["dram_bytes"] / float(np.mean(gather_bytes + commit_bytes))
                          if traffic else None),
                "note": "DRAM read + write bytes of the whole launch (ncu, " + NCU_CAPTURE
                        + ") over the lookup's and the commit's algorithmic bytes; the copy's "
                          "device writes mostly stay in L2 within the launch"},
            "copy_window": {"gbs": float(np.mean(copy_window)), "peak": h2d_peak,
                            "frac": float(np.mean(copy_window)) / h2d_peak,
                            "span": "first lookup end to the last warp's copy end"},
            "unique_misses_per_step": float(np.mean(U_timed)),
            "miss_copy_mb_per_step": float(np.mean(U_timed)) * w.row_bytes / 1e6,
            "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms),
            "step_ms_max": max(step_ms),
            "other_launch_mode": {"launch": alt, "ms_per_step": alt_ms, "steps": n_alt,
                                  "value": whole_job_rate(w.entries, 1, alt_ms)},
            "all_hit_replay": {"ms_median": ah_ms, "unique_misses_per_step": ah_misses,
                               "copy_share_ms": statistics.median(step_ms) - ah_ms,
                               "how": "each call repeated at once (direct launches); the "
                                      "repeat finds its tokens resident and copies nothing "
                                      "when they fit the hot buffer (an overflowing "
                                      "workload still misses: see unique_misses_per_step)"},
        },
        "multi_vs_sequential": f1,
        "copy_ceiling": ceiling,
        "decode_step_extra_page": decode,
        "deferred_copy_pipeline": pipeline,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:  # the oracle baseline: N = 1 only
        line["cpu_baseline"] = cpu_baseline_oracle(w, calls, rpi_np, sl_np, args.cpu_seconds,
                                                   pool.numpy())
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
