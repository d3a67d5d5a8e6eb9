"""Routed-attention throughput benchmark (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 720p|1080p|480p]
                    [--impl ours|reference]

A step is one steady-state pass of the hot path for one layer: the fused
append/evict of the current block's K/V into the restructured cache
(hc_cache_append) followed by routed attention of the block's queries
(hc_routed_attention).  The cache was built by the one-time pipeline
(hc_classify on the window that just filled, then hc_cache_restructure),
which is timed separately, as is the in-house full attention
(hc_full_attention) on the same queries and window.

value     query tokens/s over the K timed steps, inputs resident in HBM,
          L2 flushed (512 MB write) before every step, CUDA events on the
          launching stream; the sum over ranks for N > 1 (replicas, weak
          scaling, no collective on the data path).
e2e       the same metric through the same calls with HOST buffers: each
          step copies Q and the block's K/V from pinned host memory and
          copies O back, inside the timed region.
roofline  the routed-attention kernel: algorithmic FLOPs per launch
          (4*Nq*|keys|*d per head over its own key set) / its mean event
          time, against the measured dense bf16 peak.
cpu_baseline  the fp64 NumPy oracle on a bounded sample of the same step
          (rank 0 only).

--impl reference runs that oracle as the benchmark's reference arm.
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
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "routed-attention query tokens/s at 720P/1080P shapes; x vs own full-attn; %roofline"
UNIT = "query-tok/s"
FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="720p", choices=["480p", "720p", "1080p", "rollout", "sweep", "agreement", "stability"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-paths", action="store_true",
                    help="skip the per-pathway timing (every head on one pathway)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the 480P and 1080P layer lines")
    return ap.parse_args()


def workload_config(shape):
    mix = "".join("SDPG"[a] for a in shape.mix)
    return {"workload": f"{shape.name} layer", "n_heads": shape.n_heads, "head_dim": shape.head_dim,
            "frame": f"{shape.frame_h}x{shape.frame_w}", "block_frames": shape.frames_per_block,
            "window_frames": shape.window_frames, "query_tokens": shape.n_q,
            "window_keys": shape.n_k, "head_mix": mix,
            "step": "hc_cache_append + hc_routed_attention",
            "l2": "flushed before every step (512 MB write)",
            "parallelism": "replicas (one independent layer per GPU)"}


def routed_flops(shape, labels, sliding=False):
    """Algorithmic FLOPs of routed attention: 4*|q|*|keys|*d per (query, head)
    (Spatial: the query's cell, or with `sliding` its clipped centred window)."""
    F, d, nq = shape.frame_tokens, shape.head_dim, shape.n_q
    total = 0
    for a in labels:
        if a in (synth.SINK, synth.DUMMY):
            keys = nq * shape.n_q
        elif a == synth.GLOBAL:
            keys = nq * shape.n_k
        elif sliding:
            keys = nq * shape.window_frames * _window_sum(shape.frame_h) * _window_sum(shape.frame_w) // (
                shape.frame_h * shape.frame_w)
        else:
            keys = 0
            for hz in _cells(shape.frame_h):
                for wz in _cells(shape.frame_w):
                    c = hz * wz
                    keys += (shape.frames_per_block * c) * (shape.window_frames * c)
        total += 4 * keys * d
    return total


def _window_sum(n, c=10):
    """Sum over positions x in [0, n) of the clipped length of the window
    [x - c//2, x - c//2 + c) on an axis of length n."""
    return sum(min(n, x - c // 2 + c) - max(0, x - c // 2) for x in range(n))


def _cells(n, c=10):
    k = max(1, int(n / c + 0.5))
    return [c] * (k - 1) + [n - c * (k - 1)]


def routed_bytes(shape, labels, esize=2):
    """Algorithmic bytes: every head's key set K and V read once, Q read once, O written once."""
    F, d, nq = shape.frame_tokens, shape.head_dim, shape.n_q
    kv = 0
    for a in labels:
        rows = nq if a in (synth.SINK, synth.DUMMY) else shape.n_k
        kv += 2 * rows * d * esize
    return kv + 2 * nq * shape.n_heads * d * esize


def path_measurements(hc, shape, cfg, k, v, q, o, flush, stream, reps, peak_tf, peak_bw):
    """Routed attention with every head on one pathway (the per-path rows of
    the method): mean CUDA-event time over `reps` launches, L2 flushed before
    each, with its algorithmic FLOP and byte rates against the measured peaks."""
    import torch
    out = {}
    for arch, name in ((synth.SINK, "sink"), (synth.DUMMY, "dummy"), (synth.SPATIAL, "spatial"),
                       (synth.GLOBAL, "global"), (synth.SPATIAL, "spatial_sliding")):
        labels = [arch] * shape.n_heads
        ccfg = hc.config_for(shape, spatial_mode=hc.HC_SPATIAL_SLIDING) if name == "spatial_sliding" else cfg
        cache = hc.hc_cache_create(ccfg, labels, device=q.device)
        cache.restructure(k, v, 0)
        times = []
        for i in range(reps + 3):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            cache.routed_attention(q, o)
            b.record(stream)
            if i >= 3:
                times.append((a, b))
        torch.cuda.synchronize()
        ms = statistics.mean(x.elapsed_time(y) for x, y in times)
        fl = routed_flops(shape, labels, sliding=name == "spatial_sliding")
        by = routed_bytes(shape, labels)
        out[name] = {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12, "gbs": by / (ms * 1e-3) / 1e9,
                     "frac_tensor": fl / (ms * 1e-3) / 1e12 / peak_tf,
                     "frac_hbm": by / (ms * 1e-3) / 1e9 / peak_bw,
                     "flops": fl, "bytes": by}
        cache.close()
        del cache
    return out


def timed_launches(fn, reps, flush, stream, warm=3):
    """Mean CUDA-event time (ms) of fn() over `reps` launches on `stream`,
    after `warm` untimed ones, with L2 flushed before each."""
    import torch
    evs = []
    for i in range(reps + warm):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        if i >= warm:
            evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.mean(x.elapsed_time(y) for x, y in evs)


def other_layers(hc, names, dev, stream, flush, peak_tf, clock_index, reps=10):
    """The other layer shapes the metric is quoted at: for each, the planted
    window is classified, the cache restructured from the labels the library
    returned, and routed attention of the block's queries and the library's
    full attention on the same inputs are timed (CUDA events, L2 flushed
    before every launch, clocks sampled meanwhile)."""
    import torch
    out = {}
    for name in names:
        shape = synth.SHAPES[name]
        inp = synth.make_layer(shape)

        def to_dev(x):
            return torch.from_numpy(x.raw.view(np.int16).copy()).view(torch.bfloat16).to(dev)

        q, k, v = to_dev(inp.q), to_dev(inp.k), to_dev(inp.v)
        del inp
        cfg = hc.config_for(shape)
        scratch = torch.empty(hc.hc_classify_scratch_bytes(cfg), dtype=torch.uint8, device=dev)
        labels_dev = torch.empty(shape.n_heads, dtype=torch.int8, device=dev)
        labels, _, _ = hc.hc_classify(cfg, q, k, v, labels_dev=labels_dev, scratch=scratch)
        if list(labels) != list(shape.mix):
            raise RuntimeError(f"{name}: classification gave {list(labels)}, planted {list(shape.mix)}")
        cache = hc.hc_cache_create(cfg, labels, device=dev)
        cache.restructure(k, v, 0)
        o = torch.empty_like(q)
        clock = ClockSampler(clock_index)
        clock.start()
        routed_ms = timed_launches(lambda: cache.routed_attention(q, o), reps, flush, stream)
        full_ms = timed_launches(lambda: hc.hc_full_attention(cfg, q, k, v, o=o), max(3, reps // 2), flush, stream)
        classify_ms = timed_launches(lambda: hc.hc_classify(cfg, q, k, v, labels_dev=labels_dev, scratch=scratch,
                                                            copy_labels=False), 3, flush, stream, warm=1)
        clocks = clock.stop()
        hc.hc_get_last_error()
        fl = routed_flops(shape, labels)
        achieved = fl / (routed_ms * 1e-3) / 1e12
        out[name] = {"routed_attention_ms": routed_ms, "query_tok_s": shape.n_q / (routed_ms * 1e-3),
                     "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                                  "frac": achieved / peak_tf, "algorithmic_flops_per_launch": fl},
                     "full_attention_ms": full_ms, "speedup_vs_full_attention": full_ms / routed_ms,
                     "classify_ms": classify_ms, "split_bytes": cache.info()["split_bytes"],
                     "clocks": clocks, "config": workload_config(shape)}
        cache.close()
        del cache, q, k, v, o, scratch
        torch.cuda.empty_cache()
    return out


def max_over_ranks(ms, dist, device):
    """The slowest rank's time: the job's time for weak scaling."""
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank_step, steps, max_ms, world):
    """Whole-job throughput: the units all ranks processed / the max time."""
    return world * units_per_rank_step * steps / (max_ms * 1e-3)


def cache_kernel_rates(shape, labels, restructure_ms, append_ms, peak_bw):
    """HBM rates of the cache kernels (bytes they must move / CUDA-event time):
    the restructure reads the whole monolithic window and writes every head's
    region; a steady-state append of a later block reads the block's K/V and
    writes it for every head but the Sink heads (block 0 only)."""
    row = 2 * shape.head_dim * 2                       # K and V of one (token, head), bf16
    window_rows = shape.n_k * shape.n_heads
    region_rows = sum(shape.n_q if a in (synth.SINK, synth.DUMMY) else shape.n_k for a in labels)
    restructure_b = row * (window_rows + region_rows)
    append_b = row * (shape.n_q * shape.n_heads + shape.n_q * sum(1 for a in labels if a != synth.SINK))
    out = {}
    for name, b, ms in (("restructure", restructure_b, restructure_ms), ("append", append_b, append_ms)):
        gbs = b / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "bytes": b, "gbs": gbs, "frac_hbm": gbs / peak_bw}
    return out


class ClockSampler:
    """nvidia-smi samples taken while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.25)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks(sustained=False):
    """(bf16 TF/s, HBM GB/s, "measured" | "fallback").  sustained=True gives the
    bf16 figure of a seconds-long loop under the power cap, the denominator for
    work timed over a long run; the default is the burst figure."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        tf = j.get("bf16_tflops", 1800.0)
        if sustained:
            tf = j.get("bf16_tflops_sustained", tf)
        return tf, j.get("hbm_gbs", 6400.0), "measured"
    return (1400.0 if sustained else 1800.0), 6400.0, "fallback"


KERNEL_SOURCES = ("attn_tc.cu", "hc_internal.h")   # the attention kernel's own code


def kernel_source_hash():
    import hashlib
    src = os.path.join(ROOT, "head_routed_kv_classify_b300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(src, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_from_profile(kernel_tag):
    """Per-launch DRAM bytes recorded by an ncu capture of the current kernel
    source (attn_tc.cu and hc_internal.h), or None if none matches."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return None
    digest = kernel_source_hash()
    tb, sha = None, None
    for line in open(path):
        if line.startswith("traffic_bytes_per_launch:"):
            tb = float(line.split(":", 1)[1].split()[0])
        if line.startswith("csrc_sha256_16:"):
            sha = line.split(":", 1)[1].strip()
    return tb if (tb is not None and sha == digest) else None


# --------------------------------------------------------------------------- oracle arms

class OracleStep:
    """The oracle's routed attention for a query sample of one layer.

    Set-up (untimed) puts the window's blocks in the oracle's cache model and
    takes each head's pathway keys and values out of it once (the oracle's
    routed_attention rebuilds the whole window for every head on every call,
    several seconds at 720P that would swamp a small sample); a timed step
    then runs the oracle's own attention routines on the sample: the dense
    softmax attention for Sink, Dummy and Global heads and the per-position
    cell attention for Spatial heads."""

    def __init__(self, shape, inp, labels):
        from oracle import headcast_ref as ref
        self.ref = ref
        self.geom = ref.geometry_of(shape)
        cache = ref.CacheModel(self.geom)
        blk = shape.n_q
        for b in range(shape.blocks_per_window):
            cache.put(b, inp.k.values[b * blk:(b + 1) * blk], inp.v.values[b * blk:(b + 1) * blk])
        win_k, win_v = cache.window()
        sink_k, sink_v = cache.sink()
        cur_k, cur_v = cache.current()
        self.q = inp.q.values
        self.scale = ref.default_scale(shape.head_dim)
        self.labels = [int(a) for a in labels]
        self.kv = []
        for h, a in enumerate(self.labels):
            k, v = {ref.SINK: (sink_k, sink_v), ref.DUMMY: (cur_k, cur_v)}.get(a, (win_k, win_v))
            self.kv.append((np.ascontiguousarray(k[:, h, :]), np.ascontiguousarray(v[:, h, :])))
        self.n_q = shape.n_q

    def __call__(self, n_queries, seed):
        ref = self.ref
        n_queries = min(n_queries, self.n_q)
        idx = np.sort(np.random.default_rng(seed).choice(self.n_q, n_queries, replace=False))
        t0 = time.perf_counter()
        for h, a in enumerate(self.labels):
            qh = np.asarray(self.q[:, h, :], np.float64)
            kh, vh = self.kv[h]
            if a == ref.SPATIAL:
                ref.attend_by_position(qh, kh, vh, self.geom, kh.shape[0] // self.geom.F, ref.cell_keys,
                                       self.scale, idx)
            else:
                ref.attend_chunked(qh[idx], kh, vh, self.scale)
        return time.perf_counter() - t0


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(shape, inp, labels, seconds):
    """The oracle as it stands, on growing query samples until ~seconds of work."""
    step = OracleStep(shape, inp, labels)
    done, spent, n = 0, 0.0, min(16, shape.n_q)
    seed = 0
    while spent < seconds:
        spent += step(n, seed)
        done += n
        seed += 1
        n = min(2 * n, 256)
    return {"value": done / spent, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"{done} query tokens (all {shape.n_heads} heads, routed key sets) of the "
                      f"{shape.name} layer, fp64 NumPy, {spent:.1f} s"}


def run_reference(args, shape, rank, world, budget_s=150.0):
    """The oracle as the reference arm: every step is a query sample of the
    same workload, sized (from an untimed calibration step) so that warm-up
    and timed steps together take about `budget_s` of host time."""
    if rank != 0:
        return
    inp = synth.make_layer(shape)
    labels = np.array(shape.mix, np.int8)
    step = OracleStep(shape, inp, labels)
    per_query = step(8, 999) / 8
    nq = int(max(1, min(256, shape.n_q, budget_s / max(1, args.steps + args.warmup) / per_query)))
    for s in range(args.warmup):
        step(nq, 1000 + s)
    t = 0.0
    for s in range(args.steps):
        t += step(nq, s)
    value = nq * args.steps / t
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(shape),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "sample": f"{nq} query tokens per step (all {shape.n_heads} heads, routed "
                                       f"key sets) of the {shape.name} layer, fp64 NumPy"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- 30-layer rollout

def run_rollout(args, rank, world, local_rank):
    """The 30-layer 720P rollout.  Every layer's window (seeded, with its own
    per-(layer, head) archetypes planted) is classified by hc_classify and
    the layer's cache is restructured from the labels the library returned;
    then 7 further AR blocks x 4 denoising steps of append + routed attention
    run over all 30 layers.  One timed step is one denoising step of the
    whole stack (30 appends + 30 routed launches).  The classifications are
    timed separately, as the pages report them, and the same steps are run
    through the library's full attention over monolithic per-layer rings.

    Inputs: the per-layer windows are the ones the oracle golden files
    classify (seed 4*100 + layer); the steady-state blocks are a pool of 4
    seeded blocks that the (layer, block, step) triples cycle through, since
    fresh draws for all 840 triples would be 83 GB of host data."""
    import concurrent.futures as cf
    import torch
    import head_routed_kv_classify_b300 as hc
    from head_routed_kv_classify_b300 import build as hcb

    if not os.path.exists(hc.LIB_PATH):
        hcb.build()
    hc.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    R = synth.ROLLOUT_720P
    shape, L, NB, NS = R["shape"], R["layers"], R["blocks"], R["steps"]
    mix = synth.rollout_mix(L, shape.n_heads, R["seed"] + 1000 * rank)

    def to_dev(x):
        return torch.from_numpy(x.raw.view(np.int16).copy()).view(torch.bfloat16).to(dev)

    cfg = hc.config_for(shape)
    pool = [synth.make_block(shape, seed=R["seed"] + 50 + i + 1000 * rank, mix=mix[0]) for i in range(4)]
    qb = [to_dev(b[0]) for b in pool]
    kb = [to_dev(b[1]) for b in pool]
    vb = [to_dev(b[2]) for b in pool]
    o = torch.empty_like(qb[0])

    def ev():
        return torch.cuda.Event(enable_timing=True)

    # One-time phase, per layer: classify its window, then restructure it
    # into the layer's cache by the returned labels.  The windows are drawn
    # on host threads ahead of the device work.
    scratch = torch.empty(hc.hc_classify_scratch_bytes(cfg), dtype=torch.uint8, device=dev)
    labels_dev = torch.empty(shape.n_heads, dtype=torch.int8, device=dev)
    caches, classify_ms, labels_all = [], 0.0, []

    def window(layer):
        return synth.make_layer(shape, seed=R["seed"] * 100 + layer + 1000 * rank,
                                mix=tuple(int(a) for a in mix[layer]))

    with cf.ThreadPoolExecutor(max_workers=min(4, os.cpu_count() or 1)) as ex:
        futs = [ex.submit(window, layer) for layer in range(L)]
        for layer in range(L):
            inp = futs[layer].result()
            futs[layer] = None
            q0, k, v = to_dev(inp.q), to_dev(inp.k), to_dev(inp.v)
            del inp
            if layer == 0:   # untimed first call
                hc.hc_classify(cfg, q0, k, v, labels_dev=labels_dev, scratch=scratch, copy_labels=False)
            e0, e1 = ev(), ev()
            torch.cuda.synchronize()
            e0.record(stream)
            hc.hc_classify(cfg, q0, k, v, labels_dev=labels_dev, scratch=scratch, copy_labels=False)
            e1.record(stream)
            labels = labels_dev.cpu().numpy()
            classify_ms += e0.elapsed_time(e1)
            labels_all.append("".join("SDPG"[int(a)] for a in labels))
            c = hc.hc_cache_create(cfg, labels, device=dev)
            c.restructure(k, v, 0)
            caches.append(c)
            del q0, k, v
    hc.hc_get_last_error()
    agree = sum(int(a == "".join("SDPG"[int(x)] for x in m)) for a, m in zip(labels_all, mix))
    k, v = None, None
    first = shape.blocks_per_window
    cache_bytes = sum(c.info()["bytes"] for c in caches)
    mono_bytes = sum(c.info()["monolithic_bytes"] for c in caches)

    def step(s, routed=True):
        blk, st = divmod(s, NS)
        for layer in range(L):
            i = (layer + blk + st) % 4
            caches[layer].append(first + blk, kb[i], vb[i])
            caches[layer].routed_attention(qb[i], o)

    for s in range(min(args.warmup, NS)):
        step(s)
    torch.cuda.synchronize()
    hc.hc_get_last_error()
    clock = ClockSampler(local_rank) if rank == 0 else None
    if clock:
        clock.start()
    n_steps = NB * NS
    evs = [(ev(), ev()) for _ in range(n_steps)]
    torch.cuda.synchronize()
    for s in range(n_steps):
        evs[s][0].record(stream)
        step(s)
        evs[s][1].record(stream)
    torch.cuda.synchronize()
    clocks = clock.stop() if clock else None
    hc.hc_get_last_error()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = sum(step_ms)

    # The same steps through full attention over per-layer monolithic rings
    # (zero-filled: the values do not change the time).
    rings = [(torch.zeros((shape.n_k, shape.n_heads, shape.head_dim), dtype=torch.bfloat16, device=dev),
              torch.zeros((shape.n_k, shape.n_heads, shape.head_dim), dtype=torch.bfloat16, device=dev))
             for _ in range(L)]
    full_steps = min(n_steps, 8)
    fe = [(ev(), ev()) for _ in range(full_steps)]
    for s in range(full_steps):
        blk, st = divmod(s, NS)
        slot = (first + blk) % shape.blocks_per_window
        rows = slice(slot * shape.n_q, (slot + 1) * shape.n_q)
        fe[s][0].record(stream)
        for layer in range(L):
            i = (layer + blk + st) % 4
            kr, vr = rings[layer]
            kr[rows].copy_(kb[i], non_blocking=True)
            vr[rows].copy_(vb[i], non_blocking=True)
            hc.hc_full_attention(cfg, qb[i], kr, vr, o=o)
        fe[s][1].record(stream)
    torch.cuda.synchronize()
    full_step_ms = statistics.mean(a.elapsed_time(b) for a, b in fe)
    if rank != 0:
        return
    # The timed region runs for seconds at the power cap: sustained peak.
    peak_tf, peak_bw, peak_kind = measured_peaks(sustained=True)
    burst_tf = measured_peaks()[0]
    flops = sum(routed_flops(shape, ["SDPG".index(a) for a in labels_all[layer]]) for layer in range(L))
    achieved = flops / (statistics.mean(step_ms) * 1e-3) / 1e12
    value = world * L * shape.n_q * n_steps / (total_ms * 1e-3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": n_steps,
        "warmup": min(args.warmup, NS), "ms_per_step": total_ms / n_steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (per-layer seeded windows with planted archetypes, classified by the library; "
                "a pool of 4 seeded blocks; 720P shapes)",
        "config": {"workload": "720p rollout", "layers": L, "n_heads": shape.n_heads,
                   "head_dim": shape.head_dim, "frame": f"{shape.frame_h}x{shape.frame_w}",
                   "blocks": NB, "denoising_steps": NS, "window_frames": shape.window_frames,
                   "step": "30 x (hc_cache_append + hc_routed_attention)",
                   "l2": f"inputs larger than L2 (30 layers' caches, {cache_bytes / 1e9:.1f} GB)",
                   "head_mix": "uniform over the 4 archetypes per (layer, head), seed 4"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": None,
                     "kernel": "one denoising step (30 appends + 30 routed launches)",
                     "algorithmic_flops_per_step": flops,
                     "frac_of_burst_peak": achieved / burst_tf,
                     "peak_source": f"{peak_kind} bf16 dense (sustained, seconds-long loop at the power cap)"},
        "gpu_launches": n_steps * sum(2 + (1 if c.info()["split_bytes"] else 0) for c in caches),
        "clocks": clocks,
        "full_attention_step_ms": full_step_ms,
        "step_speedup_vs_full": full_step_ms / (total_ms / n_steps),
        "classify_ms_all_layers": classify_ms,
        "classification_overhead_pct": 100.0 * classify_ms / (classify_ms + total_ms),
        "labels_match_planted_layers": agree, "labels": labels_all,
        "cache_bytes": cache_bytes, "monolithic_cache_bytes": mono_bytes,
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- threshold sweep

def run_sweep(args, rank, world, local_rank):
    """The FPS side of the threshold ablation (Figure 5 caption of the Pith
    review of HeadCast): on the planted 720P layer, classify with theta (all
    three cosine gates) over a grid at theta_sc = 0.755, and with theta_sc over
    a grid at theta = 0.95; for each setting, the archetype mix the classifier
    picks, the steady-state cache bytes, the routed-attention time and its
    speedup over full attention.  (The quality side needs a trained model.)"""
    import torch
    import head_routed_kv_classify_b300 as hc
    from head_routed_kv_classify_b300 import build as hcb

    if not os.path.exists(hc.LIB_PATH):
        hcb.build()
    hc.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    shape = synth.SHAPES["720p"]
    inp = synth.make_layer(shape, seed=shape.seed + 1000 * rank)

    def to_dev(x):
        return torch.from_numpy(x.raw.view(np.int16).copy()).view(torch.bfloat16).to(dev)

    q, k, v = to_dev(inp.q), to_dev(inp.k), to_dev(inp.v)
    o = torch.empty_like(q)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def timed(fn, reps):
        evs = []
        for i in range(reps + 3):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            if i >= 3:
                evs.append((a, b))
        torch.cuda.synchronize()
        return statistics.mean(x.elapsed_time(y) for x, y in evs)

    base = hc.config_for(shape)
    full_ms = timed(lambda: hc.hc_full_attention(base, q, k, v, o=o), 5)
    # The planted heads clear their gates by wide margins, so theta has to
    # come down to where unplanted (Global) heads' similarities lie before
    # the mix, and with it the FPS side, moves.
    grid = [(t, 0.755) for t in (0.20, 0.30, 0.40, 0.50, 0.60, 0.70, 0.80, 0.90, 0.95, 0.99)]
    grid += [(0.95, sc) for sc in (0.50, 0.70, 0.85, 0.95, 0.99)]
    rows = []
    for theta, theta_sc in grid:
        cfg = hc.config_for(shape, theta_sink=theta, theta_dummy=theta, theta_spatial=theta,
                            theta_score=theta_sc)
        labels, _, _ = hc.hc_classify(cfg, q, k, v)
        cache = hc.hc_cache_create(cfg, labels, device=dev)
        cache.restructure(k, v, 0)
        ms = timed(lambda: cache.routed_attention(q, o), 10)
        rows.append({"theta": theta, "theta_sc": theta_sc,
                     "mix": "".join("SDPG"[int(a)] for a in labels),
                     "routed_ms": ms, "speedup_vs_full": full_ms / ms,
                     "cache_bytes": cache.info()["bytes"]})
        cache.close()
    hc.hc_get_last_error()
    if rank != 0:
        return
    at_default = [r for r in rows if r["theta"] == 0.95 and r["theta_sc"] == 0.755][0]
    line = {"metric": METRIC, "value": shape.n_q / (at_default["routed_ms"] * 1e-3), "unit": UNIT,
            "n_gpus": world, "steps": 10, "warmup": 3, "ms_per_step": at_default["routed_ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) Q/K/V with planted archetypes; 720P shapes)",
            "config": {"workload": "720p threshold sweep", "planted_mix": "".join("SDPG"[a] for a in shape.mix),
                       "l2": "flushed before every launch (512 MB write)"},
            "full_attention_ms": full_ms, "sweep": rows}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- proxy vs deployed

def run_agreement(args, rank, world, local_rank):
    """How well the classifier's Spatial proxy (the (2r+1)x(2r+1)
    neighbourhood, r = 2) stands for the deployed path (the query's 10x10
    cell), the comparison the Pith review of HeadCast asks for (major comment
    2): every layer is classified twice, once with each proxy, and the line
    reports per head c_spatial, P5, MSE and score under both, and how many
    labels agree.  Layers: the planted 720P layer and the first six layers of
    the 30-layer rollout mix."""
    import torch
    import head_routed_kv_classify_b300 as hc
    from head_routed_kv_classify_b300 import build as hcb

    if not os.path.exists(hc.LIB_PATH):
        hcb.build()
    hc.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    shape = synth.SHAPES["720p"]
    R = synth.ROLLOUT_720P
    mixes = [tuple(shape.mix)] + [tuple(int(a) for a in m) for m in synth.rollout_mix(R["layers"], shape.n_heads, R["seed"])[:6]]

    def to_dev(x):
        return torch.from_numpy(x.raw.view(np.int16).copy()).view(torch.bfloat16).to(dev)

    layers, agree, total, t_ms = [], 0, 0, []
    for n, mix in enumerate(mixes):
        inp = synth.make_layer(shape, seed=(shape.seed if n == 0 else R["seed"] * 100 + n - 1) + 1000 * rank, mix=mix)
        q, k, v = to_dev(inp.q), to_dev(inp.k), to_dev(inp.v)
        out = {}
        for mode, name in ((hc.HC_PROXY_NEIGHBOURHOOD, "neighbourhood"), (hc.HC_PROXY_CELL, "cell")):
            cfg = hc.config_for(shape, proxy_mode=mode)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            labels, _, stats = hc.hc_classify(cfg, q, k, v)
            b.record()
            torch.cuda.synchronize()
            t_ms.append((name, a.elapsed_time(b)))
            out[name] = (labels, stats.cpu().numpy())
        ln, sn = out["neighbourhood"]
        lc, sc = out["cell"]
        agree += int(np.sum(ln == lc))
        total += len(ln)
        layers.append({"planted": "".join("SDPG"[a] for a in mix),
                       "labels_neighbourhood": "".join("SDPG"[int(a)] for a in ln),
                       "labels_cell": "".join("SDPG"[int(a)] for a in lc),
                       "c_spatial": [[round(float(x), 4), round(float(y), 4)] for x, y in zip(sn[:, 2], sc[:, 2])],
                       "p5": [[round(float(x), 4), round(float(y), 4)] for x, y in zip(sn[:, 3], sc[:, 3])],
                       "score": [[round(float(x), 4), round(float(y), 4)] for x, y in zip(sn[:, 5], sc[:, 5])]})
    hc.hc_get_last_error()
    if rank != 0:
        return
    cls_ms = statistics.mean(t for nm, t in t_ms if nm == "neighbourhood")
    line = {"metric": METRIC, "value": None, "unit": UNIT, "n_gpus": world, "steps": len(mixes),
            "warmup": 0, "ms_per_step": cls_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) Q/K/V with planted archetypes; 720P shapes)",
            "config": {"workload": "720p proxy vs deployed Spatial agreement", "layers": len(mixes),
                       "stat_pairs": "[neighbourhood proxy, deployed cell] per head"},
            "label_agreement": agree / total, "heads": total,
            "classify_ms": {nm: statistics.mean(t for m, t in t_ms if m == nm) for nm in ("neighbourhood", "cell")},
            "layers": layers}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- stability

def run_stability(args, rank, world, local_rank):
    """Re-classification stability on synthetic streams (the pages report the
    share of identical archetypes across AR steps; Pith review of HeadCast,
    "Core claim" / major comment 1).  A 480P-shaped layer (2/3/4/3 planted
    heads) streams 13 blocks whose planted structure persists; after the
    window first fills (block 6) a fraction `drift` of each planted query
    term is replaced by an unrelated one.  The layer is classified at block 6
    and again at blocks 7, 9 and 12, each time over the Sink block plus the
    six newest blocks, and the line reports the share of heads whose label is
    unchanged, per drift level.  (The timestep axis needs a diffusion model.)"""
    import torch
    import head_routed_kv_classify_b300 as hc
    from head_routed_kv_classify_b300 import build as hcb

    if not os.path.exists(hc.LIB_PATH):
        hcb.build()
    hc.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    shape = synth.SHAPES["480p"]
    cfg = hc.config_for(shape)
    fill = shape.blocks_per_window - 1
    checks = (fill + 1, fill + 3, fill + 6)

    def to_dev(x):
        return torch.from_numpy(x.raw.view(np.int16).copy()).view(torch.bfloat16).to(dev)

    results = []
    for drift in (0.0, 0.3, 0.6):
        blocks = synth.make_stream(shape, seed=shape.seed + 500 + 1000 * rank, n_blocks=checks[-1] + 1,
                                   drift=drift)
        dq = [to_dev(b[0]) for b in blocks]
        dk = [to_dev(b[1]) for b in blocks]
        dv = [to_dev(b[2]) for b in blocks]

        def classify_at(b):
            ids = [0] + list(range(b - shape.blocks_per_window + 2, b + 1))
            k = torch.cat([dk[i] for i in ids])
            v = torch.cat([dv[i] for i in ids])
            labels, _, _ = hc.hc_classify(cfg, dq[b], k, v)
            return labels

        first = classify_at(fill)
        row = {"drift": drift, "labels_at_fill": "".join("SDPG"[int(a)] for a in first),
               "planted": "".join("SDPG"[a] for a in shape.mix), "later": []}
        for b in checks:
            lab = classify_at(b)
            row["later"].append({"block": b, "labels": "".join("SDPG"[int(a)] for a in lab),
                                 "identical": float(np.mean(lab == first))})
        row["identical_mean"] = float(np.mean([x["identical"] for x in row["later"]]))
        results.append(row)
        del dq, dk, dv, blocks
    hc.hc_get_last_error()
    if rank != 0:
        return
    line = {"metric": METRIC, "value": None, "unit": UNIT, "n_gpus": world, "steps": len(checks),
            "warmup": 0, "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded streams with persistent planted archetypes and query drift; 480P shapes)",
            "config": {"workload": "480p re-classification stability",
                       "window_at_block_b": "block 0 (Sink) + blocks b-5..b"},
            "stability": results}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- our arm

def run_ours(args, shape, rank, world, local_rank):
    import torch
    import head_routed_kv_classify_b300 as hc
    from head_routed_kv_classify_b300 import build as hcb

    if not os.path.exists(hc.LIB_PATH):
        hcb.build()
    hc.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()
    dist = None
    if world > 1:
        import torch.distributed as dist

    def to_dev(x):
        return torch.from_numpy(x.raw.view(np.int16).copy()).view(torch.bfloat16).to(dev)

    inp = synth.make_layer(shape, seed=shape.seed + 1000 * rank)
    q, k, v = to_dev(inp.q), to_dev(inp.k), to_dev(inp.v)
    cfg = hc.config_for(shape)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    # One-time pipeline: classify the window that just filled, then restructure.
    scratch = torch.empty(hc.hc_classify_scratch_bytes(cfg), dtype=torch.uint8, device=dev)
    labels_dev = torch.empty(shape.n_heads, dtype=torch.int8, device=dev)
    stats_dev = torch.empty((shape.n_heads, 6), dtype=torch.float32, device=dev)
    for _ in range(2):
        hc.hc_classify(cfg, q, k, v, labels_dev=labels_dev, stats_dev=stats_dev, scratch=scratch,
                       copy_labels=False)
    flush.zero_()
    e0, e1 = ev(), ev()
    e0.record(stream)
    labels, _, _ = hc.hc_classify(cfg, q, k, v, labels_dev=labels_dev, stats_dev=stats_dev,
                                  scratch=scratch)
    e1.record(stream)
    torch.cuda.synchronize()
    classify_ms = e0.elapsed_time(e1)
    if list(labels) != list(shape.mix):
        raise RuntimeError(f"classification gave {list(labels)}, planted {list(shape.mix)}")
    cache = hc.hc_cache_create(cfg, labels, device=dev)
    # Restructuring the same window again rewrites the same rows: two untimed
    # calls, then the median of five, each after an L2 flush.
    for _ in range(2):
        cache.restructure(k, v, 0)
    restructure_times = []
    for _ in range(5):
        flush.zero_()
        e0.record(stream)
        cache.restructure(k, v, 0)
        e1.record(stream)
        torch.cuda.synchronize()
        restructure_times.append(e0.elapsed_time(e1))
    restructure_ms = float(np.median(restructure_times))

    # Steady-state inputs: two fresh blocks alternate (4 denoising steps per block).
    blocks = [synth.make_block(shape, seed=shape.seed + 77 + i + 1000 * rank) for i in range(2)]
    qb = [to_dev(b[0]) for b in blocks]
    kb = [to_dev(b[1]) for b in blocks]
    vb = [to_dev(b[2]) for b in blocks]
    o = torch.empty_like(q)
    state = {"step": 0}
    first_block = shape.blocks_per_window

    def block_id():
        return first_block + state["step"] // 4

    def step(i, evs):
        flush.zero_()
        s0, s1, r0 = evs
        s0.record(stream)
        cache.append(block_id(), kb[i % 2], vb[i % 2])
        r0.record(stream)
        cache.routed_attention(qb[i % 2], o)
        s1.record(stream)
        state["step"] += 1

    for i in range(args.warmup):
        step(i, (ev(), ev(), ev()))
    torch.cuda.synchronize()
    hc.hc_get_last_error()

    clock = ClockSampler(local_rank) if rank == 0 else None
    if clock:
        clock.start()
    evs = [(ev(), ev(), ev()) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        step(i, evs[i])
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks = clock.stop() if clock else None
    hc.hc_get_last_error()
    step_ms = [a.elapsed_time(b) for a, b, _ in evs]
    routed_ms = [r.elapsed_time(b) for _, b, r in evs]
    total_ms = sum(step_ms)
    if dist:
        total_ms = max_over_ranks(total_ms, dist, dev)

    # In-house full attention on the same queries over the monolithic window,
    # plus the monolithic-ring append it needs (one contiguous copy per block).
    k_ring, v_ring = k.clone(), v.clone()
    full_ms, mono_ms = [], []
    nfull = max(5, min(args.steps, 30))
    for i in range(args.warmup + nfull):
        flush.zero_()
        a0, a1, a2 = ev(), ev(), ev()
        a0.record(stream)
        slot = (first_block + i // 4) % shape.blocks_per_window
        rows = slice(slot * shape.n_q, (slot + 1) * shape.n_q)
        k_ring[rows].copy_(kb[i % 2], non_blocking=True)
        v_ring[rows].copy_(vb[i % 2], non_blocking=True)
        a1.record(stream)
        hc.hc_full_attention(cfg, qb[i % 2], k_ring, v_ring, o=o)
        a2.record(stream)
        if i >= args.warmup:
            full_ms.append((a1, a2))
            mono_ms.append((a0, a1))
    torch.cuda.synchronize()
    full_ms = [a.elapsed_time(b) for a, b in full_ms]
    mono_ms = [a.elapsed_time(b) for a, b in mono_ms]

    peak_tf, peak_bw, peak_kind = measured_peaks()
    paths = None
    if not args.no_paths:
        paths = path_measurements(hc, shape, cfg, k, v, q, o, flush, stream, 10, peak_tf, peak_bw)
    workloads = None
    if not args.no_workloads and rank == 0:
        others = [n for n in ("480p", "1080p") if n != shape.name]
        workloads = other_layers(hc, others, dev, stream, flush, peak_tf, local_rank)

    # End to end through the same public calls from pinned host buffers, as a
    # caller would pipeline it: step i's Q/K/V copy in on one stream while
    # step i-1 computes, and step i-1's output copies out on a third stream;
    # every step's copies lie inside the timed region (first copy-in of the
    # first timed step to the last copy-out).
    e2e = None
    if args.e2e_steps > 0:
        hq = [b.pin_memory() for b in (x.cpu() for x in qb)]
        hk = [b.pin_memory() for b in (x.cpu() for x in kb)]
        hv = [b.pin_memory() for b in (x.cpu() for x in vb)]
        ho = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for _ in range(2)]
        dq = [torch.empty_like(q) for _ in range(2)]
        dk = [torch.empty_like(kb[0]) for _ in range(2)]
        dv = [torch.empty_like(vb[0]) for _ in range(2)]
        do = [torch.empty_like(q) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        n = args.warmup + args.e2e_steps
        ev_in, ev_c, ev_out = [ev() for _ in range(n)], [ev() for _ in range(n)], [ev() for _ in range(n)]
        t_start = ev()
        for i in range(n):
            b = i % 2
            if i == args.warmup:
                torch.cuda.synchronize()
                t_start.record(s_in)
            if i >= 2:
                s_in.wait_event(ev_c[i - 2])          # buffers b free again
            with torch.cuda.stream(s_in):
                dq[b].copy_(hq[i % 2], non_blocking=True)
                dk[b].copy_(hk[i % 2], non_blocking=True)
                dv[b].copy_(hv[i % 2], non_blocking=True)
            ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])      # do[b] copied out
            cache.append(block_id(), dk[b], dv[b], stream=stream)
            cache.routed_attention(dq[b], do[b], stream=stream)
            ev_c[i].record(stream)
            s_out.wait_event(ev_c[i])
            with torch.cuda.stream(s_out):
                ho[b].copy_(do[b], non_blocking=True)
            ev_out[i].record(s_out)
            state["step"] += 1
        torch.cuda.synchronize()
        e2e_ms = t_start.elapsed_time(ev_out[n - 1]) / args.e2e_steps
        nb = q.numel() * q.element_size()
        e2e = {"value": world * shape.n_q / (1e-3 * e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": 3 * nb, "d2h_bytes_per_step": nb, "ms_per_step": e2e_ms,
               "pipelining": "copy-in, compute and copy-out of consecutive steps on three streams"}

    if rank != 0:
        return
    flops = routed_flops(shape, labels)
    mean_routed = statistics.mean(routed_ms)
    achieved = flops / (mean_routed * 1e-3) / 1e12
    tb = traffic_from_profile(f"routed_attention_{shape.name}")
    value = job_value(shape.n_q, args.steps, total_ms, world)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V with planted archetypes; pages' 720P shapes)",
        "config": workload_config(shape),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": tb,
                     "kernel": "routed attention (one launch, all heads)",
                     "algorithmic_flops_per_launch": flops,
                     "algorithmic_bytes_per_launch": routed_bytes(shape, labels),
                     "peak_source": f"{peak_kind} bf16 dense (burst)"},
        "e2e": e2e,
        "gpu_launches": args.steps * (2 + (1 if cache.info()["split_bytes"] else 0)),
        "clocks": clocks,
        "routed_attention_ms": mean_routed,
        "append_ms": statistics.mean(s - r for s, r in zip(step_ms, routed_ms)),
        "full_attention_ms": statistics.mean(full_ms),
        "monolithic_append_ms": statistics.mean(mono_ms),
        "speedup_vs_full_attention": statistics.mean(full_ms) / mean_routed,
        "step_speedup_vs_full": (statistics.mean(full_ms) + statistics.mean(mono_ms)) /
                                (total_ms / args.steps),
        "classify_ms": classify_ms, "restructure_ms": restructure_ms,
        "cache_kernels": cache_kernel_rates(shape, labels, restructure_ms,
                                            statistics.mean(s - r for s, r in zip(step_ms, routed_ms)),
                                            peak_bw),
        "paths": paths,
        "workloads": workloads,
        "pages_context": {"end_to_end_generation_speedup_vs_full_attention": {"720P": 1.62, "1080P": 1.95},
                          "hardware": "not stated on the pages",
                          "note": "whole-model FPS ratios (LongLive, 30 s clips), not this metric"},
        "memory": hc.memory_report(cfg, labels),
        "wall_s_timed": wall,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(shape, inp, labels, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    shape = synth.SHAPES[args.workload if args.workload in synth.SHAPES else "720p"]
    if args.impl == "reference":
        run_reference(args, shape, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if args.workload == "rollout":
        run_rollout(args, rank, world, local_rank)
    elif args.workload == "sweep":
        run_sweep(args, rank, world, local_rank)
    elif args.workload == "agreement":
        run_agreement(args, rank, world, local_rank)
    elif args.workload == "stability":
        run_stability(args, rank, world, local_rank)
    else:
        run_ours(args, shape, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
