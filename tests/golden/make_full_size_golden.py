"""Write the oracle's classification of the full-size layers to tests/golden/.

    python tests/golden/make_full_size_golden.py [--workers N] [--only NAME ...]

Calls only the fp64 CPU oracle (``oracle.headcast_ref.classify``) on the
seeded synthetic inputs of ``synth``; nothing here touches the CUDA library.
Heads are independent in the method (each head's outputs, statistics and
label depend only on that head's Q, K and V), so every head is classified
on its own, as a one-head layer, in a pool of worker processes; the result
is the same call the oracle makes for the whole layer.

Files (JSON, one per workload):
  classify_720p.json     the planted 720P layer (seed 2)
  classify_1080p.json    the planted 1080P layer (seed 3)
  classify_rollout.json  the 30 layers of the 720P rollout (seed 4*100 + layer,
                         archetypes drawn per (layer, head) from seed 4)
  classify_stream.json   480P re-classification windows of a drifting stream
                         (seed 501): block 0 plus the six newest blocks, at
                         blocks 7 and 12, drift 0.3 and 0.6
Each entry records the labels, the six per-head statistics (c_sink, c_dummy,
c_spatial, P5, MSE, score), the margins of the four gates, and a SHA-256 of
the raw input bytes so that a test can tell whether the inputs it
regenerates are the ones classified here.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import multiprocessing as mp
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import headcast_ref as ref  # noqa: E402

STREAM = dict(shape="480p", seed=501, drifts=(0.3, 0.6), blocks=(7, 12))


def _init_worker():
    from threadpoolctl import threadpool_limits
    threadpool_limits(1)


def _classify_head(geom_kw, q, k, v):
    """The oracle's classify on one head (q [nq][1][d], k/v [nk][1][d])."""
    geom = ref.Geometry(**geom_kw)
    cls = ref.classify(q, k, v, geom)
    return int(cls.labels[0]), [float(x) for x in cls.stats[0]], [float(x) for x in cls.margins[0]]


def input_digest(q_raw, k_raw, v_raw):
    return {n: hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()
            for n, a in (("q", q_raw), ("k", k_raw), ("v", v_raw))}


def _submit_layer(ex, shape, q, k, v):
    """q [nq][H][d], k/v [nk][H][d] values -> futures, one per head."""
    geom_kw = dict(n_heads=1, head_dim=shape.head_dim, frame_h=shape.frame_h, frame_w=shape.frame_w,
                   window_frames=k.shape[0] // shape.frame_tokens,
                   frames_per_block=shape.frames_per_block)
    return [ex.submit(_classify_head, geom_kw, np.ascontiguousarray(q[:, h:h + 1]),
                      np.ascontiguousarray(k[:, h:h + 1]), np.ascontiguousarray(v[:, h:h + 1]))
            for h in range(shape.n_heads)]


def _collect(futs):
    res = [f.result() for f in futs]
    return dict(labels=[r[0] for r in res], stats=[r[1] for r in res], margins=[r[2] for r in res])


def _header(extra):
    h = {"_generated_by": "tests/golden/make_full_size_golden.py (fp64 oracle only)",
         "_oracle": "oracle.headcast_ref.classify, one head at a time",
         "_stats": ["c_sink", "c_dummy", "c_spatial", "p5", "mse", "score"],
         "_margins": ["c_sink - theta_sink", "c_dummy - theta_dummy", "c_spatial - theta_spatial",
                      "score - theta_score"],
         "thresholds": dict(theta=0.95, theta_score=0.755, gamma=5.0, proxy_radius=2)}
    h.update(extra)
    return h


def _write(name, obj):
    path = os.path.join(HERE, name)
    with open(path + ".tmp", "w") as f:
        json.dump(obj, f, indent=1)
    os.replace(path + ".tmp", path)
    print("wrote", path, flush=True)


def planted(ex, name):
    shape = synth.SHAPES[name]
    t = time.time()
    inp = synth.make_layer(shape)
    futs = _submit_layer(ex, shape, inp.q.values, inp.k.values, inp.v.values)
    digest = input_digest(inp.q.raw, inp.k.raw, inp.v.raw)
    del inp
    out = _header({"workload": f"{name} layer", "seed": shape.seed, "mix": list(shape.mix),
                   "inputs_sha256": digest})
    out.update(_collect(futs))
    out["_seconds"] = round(time.time() - t, 1)
    _write(f"classify_{name}.json", out)


def rollout(ex, layers=None):
    R = synth.ROLLOUT_720P
    shape = R["shape"]
    mix = synth.rollout_mix(R["layers"], shape.n_heads, R["seed"])
    layers = range(R["layers"]) if layers is None else layers
    t = time.time()
    pending = []
    for layer in layers:
        m = tuple(int(a) for a in mix[layer])
        inp = synth.make_layer(shape, seed=R["seed"] * 100 + layer, mix=m)
        pending.append((layer, m, input_digest(inp.q.raw, inp.k.raw, inp.v.raw),
                        _submit_layer(ex, shape, inp.q.values, inp.k.values, inp.v.values)))
        del inp
        # Keep at most two unfinished layers queued ahead of the workers (memory).
        while sum(1 for p in pending if not all(f.done() for f in p[3])) > 2:
            time.sleep(0.5)
    entries = []
    for layer, m, digest, futs in pending:
        e = {"layer": layer, "seed": R["seed"] * 100 + layer, "mix": list(m), "inputs_sha256": digest}
        e.update(_collect(futs))
        entries.append(e)
        print(f"rollout layer {layer}: labels {e['labels']} mix {list(m)}", flush=True)
    out = _header({"workload": "720p rollout", "layers": entries, "_seconds": round(time.time() - t, 1)})
    _write("classify_rollout.json", out)


def stream_windows(shape, blocks, b):
    """K/V of the window classified at block b: block 0 (the Sink block) and
    the blocks_per_window - 1 newest blocks up to b."""
    ids = [0] + list(range(b - shape.blocks_per_window + 2, b + 1))
    k = np.concatenate([blocks[i][1].values for i in ids])
    v = np.concatenate([blocks[i][2].values for i in ids])
    kr = np.concatenate([blocks[i][1].raw for i in ids])
    vr = np.concatenate([blocks[i][2].raw for i in ids])
    return ids, k, v, kr, vr


def stream(ex):
    shape = synth.SHAPES[STREAM["shape"]]
    t = time.time()
    entries = []
    for drift in STREAM["drifts"]:
        blocks = synth.make_stream(shape, seed=STREAM["seed"], n_blocks=max(STREAM["blocks"]) + 1, drift=drift)
        for b in STREAM["blocks"]:
            ids, k, v, kr, vr = stream_windows(shape, blocks, b)
            futs = _submit_layer(ex, shape, blocks[b][0].values, k, v)
            e = {"drift": drift, "block": b, "window_blocks": ids,
                 "inputs_sha256": input_digest(blocks[b][0].raw, kr, vr)}
            e.update(_collect(futs))
            entries.append(e)
            print(f"stream drift {drift} block {b}: labels {e['labels']}", flush=True)
    out = _header({"workload": "480p drifting stream", "seed": STREAM["seed"], "mix": list(shape.mix),
                   "entries": entries, "_seconds": round(time.time() - t, 1)})
    _write("classify_stream.json", out)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workers", type=int, default=os.cpu_count() or 1)
    ap.add_argument("--only", nargs="*", default=["stream", "720p", "1080p", "rollout"])
    a = ap.parse_args()
    ctx = mp.get_context("spawn")
    with cf.ProcessPoolExecutor(max_workers=a.workers, mp_context=ctx, initializer=_init_worker) as ex:
        for name in a.only:
            if name in ("720p", "1080p"):
                planted(ex, name)
            elif name == "rollout":
                rollout(ex)
            elif name == "stream":
                stream(ex)
            else:
                raise SystemExit(f"unknown workload {name}")


if __name__ == "__main__":
    main()
