"""Plain fp64 CPU oracle for HeadCast's head-routed attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, links or runs this
module: only the test-suite, the package entry point's smoke check and the
benchmark's CPU-baseline/reference arm may call it.  It shares no code with
the CUDA path (no kernels, helpers, tables or constants), and it is written
to be read against the pages, not to be fast.

Source pages (cited by title and section):
  [HC-abs]   "HeadCast: Casting Attention Heads for Efficient Autoregressive
             Video Generation", abstract (arXiv 2607.20125 record).
  [HC-pith]  Pith review of the same paper: "The pith", "Core claim",
             "What carries the argument", "Referee Report" (major comments),
             "Axiom & Free-Parameter Ledger", Figure 2 and Figure 3 captions.

What the method computes (restated, not quoted):
  * Every attention head is typed once, when the sliding window first fills,
    at the maximum-noise step, by comparing its full-context attention output
    with the outputs of three restricted contexts: the first block only
    (Sink), the current block only (Dummy) and a (2r+1)x(2r+1) neighbourhood
    across history with r = 2 (Spatial).  The first archetype whose cosine
    similarity clears theta = 0.95 wins, with a conservative
    5th-percentile-plus-MSE score (gamma = 5, threshold 0.755) gating
    Spatial; a head that passes none is Global.
    [HC-pith "What carries the argument"; Ledger: theta, theta_sc, gamma, r]
  * After typing, each head attends only over its pathway: Sink -> the first
    block, Dummy -> the newest block, Spatial -> its own cell of a
    non-overlapping 10x10 partition of every cached frame ("with rounded
    remainder"), Global -> the whole sliding window.
    [HC-pith "The pith", "Core claim", major comment 2, Ledger "deployed
    spatial grid cell", Figure 3 caption; HC-abs]

Readings of points the pages leave open (each is listed with its reason in
the design notes and used identically by the CUDA library):
  o1  the archetype similarity of a head is the mean over the block's query
      tokens of the per-token cosine between output vectors;
  o2  score = P5(cos_spatial) - gamma * MSE(O_spatial, O_full), MSE averaged
      over tokens and head-dim channels ("plus MSE" read as an MSE penalty);
  o3  Spatial needs both c_spatial >= theta and score >= theta_sc;
  o4  P5 is the linearly interpolated 5th percentile at rank 0.05*(n-1);
  o5  "clears" means >=, tested in the order Sink, Dummy, Spatial;
  o6  the window includes the current block;
  o7  Sink means block 0 of the stream, kept forever;
  o8  Sink sees only block 0 and Dummy only the current block;
  o9  cells per axis n = max(1, floor(N/10 + 1/2)); the first n-1 cells are
      10 wide and the last takes the remainder;
  o10 the proxy covers every window frame;
  o11 softmax scale 1/sqrt(d), no bias, inputs are post-RoPE;
  o12 cosine of two zero vectors is 1, of one zero vector 0;
  o15 a repeated block id overwrites the newest block; id+1 advances the
      window and evicts its oldest block.

Parity unpinned: o1-o4 (how per-token cosines become a head's similarity, the
composition of the score, the percentile definition) have no worked example
on the pages, so no printed value pins them.  The arithmetic of each reading
is pinned (tests/test_oracle.py: decision-rule boundaries, percentile and
cosine/MSE closed forms); the readings themselves are not.
"""
from __future__ import annotations

from dataclasses import dataclass
import math
import numpy as np

SINK, DUMMY, SPATIAL, GLOBAL = 0, 1, 2, 3


@dataclass(frozen=True)
class Geometry:
    """Token grid of one layer.  A block is ``frames_per_block`` frames; the
    window holds ``window_frames`` frames including the current block."""
    n_heads: int
    head_dim: int
    frame_h: int
    frame_w: int
    window_frames: int
    frames_per_block: int = 3
    proxy_radius: int = 2          # r  [HC-pith Ledger "Spatial proxy radius r = 2"]
    cell_h: int = 10               # [HC-pith Ledger "deployed spatial grid cell = 10x10"]
    cell_w: int = 10
    # Key set of the classifier's Spatial proxy: "neighbourhood" (the
    # paper's (2r+1)x(2r+1) window) or "cell" (the deployed cell, to measure
    # how well the proxy stands for the deployed path) [HC-pith major comment 2].
    proxy_mode: str = "neighbourhood"
    # Deployed Spatial key set: "cells" (the query's own non-overlapping
    # cell, the reading of the pages' "non-overlapping 10x10 cells") or
    # "sliding" (the cell_h x cell_w window centred on the query, rows
    # h - cell_h//2 .. h + cell_h - cell_h//2 - 1 and likewise for columns,
    # clipped; the "10x10 grid around the query's position" wording).
    spatial_mode: str = "cells"

    @property
    def F(self):
        return self.frame_h * self.frame_w

    @property
    def block_tokens(self):
        return self.frames_per_block * self.F

    @property
    def n_k(self):
        return self.window_frames * self.F

    @property
    def blocks_per_window(self):
        return self.window_frames // self.frames_per_block


@dataclass(frozen=True)
class Thresholds:
    """[HC-pith Ledger]: theta_s = theta_d = theta_sp = 0.95, theta_sc = 0.755,
    gamma = 5."""
    theta_sink: float = 0.95
    theta_dummy: float = 0.95
    theta_spatial: float = 0.95
    theta_score: float = 0.755
    gamma: float = 5.0


def geometry_of(shape, **kw) -> Geometry:
    """Build a Geometry from any object with the synthetic-layer fields."""
    return Geometry(shape.n_heads, shape.head_dim, shape.frame_h, shape.frame_w,
                    shape.window_frames, shape.frames_per_block, **kw)


# --------------------------------------------------------------------------
# Attention on an explicit key set.

def softmax_attention(q, k, v, scale):
    """o = softmax(q k^T * scale) v for one head, in fp64.

    q [m][d], k [n][d], v [n][d] -> [m][d].  Rows are normalised after
    subtracting their maximum, the textbook stable form."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = (q @ k.T) * scale
    s -= s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


def attend_chunked(q, k, v, scale, chunk=256):
    """softmax_attention over all n keys, in query chunks to bound memory."""
    out = np.empty((q.shape[0], v.shape[1]), dtype=np.float64)
    for i in range(0, q.shape[0], chunk):
        out[i:i + chunk] = softmax_attention(q[i:i + chunk], k, v, scale)
    return out


def default_scale(d):
    return 1.0 / math.sqrt(d)                      # o11


# --------------------------------------------------------------------------
# Key sets.  Token index inside a run of frames: t = f*F + h*W + w.

def token_position(t, geom: Geometry):
    """(frame, row, col) of token t counted from the first frame of a run."""
    f, rem = divmod(t, geom.F)
    return f, rem // geom.frame_w, rem % geom.frame_w


def proxy_keys(h, w, n_frames, geom: Geometry):
    """Spatial proxy: every frame's (2r+1)x(2r+1) neighbourhood of (h, w),
    clipped at the frame edge, across all window frames (o10).
    [HC-pith "What carries the argument" ("only a local neighborhood"),
    major comment 2 ("sliding (2r+1)x(2r+1) neighborhood with r=2")]"""
    r = geom.proxy_radius
    hs = range(max(0, h - r), min(geom.frame_h - 1, h + r) + 1)
    ws = range(max(0, w - r), min(geom.frame_w - 1, w + r) + 1)
    return np.array([f * geom.F + hh * geom.frame_w + ww
                     for f in range(n_frames) for hh in hs for ww in ws], dtype=np.int64)


def cell_partition(n, cell):
    """Cells along one axis of length n (o9): [(start, size), ...].

    n_cells = max(1, floor(n/cell + 1/2)); all but the last are ``cell`` wide,
    the last takes what remains.  [HC-pith Ledger "10x10 with rounded
    remainder"; major comment 2 "non-overlapping 10x10 cells"]"""
    n_cells = max(1, int(math.floor(n / cell + 0.5)))
    cells = [(i * cell, cell) for i in range(n_cells - 1)]
    start = (n_cells - 1) * cell
    cells.append((start, n - start))
    return cells


def cell_of(x, cells):
    for i, (s, z) in enumerate(cells):
        if s <= x < s + z:
            return i
    raise ValueError(x)


def cell_keys(h, w, n_frames, geom: Geometry):
    """Deployed Spatial path: the keys of (h, w)'s own cell in every window
    frame.  [HC-pith Figure 3 caption, major comment 2, "Core claim"
    ("fixed 10x10 grid across history")]"""
    ch = cell_partition(geom.frame_h, geom.cell_h)
    cw = cell_partition(geom.frame_w, geom.cell_w)
    h0, hz = ch[cell_of(h, ch)]
    w0, wz = cw[cell_of(w, cw)]
    return np.array([f * geom.F + hh * geom.frame_w + ww
                     for f in range(n_frames)
                     for hh in range(h0, h0 + hz) for ww in range(w0, w0 + wz)], dtype=np.int64)


def sliding_keys(h, w, n_frames, geom: Geometry):
    """Deployed Spatial path, sliding variant: the cell_h x cell_w window
    whose rows are h - cell_h//2 .. h + cell_h - cell_h//2 - 1 (columns
    likewise), clipped to the frame, in every window frame."""
    h0, w0 = h - geom.cell_h // 2, w - geom.cell_w // 2
    hs = range(max(0, h0), min(geom.frame_h, h0 + geom.cell_h))
    ws = range(max(0, w0), min(geom.frame_w, w0 + geom.cell_w))
    return np.array([f * geom.F + hh * geom.frame_w + ww
                     for f in range(n_frames) for hh in hs for ww in ws], dtype=np.int64)


def attend_by_position(q_h, k_h, v_h, geom: Geometry, n_frames, keyset, scale, query_idx):
    """Attention where each query's key set depends only on its (row, col).

    q_h [nq][d] holds the current block's queries (block-local token order);
    queries sharing a position share one key set and are done together."""
    out = np.empty((len(query_idx), v_h.shape[1]), dtype=np.float64)
    groups = {}
    for n, i in enumerate(query_idx):
        _, h, w = token_position(int(i), geom)
        groups.setdefault((h, w), []).append(n)
    for (h, w), rows in groups.items():
        keys = keyset(h, w, n_frames, geom)
        out[rows] = softmax_attention(q_h[query_idx[rows]], k_h[keys], v_h[keys], scale)
    return out


# --------------------------------------------------------------------------
# Classification.  [HC-pith "What carries the argument"; Ledger]

def cosine_rows(a, b):
    """Per-row cosine similarity, with the o12 convention for zero rows."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    na = np.sqrt((a * a).sum(axis=1))
    nb = np.sqrt((b * b).sum(axis=1))
    dot = (a * b).sum(axis=1)
    out = np.empty(a.shape[0])
    for i in range(a.shape[0]):
        if na[i] == 0.0 and nb[i] == 0.0:
            out[i] = 1.0
        elif na[i] == 0.0 or nb[i] == 0.0:
            out[i] = 0.0
        else:
            out[i] = dot[i] / (na[i] * nb[i])
    return out


def percentile_linear(x, pct):
    """pct-th percentile with linear interpolation between order statistics
    at rank pct/100*(n-1) (o4)."""
    v = np.sort(np.asarray(x, dtype=np.float64))
    pos = pct / 100.0 * (len(v) - 1)
    lo = int(math.floor(pos))
    hi = min(lo + 1, len(v) - 1)
    return v[lo] + (pos - lo) * (v[hi] - v[lo])


def head_statistics(cos_sink, cos_dummy, cos_spatial, o_spatial, o_full, gamma):
    """(c_s, c_d, c_sp, P5, MSE, score) of one head (o1, o2)."""
    c_s = float(np.mean(cos_sink))
    c_d = float(np.mean(cos_dummy))
    c_sp = float(np.mean(cos_spatial))
    p5 = float(percentile_linear(cos_spatial, 5.0))
    diff = np.asarray(o_spatial, np.float64) - np.asarray(o_full, np.float64)
    mse = float(np.mean(diff * diff))
    return c_s, c_d, c_sp, p5, mse, p5 - gamma * mse


def decide(stats, th: Thresholds = Thresholds()):
    """First archetype whose similarity clears its threshold, in the order
    Sink, Dummy, Spatial (the last also needs score >= theta_sc); else
    Global.  (o3, o5)"""
    c_s, c_d, c_sp, _p5, _mse, score = stats
    if c_s >= th.theta_sink:
        return SINK
    if c_d >= th.theta_dummy:
        return DUMMY
    if c_sp >= th.theta_spatial and score >= th.theta_score:
        return SPATIAL
    return GLOBAL


def margins(stats, th: Thresholds = Thresholds()):
    """Signed distance of every gate from its threshold (positive = passes)."""
    c_s, c_d, c_sp, _p5, _mse, score = stats
    return (c_s - th.theta_sink, c_d - th.theta_dummy,
            c_sp - th.theta_spatial, score - th.theta_score)


@dataclass
class HeadProxies:
    o_full: np.ndarray
    o_sink: np.ndarray
    o_dummy: np.ndarray
    o_spatial: np.ndarray


def classification_outputs(q, k, v, geom: Geometry, head, scale=None, query_idx=None):
    """The four attention outputs of one head at classification time.

    q [n_q][H][d]: the current block's queries; k, v [n_k][H][d]: the window,
    oldest frame first, which has just filled, so its first block is block 0
    of the stream and its last block is the current one."""
    scale = default_scale(geom.head_dim) if scale is None else scale
    n_frames = k.shape[0] // geom.F
    blk = geom.block_tokens
    qi = np.arange(q.shape[0]) if query_idx is None else np.asarray(query_idx)
    qh = np.asarray(q[:, head, :], np.float64)
    kh = np.asarray(k[:, head, :], np.float64)
    vh = np.asarray(v[:, head, :], np.float64)
    nk = kh.shape[0]
    o_full = attend_chunked(qh[qi], kh, vh, scale)
    o_sink = attend_chunked(qh[qi], kh[:blk], vh[:blk], scale)
    o_dummy = attend_chunked(qh[qi], kh[nk - blk:], vh[nk - blk:], scale)
    keyset = cell_keys if geom.proxy_mode == "cell" else proxy_keys
    o_sp = attend_by_position(qh, kh, vh, geom, n_frames, keyset, scale, qi)
    return HeadProxies(o_full, o_sink, o_dummy, o_sp)


@dataclass
class Classification:
    labels: np.ndarray        # int8 [H]
    stats: np.ndarray         # [H][6]: c_s, c_d, c_sp, P5, MSE, score
    margins: np.ndarray       # [H][4]
    outputs: list             # HeadProxies per head


def classify(q, k, v, geom: Geometry, th: Thresholds = Thresholds(), scale=None):
    """One-time head classification over the current block's queries."""
    H = geom.n_heads
    stats = np.zeros((H, 6))
    outs = []
    for h in range(H):
        o = classification_outputs(q, k, v, geom, h, scale)
        st = head_statistics(cosine_rows(o.o_full, o.o_sink), cosine_rows(o.o_full, o.o_dummy),
                             cosine_rows(o.o_full, o.o_spatial), o.o_spatial, o.o_full, th.gamma)
        stats[h] = st
        outs.append(o)
    labels = np.array([decide(s, th) for s in stats], dtype=np.int8)
    return Classification(labels, stats, np.array([margins(s, th) for s in stats]), outs)


# --------------------------------------------------------------------------
# The sliding-window cache and routed attention.

class CacheModel:
    """Per-block model of the window (o6, o7, o15).

    Blocks are kept by id; the window is the newest ``blocks_per_window``
    blocks, and block 0 is kept forever as the Sink block."""

    def __init__(self, geom: Geometry):
        self.geom = geom
        self.blocks = {}
        self.newest = None

    def put(self, block_id, k_blk, v_blk):
        if self.newest is not None and block_id not in (self.newest, self.newest + 1):
            raise ValueError("block id must repeat the newest block or follow it")
        self.blocks[block_id] = (np.array(k_blk, np.float64), np.array(v_blk, np.float64))
        self.newest = block_id if self.newest is None else max(self.newest, block_id)
        oldest = self.newest - self.geom.blocks_per_window + 1
        for b in [b for b in self.blocks if b < oldest and b != 0]:
            del self.blocks[b]

    def window_ids(self):
        lo = max(0, self.newest - self.geom.blocks_per_window + 1)
        return list(range(lo, self.newest + 1))

    def window(self):
        ids = self.window_ids()
        k = np.concatenate([self.blocks[b][0] for b in ids], axis=0)
        v = np.concatenate([self.blocks[b][1] for b in ids], axis=0)
        return k, v

    def sink(self):
        return self.blocks[0]

    def current(self):
        return self.blocks[self.newest]


def routed_head(q, cache: CacheModel, label, head, scale=None, query_idx=None):
    """One head's output over its own pathway.  [HC-pith "The pith",
    "Core claim", Figure 3 caption; HC-abs]"""
    geom = cache.geom
    scale = default_scale(geom.head_dim) if scale is None else scale
    qi = np.arange(q.shape[0]) if query_idx is None else np.asarray(query_idx)
    qh = np.asarray(q[:, head, :], np.float64)
    if label == SINK:
        k, v = cache.sink()
    elif label == DUMMY:
        k, v = cache.current()
    else:
        k, v = cache.window()
    kh, vh = k[:, head, :], v[:, head, :]
    if label == SPATIAL:
        n_frames = kh.shape[0] // geom.F
        keyset = sliding_keys if geom.spatial_mode == "sliding" else cell_keys
        return attend_by_position(qh, kh, vh, geom, n_frames, keyset, scale, qi)
    return attend_chunked(qh[qi], kh, vh, scale)


def routed_attention(q, cache: CacheModel, labels, scale=None, query_idx=None):
    """All heads, each over its pathway: [n_sel][H][d]."""
    geom = cache.geom
    qi = np.arange(q.shape[0]) if query_idx is None else np.asarray(query_idx)
    out = np.empty((len(qi), geom.n_heads, geom.head_dim))
    for h in range(geom.n_heads):
        out[:, h, :] = routed_head(q, cache, int(labels[h]), h, scale, qi)
    return out


def full_attention(q, k, v, scale=None, query_idx=None):
    """Every head over every key: the comparison path.  [HC-pith "If this is
    right" (speedups are against full attention)]"""
    d = q.shape[2]
    scale = default_scale(d) if scale is None else scale
    qi = np.arange(q.shape[0]) if query_idx is None else np.asarray(query_idx)
    out = np.empty((len(qi), q.shape[1], d))
    for h in range(q.shape[1]):
        out[:, h, :] = attend_chunked(np.asarray(q[qi, h, :], np.float64),
                                      np.asarray(k[:, h, :], np.float64),
                                      np.asarray(v[:, h, :], np.float64), scale)
    return out
