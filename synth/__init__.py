"""Seeded synthetic inputs for head-routed attention over a video DiT KV cache.

This module holds shapes and random draws only.  None of the attention,
classification or cache arithmetic lives here: both the fp64 CPU oracle and
the CUDA library consume the arrays it returns, so a shared mistake here can
only change the inputs, never the method.

Workloads (the HeadCast pages measure real Wan-family latents at 480P, 720P
and 1080P with a 21-frame sliding window of 3-frame blocks; the trained
backbones are not available, so these synthetic layers stand in for them
with the same token grids, window and head geometry):

  tiny   4 heads,  d=64,  fp32,  8x8 grid,   12-frame window
  480p  12 heads, d=128,  bf16, 30x52 grid,  21-frame window
  720p  12 heads, d=128,  bf16, 45x80 grid,  21-frame window
  1080p 12 heads, d=128,  bf16, 68x120 grid, 21-frame window

Values: Q, K, V ~ N(0, 1) from ``numpy.random.default_rng(seed)``, then a
planted per-head structure (below), then rounding to the storage dtype.

Planting (so that a classifier has something to find):
  * Sink head: every current-block query gets ``c*u`` added (u a seeded unit
    vector, c**2 = 3*sqrt(d)); then the keys of the stream's first block get
    ``4*q_mean`` added, q_mean the mean of that head's current-block queries.
    The logit boost on those keys is about 4*c**2/sqrt(d) = 12 nats.
  * Dummy head: the same, on the keys of the current (newest) block.
  * Spatial head: a random-Fourier-feature map s(h, w) in R^d
    (s = sqrt(2/d) cos(Omega @ (h, w) + phi), Omega ~ N(0, I), phi ~ U[0, 2pi))
    whose inner products approximate exp(-|x - y|^2 / 2); queries get
    ``4*a*s(h, w)`` and keys at every cached frame get ``a*s(h, w)``,
    a**2 = 3*sqrt(d), so a key at the query's own position gains ~12 nats.
    (The factor 4 sits on the query side so that the query's own noise,
    projected on the key plant, stays near 0.5 nats: on the key side it is
    about 2 nats and lets a far position win for a few queries.)
  * Global head: unplanted.
"""
from __future__ import annotations

from dataclasses import dataclass, field
import numpy as np

SINK, DUMMY, SPATIAL, GLOBAL = 0, 1, 2, 3
ARCHETYPE_NAMES = ("sink", "dummy", "spatial", "global")

# Head -> archetype assignment used for the 12-head layers: 2 Sink, 3 Dummy,
# 4 Spatial, 3 Global.
MIX_12 = (SINK, SINK, DUMMY, DUMMY, DUMMY, SPATIAL, SPATIAL, SPATIAL, SPATIAL,
          GLOBAL, GLOBAL, GLOBAL)
MIX_4 = (SINK, DUMMY, SPATIAL, GLOBAL)


@dataclass(frozen=True)
class LayerShape:
    name: str
    n_heads: int
    head_dim: int
    frame_h: int
    frame_w: int
    window_frames: int
    dtype: str            # "bf16" or "fp32"
    seed: int
    mix: tuple = field(default=())
    frames_per_block: int = 3

    @property
    def frame_tokens(self) -> int:
        return self.frame_h * self.frame_w

    @property
    def n_q(self) -> int:
        return self.frames_per_block * self.frame_tokens

    @property
    def n_k(self) -> int:
        return self.window_frames * self.frame_tokens

    @property
    def blocks_per_window(self) -> int:
        return self.window_frames // self.frames_per_block


SHAPES = {
    "tiny": LayerShape("tiny", 4, 64, 8, 8, 12, "fp32", 0, MIX_4),
    "480p": LayerShape("480p", 12, 128, 30, 52, 21, "bf16", 1, MIX_12),
    "720p": LayerShape("720p", 12, 128, 45, 80, 21, "bf16", 2, MIX_12),
    "1080p": LayerShape("1080p", 12, 128, 68, 120, 21, "bf16", 3, MIX_12),
}

# The 30-layer 720P rollout: per-(layer, head) archetype uniform over the four.
ROLLOUT_720P = dict(layers=30, shape=SHAPES["720p"], seed=4, blocks=7, steps=4)


def custom_shape(name="custom", n_heads=4, head_dim=64, frame_h=8, frame_w=8,
                 window_frames=12, dtype="bf16", seed=0, mix=None) -> LayerShape:
    if mix is None:
        mix = tuple(MIX_4[h % 4] for h in range(n_heads))
    return LayerShape(name, n_heads, head_dim, frame_h, frame_w, window_frames,
                      dtype, seed, tuple(mix))


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (inputs are finite)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((b >> 16) & 1) + np.uint32(0x7FFF)
    return ((b + r) >> 16).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


@dataclass
class Tensor3:
    """A [tokens][heads][d] array in its storage dtype plus its exact values."""
    values: np.ndarray      # float32, exactly representable in the storage dtype
    raw: np.ndarray         # uint16 bit patterns (bf16) or float32 (fp32)


def _store(x: np.ndarray, dtype: str) -> Tensor3:
    if dtype == "bf16":
        bits = bf16_bits(x)
        return Tensor3(bf16_to_f32(bits), bits)
    if dtype == "fp32":
        x = np.ascontiguousarray(x, dtype=np.float32)
        return Tensor3(x, x)
    raise ValueError(dtype)


def random_unit(rng, d):
    u = rng.standard_normal(d)
    return u / np.linalg.norm(u)


def spatial_features(rng, frame_h, frame_w, d):
    """Random Fourier features s(h, w) of an RBF kernel with unit length scale."""
    omega = rng.standard_normal((d, 2))
    phi = rng.uniform(0.0, 2.0 * np.pi, size=d)
    hh, ww = np.meshgrid(np.arange(frame_h), np.arange(frame_w), indexing="ij")
    pos = np.stack([hh.ravel(), ww.ravel()], axis=1).astype(np.float64)   # [F][2]
    return np.sqrt(2.0 / d) * np.cos(pos @ omega.T + phi)                 # [F][d]


@dataclass
class LayerInputs:
    shape: LayerShape
    q: Tensor3              # [n_q][H][d]   current block's queries
    k: Tensor3              # [n_k][H][d]   window keys, oldest frame first
    v: Tensor3              # [n_k][H][d]
    planted: tuple          # archetype per head


def make_layer(shape: LayerShape, seed: int | None = None, mix=None) -> LayerInputs:
    """One layer's classification-time inputs: the window has just filled, so
    it holds blocks 0..B-1 of the stream and the current block is its last."""
    seed = shape.seed if seed is None else seed
    mix = tuple(shape.mix if mix is None else mix)
    assert len(mix) == shape.n_heads
    rng = np.random.default_rng(seed)
    H, d, F = shape.n_heads, shape.head_dim, shape.frame_tokens
    nq, nk, fpb = shape.n_q, shape.n_k, shape.frames_per_block
    q = rng.standard_normal((nq, H, d), dtype=np.float32)
    k = rng.standard_normal((nk, H, d), dtype=np.float32)
    v = rng.standard_normal((nk, H, d), dtype=np.float32)
    c = np.sqrt(3.0 * np.sqrt(d))
    blk = fpb * F
    for h, arch in enumerate(mix):
        if arch in (SINK, DUMMY):
            u = random_unit(rng, d)
            q[:, h, :] += (c * u).astype(np.float32)
            q_mean = q[:, h, :].astype(np.float64).mean(axis=0)
            rows = slice(0, blk) if arch == SINK else slice(nk - blk, nk)
            k[rows, h, :] += (4.0 * q_mean).astype(np.float32)
        elif arch == SPATIAL:
            s = spatial_features(rng, shape.frame_h, shape.frame_w, d)   # [F][d]
            a = c
            q[:, h, :] += np.tile(4.0 * a * s, (fpb, 1)).astype(np.float32)
            k[:, h, :] += np.tile(a * s, (shape.window_frames, 1)).astype(np.float32)
    return LayerInputs(shape, _store(q, shape.dtype), _store(k, shape.dtype),
                       _store(v, shape.dtype), mix)


def make_block(shape: LayerShape, seed: int, mix=None):
    """Fresh Q, K, V for one 3-frame block (a steady-state denoising step).

    All values are fresh N(0, 1) draws from ``seed``; Spatial heads also get a
    positional plant (a feature map drawn from the same generator, queries
    4*c*s and keys c*s).  Sink and Dummy heads get no plant here (streams
    whose plants persist across blocks come from ``make_stream``)."""
    mix = tuple(shape.mix if mix is None else mix)
    rng = np.random.default_rng(seed)
    H, d, F = shape.n_heads, shape.head_dim, shape.frame_tokens
    nq = shape.n_q
    q = rng.standard_normal((nq, H, d), dtype=np.float32)
    k = rng.standard_normal((nq, H, d), dtype=np.float32)
    v = rng.standard_normal((nq, H, d), dtype=np.float32)
    c = np.sqrt(3.0 * np.sqrt(d))
    for h, arch in enumerate(mix):
        if arch == SPATIAL:
            s = spatial_features(rng, shape.frame_h, shape.frame_w, d)
            q[:, h, :] += np.tile(4.0 * c * s, (shape.frames_per_block, 1)).astype(np.float32)
            k[:, h, :] += np.tile(c * s, (shape.frames_per_block, 1)).astype(np.float32)
    return (_store(q, shape.dtype), _store(k, shape.dtype), _store(v, shape.dtype))


def rollout_mix(layers: int, n_heads: int, seed: int) -> np.ndarray:
    """Per-(layer, head) archetypes drawn uniformly over the four."""
    return np.random.default_rng(seed).integers(0, 4, size=(layers, n_heads)).astype(np.int8)


def make_stream(shape: LayerShape, seed: int, n_blocks: int, drift: float = 0.0,
                drift_after: int | None = None, mix=None):
    """One layer's blocks 0..n_blocks-1 with persistent planted structure
    (Q, K, V per block, each a [3F][H][d] Tensor3).

    Plants (directions from one generator seeded by ``seed``, noise per block
    from a generator seeded by (seed, block)):
      * Sink head: one direction u; every block's queries get c*u, block 0's
        keys get 4*c*u;
      * Dummy head: a fresh direction v_b per block; block b's queries get
        c*v_b and its keys 4*c*v_b;
      * Spatial head: one feature map s(h, w); queries get 4*a*s, keys a*s;
      * Global head: none.
    Drift: for blocks after ``drift_after`` (default: the block where the
    window first fills), a fraction ``drift`` of each planted query term is
    replaced by an unrelated one of the same norm (a fresh direction, or a
    fresh feature map for Spatial heads), so the structure the classifier saw
    weakens by that fraction."""
    mix = tuple(shape.mix if mix is None else mix)
    if drift_after is None:
        drift_after = shape.blocks_per_window - 1
    H, d, nq = shape.n_heads, shape.head_dim, shape.n_q
    c = np.sqrt(3.0 * np.sqrt(d))
    plant = np.random.default_rng(seed)
    u = {h: random_unit(plant, d) for h in range(H) if mix[h] == SINK}
    s = {h: spatial_features(plant, shape.frame_h, shape.frame_w, d) for h in range(H) if mix[h] == SPATIAL}
    dummy_dirs = {h: [random_unit(plant, d) for _ in range(n_blocks)] for h in range(H) if mix[h] == DUMMY}
    fresh_dirs = [[random_unit(plant, d) for _ in range(H)] for _ in range(n_blocks)]
    fresh_maps = [{h: spatial_features(plant, shape.frame_h, shape.frame_w, d) for h in s} for _ in range(n_blocks)]
    blocks = []
    for b in range(n_blocks):
        rng = np.random.default_rng([seed, b])
        q = rng.standard_normal((nq, H, d), dtype=np.float32)
        k = rng.standard_normal((nq, H, d), dtype=np.float32)
        v = rng.standard_normal((nq, H, d), dtype=np.float32)
        dl = drift if b > drift_after else 0.0
        for h, arch in enumerate(mix):
            if arch == SINK:
                q[:, h, :] += (c * ((1 - dl) * u[h] + dl * fresh_dirs[b][h])).astype(np.float32)
                if b == 0:
                    k[:, h, :] += (4.0 * c * u[h]).astype(np.float32)
            elif arch == DUMMY:
                vb = dummy_dirs[h][b]
                q[:, h, :] += (c * ((1 - dl) * vb + dl * fresh_dirs[b][h])).astype(np.float32)
                k[:, h, :] += (4.0 * c * vb).astype(np.float32)
            elif arch == SPATIAL:
                sq = (1 - dl) * s[h] + dl * fresh_maps[b][h]
                q[:, h, :] += np.tile(4.0 * c * sq, (shape.frames_per_block, 1)).astype(np.float32)
                k[:, h, :] += np.tile(c * s[h], (shape.frames_per_block, 1)).astype(np.float32)
        blocks.append((_store(q, shape.dtype), _store(k, shape.dtype), _store(v, shape.dtype)))
    return blocks
