"""Pins for the fp64 CPU oracle (no GPU).

Each test ties the oracle to something other than itself: the constants the
pages print, closed forms of softmax attention, library routines
(scipy's softmax, numpy's percentile, torch's bf16 rounding), a scalar
brute-force twin that decides key membership by predicate, and invariants of
the key sets.  A dropped term, a wrong sign or index, or a transposed operand
in the oracle fails at least one of them.
"""
import dataclasses
import json
import math
import os

import numpy as np
import pytest
import scipy.special

from oracle import brute
from oracle import headcast_ref as ref
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tiny_geom(**kw):
    base = dict(n_heads=2, head_dim=4, frame_h=5, frame_w=7, window_frames=6,
                proxy_radius=1, cell_h=3, cell_w=3)
    base.update(kw)
    return ref.Geometry(**base)


def rand_qkv(geom, seed, n_q=None):
    rng = np.random.default_rng(seed)
    n_q = geom.block_tokens if n_q is None else n_q
    q = rng.standard_normal((n_q, geom.n_heads, geom.head_dim))
    k = rng.standard_normal((geom.n_k, geom.n_heads, geom.head_dim))
    v = rng.standard_normal((geom.n_k, geom.n_heads, geom.head_dim))
    return q, k, v


# ---------------------------------------------------------------- constants

def test_page_constants_are_the_defaults():
    with open(os.path.join(GOLDEN, "page_constants.json")) as f:
        c = json.load(f)
    th = ref.Thresholds()
    assert (th.theta_sink, th.theta_dummy, th.theta_spatial) == (
        c["theta_sink"], c["theta_dummy"], c["theta_spatial"])
    assert th.theta_score == c["theta_score"] and th.gamma == c["gamma"]
    g = ref.Geometry(1, 8, 8, 8, 12)
    assert g.proxy_radius == c["proxy_radius"] and 2 * g.proxy_radius + 1 == c["proxy_window"]
    assert (g.cell_h, g.cell_w) == (c["cell_h"], c["cell_w"])


# ---------------------------------------------------------------- attention

def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((17, 8)) * 3
    k = rng.standard_normal((40, 8)) * 3
    ones = np.ones((40, 3))
    o = ref.softmax_attention(q, k, ones, 0.7)
    assert np.max(np.abs(o - 1.0)) < 1e-12


def test_closed_forms():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((5, 6))
    k = rng.standard_normal((9, 6))
    const = np.tile(rng.standard_normal(6), (9, 1))
    assert np.allclose(ref.softmax_attention(q, k, const, 0.4), const[:5], atol=1e-13)
    v1 = rng.standard_normal((1, 6))
    assert np.allclose(ref.softmax_attention(q, k[:1], v1, 0.4), np.tile(v1, (5, 1)), atol=1e-13)
    same_k = np.tile(k[:1], (9, 1))
    v = rng.standard_normal((9, 6))
    assert np.allclose(ref.softmax_attention(q, same_k, v, 0.4),
                       np.tile(v.mean(axis=0), (5, 1)), atol=1e-13)


def test_large_logits_are_stable():
    q = np.array([[100.0, 0.0]])
    k = np.array([[100.0, 0.0], [99.0, 0.0], [-50.0, 0.0]])
    v = np.array([[1.0, 0.0], [0.0, 1.0], [5.0, 5.0]])
    o = ref.softmax_attention(q, k, v, 1.0)
    w = scipy.special.softmax(np.array([10000.0, 9900.0, -5000.0]))
    assert np.allclose(o[0], w @ v)


def test_block_sets_equal_masked_full_attention():
    """Sink and Dummy are full attention under a -inf block mask; the mask is
    applied here through scipy's softmax, not through the oracle."""
    geom = tiny_geom()
    q, k, v = rand_qkv(geom, 3)
    blk = geom.block_tokens
    for h in range(geom.n_heads):
        o = ref.classification_outputs(q, k, v, geom, h)
        s = (q[:, h, :] @ k[:, h, :].T) / math.sqrt(geom.head_dim)
        for sel, got in ((np.arange(geom.n_k) < blk, o.o_sink),
                         (np.arange(geom.n_k) >= geom.n_k - blk, o.o_dummy),
                         (np.ones(geom.n_k, bool), o.o_full)):
            p = scipy.special.softmax(np.where(sel[None, :], s, -np.inf), axis=1)
            assert np.allclose(got, p @ v[:, h, :], atol=1e-12)


@pytest.mark.parametrize("kind", ["full", "sink", "dummy", "proxy", "cell", "sliding"])
def test_brute_force_twin(kind):
    geom = tiny_geom()
    if kind == "sliding":
        geom = dataclasses.replace(geom, spatial_mode="sliding", cell_h=4, cell_w=3)
    q, k, v = rand_qkv(geom, 4)
    scale = 1 / math.sqrt(geom.head_dim)
    for h in range(geom.n_heads):
        want = np.array(brute.keyset_outputs(q, k, v, h, geom.frame_h, geom.frame_w,
                                             geom.block_tokens, kind, scale,
                                             radius=geom.proxy_radius, cell_h=geom.cell_h,
                                             cell_w=geom.cell_w))
        if kind in ("cell", "sliding"):
            cache = ref.CacheModel(geom)
            for b in range(geom.blocks_per_window):
                sl = slice(b * geom.block_tokens, (b + 1) * geom.block_tokens)
                cache.put(b, k[sl], v[sl])
            got = ref.routed_head(q, cache, ref.SPATIAL, h)
        else:
            o = ref.classification_outputs(q, k, v, geom, h)
            got = dict(full=o.o_full, sink=o.o_sink, dummy=o.o_dummy, proxy=o.o_spatial)[kind]
        assert np.max(np.abs(got - want)) < 1e-12


def test_proxy_covering_grid_equals_global():
    geom = tiny_geom(proxy_radius=7)
    q, k, v = rand_qkv(geom, 5)
    for h in range(geom.n_heads):
        o = ref.classification_outputs(q, k, v, geom, h)
        assert np.allclose(o.o_spatial, o.o_full, atol=1e-12)


def test_cell_covering_grid_equals_global():
    geom = tiny_geom(cell_h=8, cell_w=8)        # 5x7 grid -> one cell
    q, k, v = rand_qkv(geom, 6)
    cache = ref.CacheModel(geom)
    for b in range(geom.blocks_per_window):
        sl = slice(b * geom.block_tokens, (b + 1) * geom.block_tokens)
        cache.put(b, k[sl], v[sl])
    labels_sp = [ref.SPATIAL] * geom.n_heads
    labels_gl = [ref.GLOBAL] * geom.n_heads
    assert np.allclose(ref.routed_attention(q, cache, labels_sp),
                       ref.routed_attention(q, cache, labels_gl), atol=1e-12)
    assert np.allclose(ref.routed_attention(q, cache, labels_gl),
                       ref.full_attention(q, k, v), atol=1e-12)


def test_proxy_neighbour_count_closed_form():
    geom = ref.Geometry(1, 4, 9, 13, 6, proxy_radius=2)
    for h in range(geom.frame_h):
        for w in range(geom.frame_w):
            nh = min(h + 2, geom.frame_h - 1) - max(h - 2, 0) + 1
            nw = min(w + 2, geom.frame_w - 1) - max(w - 2, 0) + 1
            keys = ref.proxy_keys(h, w, 6, geom)
            assert len(keys) == 6 * nh * nw
            assert len(set(keys.tolist())) == len(keys)


@pytest.mark.parametrize("n,expect", [
    (8, [8]), (30, [10, 10, 10]), (52, [10, 10, 10, 10, 12]),
    (45, [10, 10, 10, 10, 5]), (80, [10] * 8), (68, [10] * 6 + [8]), (120, [10] * 12),
    (14, [14]), (15, [10, 5]), (24, [10, 14]), (25, [10, 10, 5]),
])
def test_cells_tile_the_axis(n, expect):
    cells = ref.cell_partition(n, 10)
    assert [z for _, z in cells] == expect
    assert cells[0][0] == 0
    for (s0, z0), (s1, _) in zip(cells, cells[1:]):
        assert s0 + z0 == s1
    assert cells[-1][0] + cells[-1][1] == n


def test_cell_keys_partition_each_frame():
    geom = ref.Geometry(1, 4, 13, 17, 3, cell_h=4, cell_w=5)
    seen = np.zeros(geom.n_k, int)
    ch = ref.cell_partition(geom.frame_h, geom.cell_h)
    cw = ref.cell_partition(geom.frame_w, geom.cell_w)
    for h0, _ in ch:
        for w0, _ in cw:
            seen[ref.cell_keys(h0, w0, 3, geom)] += 1
    assert np.all(seen == 1)


def test_frame_permutation_invariance():
    """Global and cell outputs do not depend on the order of cached frames,
    which is what lets a ring buffer hold them in slot order."""
    geom = tiny_geom()
    q, k, v = rand_qkv(geom, 7)
    perm = np.random.default_rng(0).permutation(geom.window_frames)
    idx = np.concatenate([np.arange(f * geom.F, (f + 1) * geom.F) for f in perm])
    for keyset in (ref.cell_keys, ref.proxy_keys):
        a = ref.attend_by_position(q[:, 0], k[:, 0], v[:, 0], geom, geom.window_frames, keyset,
                                   0.5, np.arange(geom.block_tokens))
        b = ref.attend_by_position(q[:, 0], k[idx, 0], v[idx, 0], geom, geom.window_frames,
                                   keyset, 0.5, np.arange(geom.block_tokens))
        assert np.allclose(a, b, atol=1e-12)


# ---------------------------------------------------------------- statistics

def test_cosine_pins():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((6, 5))
    assert np.allclose(ref.cosine_rows(x, x), 1.0)
    assert np.allclose(ref.cosine_rows(x, -x), -1.0)
    assert np.allclose(ref.cosine_rows(x, 3.5 * x), 1.0)
    e = np.eye(5)
    assert np.allclose(ref.cosine_rows(e[:4], e[1:5]), 0.0)
    z = np.zeros((2, 5))
    assert list(ref.cosine_rows(z, z)) == [1.0, 1.0]
    assert list(ref.cosine_rows(z, x[:2])) == [0.0, 0.0]
    for a, b in zip(x, x[::-1]):
        assert abs(ref.cosine_rows(a[None], b[None])[0] - brute.cosine(a, b)) < 1e-14


def test_percentile_pins():
    assert ref.percentile_linear(np.arange(101), 5.0) == 5.0
    assert ref.percentile_linear(np.arange(21)[::-1], 5.0) == 1.0
    assert ref.percentile_linear([3.0], 5.0) == 3.0
    assert abs(ref.percentile_linear([0.0, 1.0], 5.0) - 0.05) < 1e-15
    rng = np.random.default_rng(9)
    for n in (2, 3, 7, 192, 1000, 4680):
        x = rng.standard_normal(n)
        assert abs(ref.percentile_linear(x, 5.0) - np.percentile(x, 5.0, method="linear")) < 1e-14


def test_statistics_pins():
    rng = np.random.default_rng(10)
    o = rng.standard_normal((50, 8))
    cs = rng.uniform(0.9, 1.0, 50)
    st = ref.head_statistics(cs, cs * 0.5, cs, o, o, 5.0)
    assert st[4] == 0.0                       # MSE of identical outputs
    assert st[5] == st[3]                     # score = P5 when MSE is 0
    assert abs(st[0] - cs.mean()) < 1e-15 and abs(st[1] - 0.5 * cs.mean()) < 1e-15
    o2 = o + 0.1                              # every channel off by 0.1 -> MSE 0.01
    st2 = ref.head_statistics(cs, cs, cs, o2, o, 5.0)
    assert abs(st2[4] - 0.01) < 1e-15
    assert abs(st2[5] - (st2[3] - 0.05)) < 1e-15


# ---------------------------------------------------------------- decision rule

EPS = 1e-6


def _st(c_s=0.0, c_d=0.0, c_sp=0.0, p5=0.0, mse=0.0):
    return (c_s, c_d, c_sp, p5, mse, p5 - 5.0 * mse)


@pytest.mark.parametrize("stats,label", [
    (_st(c_s=0.95), ref.SINK),
    (_st(c_s=0.95 - EPS), ref.GLOBAL),
    (_st(c_s=0.95 + EPS, c_d=1.0, c_sp=1.0, p5=1.0), ref.SINK),       # order: Sink first
    (_st(c_d=0.95), ref.DUMMY),
    (_st(c_d=0.95 - EPS), ref.GLOBAL),
    (_st(c_d=0.99, c_sp=1.0, p5=1.0), ref.DUMMY),                     # Dummy before Spatial
    (_st(c_sp=0.95, p5=0.755), ref.SPATIAL),
    (_st(c_sp=0.95 - EPS, p5=0.9), ref.GLOBAL),
    (_st(c_sp=0.99, p5=0.755 - EPS), ref.GLOBAL),                     # score gate
    (_st(c_sp=0.99, p5=0.80, mse=0.009), ref.SPATIAL),                # 0.80-0.045 = 0.755
    (_st(c_sp=0.99, p5=0.80, mse=0.0091), ref.GLOBAL),                # MSE is a penalty
    (_st(c_sp=0.99, p5=0.75, mse=0.0), ref.GLOBAL),
])
def test_decision_rule(stats, label):
    assert ref.decide(stats) == label


def test_margins_sign():
    m = ref.margins(_st(c_s=0.97, c_d=0.5, c_sp=0.96, p5=0.8, mse=0.001))
    assert m[0] > 0 and m[1] < 0 and m[2] > 0 and abs(m[3] - (0.8 - 0.005 - 0.755)) < 1e-12


# ---------------------------------------------------------------- cache model

def test_cache_model_ring():
    geom = ref.Geometry(1, 2, 2, 2, 9)     # 3 blocks per window, 12 tokens per block
    cache = ref.CacheModel(geom)
    blk = lambda b: (np.full((12, 1, 2), float(b)), np.full((12, 1, 2), -float(b)))
    for b in range(5):
        cache.put(b, *blk(b))
    assert cache.window_ids() == [2, 3, 4]
    assert sorted(cache.blocks) == [0, 2, 3, 4]          # block 0 kept as the sink
    assert cache.sink()[0][0, 0, 0] == 0.0
    cache.put(4, *blk(40))                              # same id: overwrite
    assert cache.current()[0][0, 0, 0] == 40.0
    k, _ = cache.window()
    assert list(k[::12, 0, 0]) == [2.0, 3.0, 40.0]
    with pytest.raises(ValueError):
        cache.put(6, *blk(6))


def _scipy_attention(q, k, v, scale):
    """softmax(q k^T * scale) v through scipy's softmax (not the oracle's)."""
    return scipy.special.softmax((q @ k.T) * scale, axis=1) @ v


def test_routed_sink_and_dummy_read_block_zero_and_the_newest_block():
    """Routed Sink heads attend over the block put with id 0 (kept after the
    window has slid past it), Dummy heads over the newest block (after an
    overwrite, its latest contents), Global heads over the window only.
    Swapping any two of these key sets in the oracle fails here."""
    geom = ref.Geometry(3, 4, 2, 3, 6, cell_h=1, cell_w=1)   # 2 blocks per window, 6-token blocks
    rng = np.random.default_rng(12)
    blocks = {b: (rng.standard_normal((6, 3, 4)), rng.standard_normal((6, 3, 4))) for b in range(5)}
    cache = ref.CacheModel(geom)
    for b in range(4):
        cache.put(b, *blocks[b])
    cache.put(4, *blocks[4])
    newest = (rng.standard_normal((6, 3, 4)), rng.standard_normal((6, 3, 4)))
    cache.put(4, *newest)                                     # a later denoising step of block 4
    q = rng.standard_normal((6, 3, 4))
    scale = 1 / math.sqrt(4)
    labels = [ref.SINK, ref.DUMMY, ref.GLOBAL]
    out = ref.routed_attention(q, cache, labels)
    win_k = np.concatenate([blocks[3][0], newest[0]])
    win_v = np.concatenate([blocks[3][1], newest[1]])
    for h, (k, v) in enumerate([blocks[0], newest, (win_k, win_v)]):
        want = _scipy_attention(q[:, h], k[:, h], v[:, h], scale)
        assert np.max(np.abs(out[:, h] - want)) < 1e-12, h
    # and they differ from one another on these inputs
    assert np.max(np.abs(_scipy_attention(q[:, 0], blocks[0][0][:, 0], blocks[0][1][:, 0], scale) -
                         _scipy_attention(q[:, 0], newest[0][:, 0], newest[1][:, 0], scale))) > 1e-2


# ---------------------------------------------------------------- inputs

def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(100000) * rng.choice([1e-3, 1.0, 1e3], 100000)).astype(np.float32)
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0]      # ties to even
    ours = synth.bf16_to_f32(synth.bf16_bits(x))
    theirs = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours, theirs)


# ---------------------------------------------------------------- planted heads

def _check_planted(shape):
    inp = synth.make_layer(shape)
    geom = ref.geometry_of(shape)
    cls = ref.classify(inp.q.values, inp.k.values, inp.v.values, geom)
    assert list(cls.labels) == list(inp.planted), (cls.labels, cls.stats)
    # every gate that decides is at least 0.02 away from its threshold
    for h in range(geom.n_heads):
        lab = cls.labels[h]
        m = cls.margins[h]
        deciding = {ref.SINK: [0], ref.DUMMY: [0, 1], ref.SPATIAL: [0, 1, 2, 3],
                    ref.GLOBAL: [0, 1]}[int(lab)]
        for g in deciding:
            assert abs(m[g]) >= 0.02, (h, m)
        if lab == ref.GLOBAL:
            assert m[2] <= -0.02 or m[3] <= -0.02, (h, m)
    return cls


def test_planted_tiny_recovered():
    _check_planted(synth.SHAPES["tiny"])


@pytest.mark.slow
def test_planted_480p_recovered():
    _check_planted(synth.SHAPES["480p"])


def test_cell_proxy_mode_uses_the_deployed_cells():
    """With the cell proxy the classifier's Spatial output is exactly the
    deployed Spatial path's output (the same key sets), and a cell covering
    the grid turns it into the full-context output."""
    shape = synth.custom_shape("cellproxy", n_heads=2, head_dim=16, frame_h=13, frame_w=11,
                               window_frames=6, dtype="fp32", seed=21, mix=(2, 3))
    inp = synth.make_layer(shape)
    q, k, v = inp.q.values, inp.k.values, inp.v.values
    geom = ref.geometry_of(shape, proxy_mode="cell")
    cache = ref.CacheModel(geom)
    blk = shape.n_q
    for b in range(shape.blocks_per_window):
        cache.put(b, k[b * blk:(b + 1) * blk], v[b * blk:(b + 1) * blk])
    for h in range(2):
        o = ref.classification_outputs(q, k, v, geom, h)
        want = ref.routed_head(q, cache, ref.SPATIAL, h)
        assert np.array_equal(o.o_spatial, want)
    big = ref.geometry_of(shape, proxy_mode="cell", cell_h=64, cell_w=64)
    o = ref.classification_outputs(q, k, v, big, 0)
    assert np.max(np.abs(o.o_spatial - o.o_full)) < 1e-12
    # the neighbourhood proxy differs from the cell proxy on this grid
    o_n = ref.classification_outputs(q, k, v, ref.geometry_of(shape), 0)
    assert np.max(np.abs(o_n.o_spatial - ref.classification_outputs(q, k, v, geom, 0).o_spatial)) > 1e-3


def test_sliding_window_pins():
    """The sliding Spatial key set: a centred window covering the grid from
    every position equals Global; an interior query of a 10x10 window sees
    exactly 100 keys per frame with itself at offset (5, 5); at a corner the
    window is clipped to rows/cols 0..4."""
    geom = tiny_geom()
    big = dataclasses.replace(geom, spatial_mode="sliding", cell_h=2 * geom.frame_h, cell_w=2 * geom.frame_w)
    q, k, v = rand_qkv(geom, 5)
    cache = ref.CacheModel(big)
    for b in range(geom.blocks_per_window):
        sl = slice(b * geom.block_tokens, (b + 1) * geom.block_tokens)
        cache.put(b, k[sl], v[sl])
    for h in range(geom.n_heads):
        got = ref.routed_head(q, cache, ref.SPATIAL, h)
        want = ref.full_attention(q, k, v)[:, h, :]
        assert np.max(np.abs(got - want)) < 1e-12
    g = ref.Geometry(1, 8, 30, 52, 21, spatial_mode="sliding")
    keys = ref.sliding_keys(12, 20, 1, g)
    assert len(keys) == 100
    rows, cols = keys // 52, keys % 52
    assert rows.min() == 7 and rows.max() == 16 and cols.min() == 15 and cols.max() == 24
    corner = ref.sliding_keys(0, 0, 2, g)
    assert len(corner) == 2 * 25 and (corner % g.F // 52).max() == 4 and (corner % g.F % 52).max() == 4
