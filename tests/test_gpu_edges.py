"""GPU parity on the edge cases of the method and the ABI: no queries, a
cache still in warm-up (window not full yet, so Global and Spatial heads see
fewer frames and the Sink block is also the newest), the maximum head count,
a proxy radius of 0 (each query's own position), a cell covering one axis
only, a single-head d = 64 layer, key runs split across CTAs whose pieces
are empty while the window fills, and a classification whose per-token
values are all tied."""
import numpy as np
import pytest

import synth
from oracle import headcast_ref as ref
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

hc = pytest.importorskip("head_routed_kv_classify_b300")


def _model(shape, inp, n_blocks):
    geom = ref.geometry_of(shape)
    cache = ref.CacheModel(geom)
    blk = shape.n_q
    for b in range(n_blocks):
        cache.put(b, inp.k.values[b * blk:(b + 1) * blk], inp.v.values[b * blk:(b + 1) * blk])
    return geom, cache


def test_full_attention_with_no_queries_is_a_no_op():
    shape = synth.custom_shape("e0", n_heads=2, head_dim=64, frame_h=5, frame_w=6, window_frames=6,
                               dtype="bf16", seed=31)
    inp = synth.make_layer(shape)
    cfg = hc.config_for(shape)
    q = gu.to_dev(inp.q, "bf16")[:0].contiguous()
    k, v = gu.to_dev(inp.k, "bf16"), gu.to_dev(inp.v, "bf16")
    o = hc.hc_full_attention(cfg, q, k, v)
    assert o.shape[0] == 0
    hc.hc_get_last_error()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("n_blocks", [1, 2])
def test_routed_attention_during_warm_up(dtype, n_blocks):
    """Restructure from a window holding only the first n blocks (warm-up),
    then route: Global/Spatial heads see 3*n frames, Sink = block 0."""
    shape = synth.custom_shape("warm", n_heads=4, head_dim=64, frame_h=11, frame_w=13,
                               window_frames=12, dtype=dtype, seed=32)
    inp = synth.make_layer(shape)
    cfg = hc.config_for(shape, cell_h=4, cell_w=5)
    geom = ref.geometry_of(shape, cell_h=4, cell_w=5)
    cache_ref = ref.CacheModel(geom)
    blk = shape.n_q
    for b in range(n_blocks):
        cache_ref.put(b, inp.k.values[b * blk:(b + 1) * blk], inp.v.values[b * blk:(b + 1) * blk])
    labels = np.array([0, 1, 2, 3], np.int8)
    cache = hc.hc_cache_create(cfg, labels)
    rows = n_blocks * blk
    cache.restructure(gu.to_dev(inp.k, dtype)[:rows].contiguous(), gu.to_dev(inp.v, dtype)[:rows].contiguous(), 0,
                      n_blocks)
    info = cache.info()
    assert info["valid_frames"] == 3 * n_blocks and info["newest_block"] == n_blocks - 1
    # queries of the newest block in the window
    q = gu.to_dev(inp.q, dtype)
    o = gu.to_host(cache.routed_attention(q))
    want = ref.routed_attention(inp.q.values, cache_ref, labels)
    gu.assert_close(o, want, dtype, f"warm-up {n_blocks} block(s) {dtype}")
    hc.hc_get_last_error()


def test_maximum_head_count():
    shape = synth.custom_shape("h64", n_heads=64, head_dim=64, frame_h=4, frame_w=6, window_frames=6,
                               dtype="bf16", seed=33)
    inp = synth.make_layer(shape)
    cfg = hc.config_for(shape, cell_h=3, cell_w=4)
    geom = ref.geometry_of(shape, cell_h=3, cell_w=4)
    _, cache_ref = (None, ref.CacheModel(geom))
    blk = shape.n_q
    for b in range(shape.blocks_per_window):
        cache_ref.put(b, inp.k.values[b * blk:(b + 1) * blk], inp.v.values[b * blk:(b + 1) * blk])
    labels = np.array([h % 4 for h in range(64)], np.int8)
    q, k, v = (gu.to_dev(x, "bf16") for x in (inp.q, inp.k, inp.v))
    cache = hc.hc_cache_create(cfg, labels)
    cache.restructure(k, v, 0)
    gu.assert_close(gu.to_host(cache.routed_attention(q)), ref.routed_attention(inp.q.values, cache_ref, labels),
                    "bf16", "64 heads routed")
    gu.assert_close(gu.to_host(hc.hc_full_attention(cfg, q, k, v)),
                    ref.full_attention(inp.q.values, inp.k.values, inp.v.values), "bf16", "64 heads full")
    hc.hc_get_last_error()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_classification_with_proxy_radius_zero(dtype):
    """r = 0: the Spatial proxy is each query's own position in every frame."""
    shape = synth.custom_shape("r0", n_heads=4, head_dim=64, frame_h=9, frame_w=10, window_frames=6,
                               dtype=dtype, seed=34)
    inp = synth.make_layer(shape)
    cfg = hc.config_for(shape, proxy_radius=0)
    q, k, v = (gu.to_dev(x, dtype) for x in (inp.q, inp.k, inp.v))
    labels, _, stats = hc.hc_classify(cfg, q, k, v)
    cls = ref.classify(inp.q.values, inp.k.values, inp.v.values, ref.geometry_of(shape, proxy_radius=0))
    assert list(labels) == list(cls.labels), (labels, cls.labels, cls.margins)
    np.testing.assert_allclose(gu.to_host(stats)[:, [0, 1, 2, 3, 5]], cls.stats[:, [0, 1, 2, 3, 5]], atol=2e-3)
    hc.hc_get_last_error()


def test_cell_covering_one_axis_and_single_head():
    """Cells 64 tall (one cell row covers the frame) x 4 wide, one head of
    d = 64 on the Spatial path."""
    shape = synth.custom_shape("axis", n_heads=1, head_dim=64, frame_h=7, frame_w=17, window_frames=9,
                               dtype="bf16", seed=35, mix=(2,))
    inp = synth.make_layer(shape)
    cfg = hc.config_for(shape, cell_h=64, cell_w=4)
    geom = ref.geometry_of(shape, cell_h=64, cell_w=4)
    cache_ref = ref.CacheModel(geom)
    blk = shape.n_q
    for b in range(shape.blocks_per_window):
        cache_ref.put(b, inp.k.values[b * blk:(b + 1) * blk], inp.v.values[b * blk:(b + 1) * blk])
    cache = hc.hc_cache_create(cfg, [2])
    cache.restructure(gu.to_dev(inp.k, "bf16"), gu.to_dev(inp.v, "bf16"), 0)
    o = gu.to_host(cache.routed_attention(gu.to_dev(inp.q, "bf16")))
    gu.assert_close(o, ref.routed_attention(inp.q.values, cache_ref, [2]), "bf16", "one-axis cell")
    hc.hc_get_last_error()


def test_split_key_runs_with_empty_pieces_during_warm_up():
    """One-frame blocks and a 16-frame window: a Global head's run of 16 x 480
    keys (60 tiles) is split into 8 pieces, so with one frame in the window
    (4 tiles) half of the pieces hold no key and must merge as empty shares.
    Checked against the oracle while the window fills and after it wraps."""
    shape = synth.LayerShape("split", 2, 64, 24, 20, 16, "bf16", 36, (3, 1), frames_per_block=1)
    cfg = hc.config_for(shape)
    info = hc.hc_cache_plan_info(cfg, [3, 1])
    assert info["split_bytes"] >= 2 * 8 * 256 * 66 * 4      # 2 items x 8 pieces
    geom = ref.geometry_of(shape)
    cache_ref = ref.CacheModel(geom)
    cache = hc.hc_cache_create(cfg, [3, 1])
    labels = [3, 1]
    for b in range(18):
        q, k, v = synth.make_block(shape, seed=700 + b)
        cache.append(b, gu.to_dev(k, "bf16"), gu.to_dev(v, "bf16"))
        cache_ref.put(b, k.values, v.values)
        if b in (0, 1, 5, 15, 17):
            o = gu.to_host(cache.routed_attention(gu.to_dev(q, "bf16")))
            want = ref.routed_attention(q.values, cache_ref, labels)
            gu.assert_close(o, want, "bf16", f"split runs after block {b}")
    hc.hc_get_last_error()


def test_classification_with_every_token_tied():
    """Every query of a head the same vector and a proxy neighbourhood that
    covers the whole frame: every token of a head has the same four output
    rows, so its per-token cosines are exactly equal on the GPU (the 5th
    percentile is taken over ties: its two ranks are one value), and the
    proxy equals full attention, so the proxy cosine and P5 are 1 and the
    MSE 0 in the oracle.  Labels as the oracle's (the planted Sink and Dummy
    heads, the other two Spatial)."""
    shape = synth.custom_shape("tied", n_heads=4, head_dim=64, frame_h=8, frame_w=8, window_frames=12,
                               dtype="bf16", seed=36)
    inp = synth.make_layer(shape)
    q = synth.Tensor3(np.repeat(inp.q.values[:1], shape.n_q, axis=0), np.repeat(inp.q.raw[:1], shape.n_q, axis=0))
    cfg = hc.config_for(shape, proxy_radius=8)
    labels, _, stats = hc.hc_classify(cfg, gu.to_dev(q, "bf16"), gu.to_dev(inp.k, "bf16"), gu.to_dev(inp.v, "bf16"))
    cls = ref.classify(q.values, inp.k.values, inp.v.values, ref.geometry_of(shape, proxy_radius=8))
    st = gu.to_host(stats)
    assert list(labels) == list(cls.labels) == [ref.SINK, ref.DUMMY, ref.SPATIAL, ref.SPATIAL], (labels, cls.labels)
    np.testing.assert_allclose(cls.stats[:, 2:4], 1.0, atol=1e-12)       # c_spatial and P5 in the oracle
    np.testing.assert_allclose(st[:, 2:4], cls.stats[:, 2:4], atol=1e-5)
    np.testing.assert_allclose(st[:, 4], cls.stats[:, 4], atol=1e-6)      # MSE
    hc.hc_get_last_error()
