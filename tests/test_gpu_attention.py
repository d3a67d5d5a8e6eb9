"""GPU parity: full attention and routed attention (after restructuring and
after appends) through the C ABI, against the fp64 oracle on the same seeded
inputs.  Small layers are compared on every output; the 720P/1080P layers on
seeded query samples that the oracle computes one by one."""
import numpy as np
import pytest

import synth
from oracle import headcast_ref as ref
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

hc = pytest.importorskip("head_routed_kv_classify_b300")


def _shape(name, **kw):
    if name in synth.SHAPES:
        return synth.SHAPES[name]
    return synth.custom_shape(name, **kw)


# Small layers that still span several tiles and a ragged tail:
#   tiny        the fp32 4-head layer (8x8 grid, one cell)
#   tiny_bf16   the same geometry in bf16 (d=64)
#   ragged      23x27 grid -> cells [10,13] x [10,10,7], F=621 (ragged 64-tiles)
#   ragged_d128 13x17 grid, d=128, H=3, 9-frame window
SMALL = {
    "tiny": dict(),
    "tiny_bf16": dict(n_heads=4, head_dim=64, frame_h=8, frame_w=8, window_frames=12,
                      dtype="bf16", seed=10),
    "ragged": dict(n_heads=4, head_dim=64, frame_h=23, frame_w=27, window_frames=12,
                   dtype="bf16", seed=11),
    "ragged_d128": dict(n_heads=3, head_dim=128, frame_h=13, frame_w=17, window_frames=9,
                        dtype="bf16", seed=12, mix=(3, 2, 1)),
}


def _inputs(name):
    shape = _shape(name, **SMALL.get(name, {}))
    return shape, synth.make_layer(shape)


def _cache_model(shape, inp):
    geom = ref.geometry_of(shape)
    cache = ref.CacheModel(geom)
    blk = shape.n_q
    for b in range(shape.blocks_per_window):
        cache.put(b, inp.k.values[b * blk:(b + 1) * blk], inp.v.values[b * blk:(b + 1) * blk])
    return geom, cache


@pytest.mark.parametrize("name", list(SMALL))
def test_full_attention_small(name):
    shape, inp = _inputs(name)
    cfg = hc.config_for(shape)
    q, k, v = (gu.to_dev(x, shape.dtype) for x in (inp.q, inp.k, inp.v))
    o = hc.hc_full_attention(cfg, q, k, v)
    want = ref.full_attention(inp.q.values, inp.k.values, inp.v.values)
    gu.assert_close(gu.to_host(o), want, shape.dtype, f"full {name}")
    hc.hc_get_last_error()


def test_full_attention_fewer_keys_and_queries():
    shape, inp = _inputs("ragged")
    cfg = hc.config_for(shape)
    nq, nkf = 333, 5
    q = gu.to_dev(inp.q, "bf16")[:nq].contiguous()
    k = gu.to_dev(inp.k, "bf16")[: nkf * shape.frame_tokens].contiguous()
    v = gu.to_dev(inp.v, "bf16")[: nkf * shape.frame_tokens].contiguous()
    o = hc.hc_full_attention(cfg, q, k, v)
    nk = nkf * shape.frame_tokens
    want = ref.full_attention(inp.q.values[:nq], inp.k.values[:nk], inp.v.values[:nk])
    gu.assert_close(gu.to_host(o), want, "bf16", "full partial")


@pytest.mark.parametrize("name", list(SMALL))
def test_routed_attention_small(name):
    shape, inp = _inputs(name)
    cfg = hc.config_for(shape)
    geom, cache_ref = _cache_model(shape, inp)
    labels = np.array(inp.planted, np.int8)
    cache = hc.hc_cache_create(cfg, labels)
    cache.restructure(gu.to_dev(inp.k, shape.dtype), gu.to_dev(inp.v, shape.dtype), 0)
    o = cache.routed_attention(gu.to_dev(inp.q, shape.dtype))
    want = ref.routed_attention(inp.q.values, cache_ref, labels)
    got = gu.to_host(o)
    for h in range(shape.n_heads):
        gu.assert_close(got[:, h], want[:, h], shape.dtype, f"routed {name} head {h} ({labels[h]})")
    hc.hc_get_last_error()


@pytest.mark.parametrize("name", ["tiny_bf16", "ragged"])
@pytest.mark.parametrize("arch", [0, 1, 2, 3])
def test_routed_single_archetype(name, arch):
    """Every head on one pathway: covers each path on its own."""
    shape, inp = _inputs(name)
    cfg = hc.config_for(shape)
    geom, cache_ref = _cache_model(shape, inp)
    labels = np.full(shape.n_heads, arch, np.int8)
    cache = hc.hc_cache_create(cfg, labels)
    cache.restructure(gu.to_dev(inp.k, shape.dtype), gu.to_dev(inp.v, shape.dtype), 0)
    o = cache.routed_attention(gu.to_dev(inp.q, shape.dtype))
    want = ref.routed_attention(inp.q.values, cache_ref, labels)
    gu.assert_close(gu.to_host(o), want, shape.dtype, f"{name} all-{arch}")
    if arch == ref.GLOBAL:       # Global == unmasked full attention
        full = ref.full_attention(inp.q.values, inp.k.values, inp.v.values)
        gu.assert_close(gu.to_host(o), full, shape.dtype, "global vs full")


def test_spatial_cell_covering_grid_equals_global():
    shape, inp = _inputs("ragged")
    cfg_sp = hc.config_for(shape, cell_h=64, cell_w=64)
    dev = [gu.to_dev(x, "bf16") for x in (inp.q, inp.k, inp.v)]
    outs = []
    for arch in (ref.SPATIAL, ref.GLOBAL):
        c = hc.hc_cache_create(cfg_sp, np.full(shape.n_heads, arch, np.int8))
        c.restructure(dev[1], dev[2], 0)
        outs.append(gu.to_host(c.routed_attention(dev[0])))
    assert np.max(np.abs(outs[0] - outs[1])) <= 2e-2


@pytest.mark.parametrize("name", ["480p"])
def test_routed_attention_480p_all_queries(name):
    shape, inp = _inputs(name)
    cfg = hc.config_for(shape)
    geom, cache_ref = _cache_model(shape, inp)
    labels = np.array(inp.planted, np.int8)
    cache = hc.hc_cache_create(cfg, labels)
    cache.restructure(gu.to_dev(inp.k, "bf16"), gu.to_dev(inp.v, "bf16"), 0)
    o = gu.to_host(cache.routed_attention(gu.to_dev(inp.q, "bf16")))
    want = ref.routed_attention(inp.q.values, cache_ref, labels)
    for h in range(shape.n_heads):
        gu.assert_close(o[:, h], want[:, h], "bf16", f"480p head {h}")


@pytest.mark.parametrize("name", ["720p", "1080p"])
def test_routed_and_full_sampled_full_size(name):
    """Full-size layers in the benchmark's launch configuration, checked on
    seeded query samples (both ends of the block included)."""
    shape, inp = _inputs(name)
    cfg = hc.config_for(shape)
    geom, cache_ref = _cache_model(shape, inp)
    labels = np.array(inp.planted, np.int8)
    q, k, v = (gu.to_dev(x, "bf16") for x in (inp.q, inp.k, inp.v))
    cache = hc.hc_cache_create(cfg, labels)
    cache.restructure(k, v, 0)
    o = gu.to_host(cache.routed_attention(q))
    of = gu.to_host(hc.hc_full_attention(cfg, q, k, v))
    # Sink, Dummy and Global heads on a seeded sample; Spatial heads on one
    # query for every frame row of every cell.
    idx = gu.sample_queries(shape.n_q, 48, seed=shape.seed)
    cells = gu.per_cell_row_sample(shape, seed=shape.seed + 5)
    for h, a in enumerate(labels):
        qi = cells if a == ref.SPATIAL else idx
        want = ref.routed_head(inp.q.values, cache_ref, int(a), h, query_idx=qi)
        gu.assert_close(o[qi, h], want, "bf16", f"{name} routed head {h} ({a})")
    idx2 = gu.sample_queries(shape.n_q, 16, seed=shape.seed + 100)
    want_f = ref.full_attention(inp.q.values, inp.k.values, inp.v.values, query_idx=idx2)
    gu.assert_close(of[idx2], want_f, "bf16", f"{name} full sample")
    hc.hc_get_last_error()


@pytest.mark.parametrize("name", list(SMALL))
def test_routed_sliding_spatial_small(name):
    """The sliding deployed Spatial variant (the cell_h x cell_w window
    centred on the query): Spatial heads stored in raster order and run as
    band items of the masked kernel, next to the other pathways."""
    shape, inp = _inputs(name)
    cfg = hc.config_for(shape, spatial_mode=hc.HC_SPATIAL_SLIDING)
    geom = ref.geometry_of(shape, spatial_mode="sliding")
    cache_ref = ref.CacheModel(geom)
    blk = shape.n_q
    for b in range(shape.blocks_per_window):
        cache_ref.put(b, inp.k.values[b * blk:(b + 1) * blk], inp.v.values[b * blk:(b + 1) * blk])
    for labels in (np.array(inp.planted, np.int8), np.full(shape.n_heads, 2, np.int8)):
        cache = hc.hc_cache_create(cfg, labels)
        cache.restructure(gu.to_dev(inp.k, shape.dtype), gu.to_dev(inp.v, shape.dtype), 0)
        o = gu.to_host(cache.routed_attention(gu.to_dev(inp.q, shape.dtype)))
        want = ref.routed_attention(inp.q.values, cache_ref, labels)
        gu.assert_close(o, want, shape.dtype, f"sliding {name} {list(labels)}")
        hc.hc_get_last_error()


def test_routed_sliding_spatial_720p_sampled_with_append():
    shape, inp = _inputs("720p")
    cfg = hc.config_for(shape, spatial_mode=hc.HC_SPATIAL_SLIDING)
    geom = ref.geometry_of(shape, spatial_mode="sliding")
    cache_ref = ref.CacheModel(geom)
    blk = shape.n_q
    for b in range(shape.blocks_per_window):
        cache_ref.put(b, inp.k.values[b * blk:(b + 1) * blk], inp.v.values[b * blk:(b + 1) * blk])
    labels = np.array(inp.planted, np.int8)
    cache = hc.hc_cache_create(cfg, labels)
    cache.restructure(gu.to_dev(inp.k, "bf16"), gu.to_dev(inp.v, "bf16"), 0)
    bq, bk, bv = synth.make_block(shape, seed=404)
    nb = shape.blocks_per_window
    cache.append(nb, gu.to_dev(bk, "bf16"), gu.to_dev(bv, "bf16"))
    cache_ref.put(nb, bk.values, bv.values)
    o = gu.to_host(cache.routed_attention(gu.to_dev(bq, "bf16")))
    idx = gu.sample_queries(shape.n_q, 40, seed=77)
    want = ref.routed_attention(bq.values, cache_ref, labels, query_idx=idx)
    gu.assert_close(o[idx], want, "bf16", "720p sliding sample")
    hc.hc_get_last_error()
