"""GPU cache tests: scripted append/evict sequences on the restructured cache,
checked through routed attention against the oracle's per-block ring model
(window of the newest blocks, block 0 kept as the Sink block), including a
window that is not yet full, wrap-around, overwrites within a block and a
restructure from a later full window; plus the host-side state errors."""
import numpy as np
import pytest

import synth
from oracle import headcast_ref as ref
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

hc = pytest.importorskip("head_routed_kv_classify_b300")

SHAPE = synth.custom_shape("cache", n_heads=4, head_dim=64, frame_h=11, frame_w=13,
                           window_frames=9, dtype="bf16", seed=21, mix=(0, 1, 2, 3))


def _block(seed):
    return synth.make_block(SHAPE, seed)


def _check(cache, model, q_t, labels, what):
    o = gu.to_host(cache.routed_attention(gu.to_dev(q_t, "bf16")))
    want = ref.routed_attention(q_t.values, model, labels)
    gu.assert_close(o, want, "bf16", what)


@pytest.mark.parametrize("labels", [(0, 1, 2, 3), (2, 3, 3, 2), (3, 3, 3, 3)])
def test_append_sequence_matches_ring_model(labels):
    labels = np.array(labels, np.int8)
    cfg = hc.config_for(SHAPE)
    cache = hc.hc_cache_create(cfg, labels)
    model = ref.CacheModel(ref.geometry_of(SHAPE))
    # blocks 0..6 with 3 window blocks: fill, wrap twice; two denoising steps per block
    seed = 100
    for b in range(7):
        for step in range(2):
            q, k, v = _block(seed)
            seed += 1
            cache.append(b, gu.to_dev(k, "bf16"), gu.to_dev(v, "bf16"))
            model.put(b, k.values, v.values)
            info = cache.info()
            assert info["newest_block"] == b
            assert info["valid_frames"] == min(3 * (b + 1), 9)
            _check(cache, model, q, labels, f"block {b} step {step}")
    hc.hc_get_last_error()


def test_restructure_then_append_wraps():
    labels = np.array((0, 1, 2, 3), np.int8)
    cfg = hc.config_for(SHAPE)
    inp = synth.make_layer(SHAPE)
    cache = hc.hc_cache_create(cfg, labels)
    cache.restructure(gu.to_dev(inp.k, "bf16"), gu.to_dev(inp.v, "bf16"), 0)
    model = ref.CacheModel(ref.geometry_of(SHAPE))
    blk = SHAPE.n_q
    for b in range(3):
        model.put(b, inp.k.values[b * blk:(b + 1) * blk], inp.v.values[b * blk:(b + 1) * blk])
    _check(cache, model, inp.q, labels, "after restructure")
    for b in range(3, 6):
        q, k, v = _block(200 + b)
        cache.append(b, gu.to_dev(k, "bf16"), gu.to_dev(v, "bf16"))
        model.put(b, k.values, v.values)
        _check(cache, model, q, labels, f"appended {b}")


def test_restructure_from_later_full_window():
    """A full window that starts after block 0 refreshes every ring slot; the
    Sink block written earlier survives."""
    labels = np.array((0, 1, 2, 3), np.int8)
    cfg = hc.config_for(SHAPE)
    cache = hc.hc_cache_create(cfg, labels)
    model = ref.CacheModel(ref.geometry_of(SHAPE))
    q0, k0, v0 = _block(300)
    cache.append(0, gu.to_dev(k0, "bf16"), gu.to_dev(v0, "bf16"))
    model.put(0, k0.values, v0.values)
    ks, vs = [], []
    for b in range(4, 7):
        _, k, v = _block(300 + b)
        ks.append(k)
        vs.append(v)
    # the oracle model must see 1..6 in order; blocks 1..3 are evicted anyway
    for b in range(1, 4):
        _, k, v = _block(400 + b)
        model.put(b, k.values, v.values)
    for b, (k, v) in zip(range(4, 7), zip(ks, vs)):
        model.put(b, k.values, v.values)
    t = gu.torch()
    kw = t.cat([gu.to_dev(k, "bf16") for k in ks])
    vw = t.cat([gu.to_dev(v, "bf16") for v in vs])
    cache.restructure(kw, vw, first_block_id=4)
    assert cache.info()["valid_frames"] == 9
    q, _, _ = _block(500)
    _check(cache, model, q, labels, "later window")


def test_state_errors():
    labels = np.array((0, 1, 2, 3), np.int8)
    cfg = hc.config_for(SHAPE)
    cache = hc.hc_cache_create(cfg, labels)
    q, k, v = _block(600)
    qd, kd, vd = (gu.to_dev(x, "bf16") for x in (q, k, v))
    with pytest.raises(hc.HeadcastError) as e:
        cache.routed_attention(qd)
    assert e.value.name == "HC_ERR_STATE"
    with pytest.raises(hc.HeadcastError) as e:
        cache.append(1, kd, vd)
    assert e.value.name == "HC_ERR_STATE"
    cache.append(0, kd, vd)
    with pytest.raises(hc.HeadcastError) as e:
        cache.append(2, kd, vd)
    assert e.value.name == "HC_ERR_STATE"
    t = gu.torch()
    kw = t.cat([kd, kd])
    with pytest.raises(hc.HeadcastError) as e:     # 2 blocks from block 1: not full, not from 0
        cache.restructure(kw, kw, first_block_id=1)
    assert e.value.name == "HC_ERR_STATE"
    # Sink heads without block 0
    c2 = hc.hc_cache_create(cfg, labels)
    kw3 = t.cat([kd, kd, kd])
    c2.restructure(kw3, kw3, first_block_id=2)
    with pytest.raises(hc.HeadcastError) as e:
        c2.routed_attention(qd)
    assert e.value.name == "HC_ERR_STATE"
    hc.hc_get_last_error()


def test_memory_accounting():
    """Steady-state cache bytes versus the monolithic window (the paper's
    App. C comparison) for the 720P layer with 2/3/4/3 heads."""
    shape = synth.SHAPES["720p"]
    cfg = hc.config_for(shape)
    cache = hc.hc_cache_create(cfg, np.array(shape.mix, np.int8))
    info = cache.info()
    F, d = shape.frame_tokens, shape.head_dim
    assert info["n_by_archetype"] == [2, 3, 4, 3]
    assert info["rows_by_archetype"] == [2 * 3 * F, 3 * 3 * F, 4 * 21 * F, 3 * 21 * F]
    assert info["monolithic_bytes"] == 2 * 21 * F * 12 * d * 2
    assert info["bytes"] < 0.66 * info["monolithic_bytes"]
