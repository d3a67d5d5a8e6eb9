"""GPU parity for the 30-layer 720P rollout: per-(layer, head) archetypes
drawn uniformly from the seed, one classification per layer at the block
where the window fills, then AR blocks of cache appends (advance, overwrite
on a later denoising step, advance again) with routed attention after each,
compared with the oracle's block-by-block cache model on seeded query
samples.  Two of the 30 layers are checked at full size (the bench runs all
30 through the same calls)."""
import numpy as np
import pytest

import synth
from oracle import headcast_ref as ref
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

hc = pytest.importorskip("head_routed_kv_classify_b300")

R = synth.ROLLOUT_720P
MIX = synth.rollout_mix(R["layers"], R["shape"].n_heads, R["seed"])


@pytest.mark.parametrize("layer", [0, 17])
def test_rollout_layer(layer):
    shape = R["shape"]
    mix = tuple(int(a) for a in MIX[layer])
    inp = synth.make_layer(shape, seed=R["seed"] * 100 + layer, mix=mix)
    cfg = hc.config_for(shape)
    q, k, v = (gu.to_dev(x, "bf16") for x in (inp.q, inp.k, inp.v))
    labels, _, stats = hc.hc_classify(cfg, q, k, v)
    assert list(labels) == list(mix), (layer, list(labels), mix, gu.to_host(stats))

    cache = hc.hc_cache_create(cfg, labels)
    cache.restructure(k, v, 0)
    model = ref.CacheModel(ref.geometry_of(shape))
    blk = shape.n_q
    for b in range(shape.blocks_per_window):
        model.put(b, inp.k.values[b * blk:(b + 1) * blk], inp.v.values[b * blk:(b + 1) * blk])
    first = shape.blocks_per_window
    # (block id, denoising step): advance, overwrite, advance.
    for n, (block, step) in enumerate([(first, 0), (first, 3), (first + 1, 0)]):
        bq, bk, bv = synth.make_block(shape, seed=R["seed"] * 1000 + layer * 10 + n, mix=mix)
        cache.append(block, gu.to_dev(bk, "bf16"), gu.to_dev(bv, "bf16"))
        model.put(block, bk.values, bv.values)
        o = gu.to_host(cache.routed_attention(gu.to_dev(bq, "bf16")))
        idx = gu.sample_queries(shape.n_q, 24, seed=layer * 7 + n)
        want = ref.routed_attention(bq.values, model, labels, query_idx=idx)
        gu.assert_close(o[idx], want, "bf16", f"rollout layer {layer} block {block} step {step}")
    info = cache.info()
    assert info["newest_block"] == first + 1 and info["valid_frames"] == shape.window_frames
    hc.hc_get_last_error()
    cache.close()
