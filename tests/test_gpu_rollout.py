"""GPU parity for the 30-layer 720P rollout: per-(layer, head) archetypes
drawn uniformly from the seed, one classification per layer at the block
where the window fills, then AR blocks of cache appends (advance, overwrite
on a later denoising step, advance again) with routed attention after each.

  * Every layer's classification against the oracle's, precomputed for the
    same seeded inputs in tests/golden/classify_rollout.json (written by
    tests/golden/make_full_size_golden.py from the oracle alone): labels
    bit-exact, the six per-head statistics within tolerance.
  * Two layers' routed attention after each append against the oracle's
    block-by-block cache model: Sink, Dummy and Global heads on a seeded
    query sample, Spatial heads on one query per frame row of every cell.
The cache of each routed layer is built from the labels the library itself
returned, as the pipeline does."""
import numpy as np
import pytest

import synth
from oracle import headcast_ref as ref
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

hc = pytest.importorskip("head_routed_kv_classify_b300")

R = synth.ROLLOUT_720P
MIX = synth.rollout_mix(R["layers"], R["shape"].n_heads, R["seed"])


def _layer_inputs(layer):
    shape = R["shape"]
    mix = tuple(int(a) for a in MIX[layer])
    return shape, mix, synth.make_layer(shape, seed=R["seed"] * 100 + layer, mix=mix)


@pytest.fixture(scope="module")
def gold():
    g = gu.golden("classify_rollout.json")
    return {e["layer"]: e for e in g["layers"]}


@pytest.mark.parametrize("layer", range(R["layers"]))
def test_rollout_classification_matches_oracle_golden(gold, layer):
    shape, mix, inp = _layer_inputs(layer)
    e = gold[layer]
    assert e["mix"] == list(mix)
    assert gu.input_digest(inp.q.raw, inp.k.raw, inp.v.raw) == e["inputs_sha256"], "inputs changed"
    cfg = hc.config_for(shape)
    q, k, v = (gu.to_dev(x, "bf16") for x in (inp.q, inp.k, inp.v))
    labels, _, stats = hc.hc_classify(cfg, q, k, v)
    hc.hc_get_last_error()
    assert list(labels) == e["labels"], (layer, list(labels), e["labels"], e["margins"])
    gu.assert_stats_close(gu.to_host(stats), e["stats"], f"rollout layer {layer}")


def _routed_vs_oracle(o, bq, model, labels, shape, seed, what):
    idx = gu.sample_queries(shape.n_q, 24, seed=seed)
    cells = gu.per_cell_row_sample(shape, seed + 1)
    for h, a in enumerate(labels):
        qi = cells if a == ref.SPATIAL else idx
        want = ref.routed_head(bq.values, model, int(a), h, query_idx=qi)
        gu.assert_close(o[qi, h], want, "bf16", f"{what} head {h} ({a})")


@pytest.mark.parametrize("layer", [0, 17])
def test_rollout_layer_routed(layer):
    shape, mix, inp = _layer_inputs(layer)
    cfg = hc.config_for(shape)
    q, k, v = (gu.to_dev(x, "bf16") for x in (inp.q, inp.k, inp.v))
    labels, _, _ = hc.hc_classify(cfg, q, k, v)
    assert list(labels) == list(mix), (layer, list(labels), mix)

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
        _routed_vs_oracle(o, bq, model, labels, shape, layer * 7 + n,
                          f"rollout layer {layer} block {block} step {step}")
    info = cache.info()
    assert info["newest_block"] == first + 1 and info["valid_frames"] == shape.window_frames
    hc.hc_get_last_error()
    cache.close()
