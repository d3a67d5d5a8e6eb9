"""GPU parity of the one-time head classification: labels bit-exact against
the oracle (and the planted archetypes), per-head statistics and the
full-context output against the oracle's."""
import numpy as np
import pytest

import synth
from oracle import headcast_ref as ref
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

hc = pytest.importorskip("head_routed_kv_classify_b300")

SMALL = {
    "tiny": synth.SHAPES["tiny"],
    "tiny_bf16": synth.custom_shape("tiny_bf16", n_heads=4, head_dim=64, frame_h=8, frame_w=8,
                                    window_frames=12, dtype="bf16", seed=10),
    "ragged": synth.custom_shape("ragged", n_heads=8, head_dim=64, frame_h=23, frame_w=27,
                                 window_frames=12, dtype="bf16", seed=11),
    "ragged_d128": synth.custom_shape("ragged_d128", n_heads=4, head_dim=128, frame_h=13,
                                      frame_w=17, window_frames=9, dtype="bf16", seed=12,
                                      mix=(3, 2, 1, 0)),
}



def _run(shape, o_full=True, **cfg_overrides):
    cfg = hc.config_for(shape, **cfg_overrides)
    inp = synth.make_layer(shape)
    q, k, v = (gu.to_dev(x, shape.dtype) for x in (inp.q, inp.k, inp.v))
    of = gu.torch().empty_like(q) if o_full else None
    labels, _, stats = hc.hc_classify(cfg, q, k, v, o_full=of)
    hc.hc_get_last_error()
    return inp, labels, gu.to_host(stats), (gu.to_host(of) if o_full else None)


def _compare_stats(got, want, what):
    gu.assert_stats_close(got, want, what)


@pytest.mark.parametrize("name", list(SMALL))
def test_classify_small(name):
    shape = SMALL[name]
    inp, labels, stats, of = _run(shape)
    geom = ref.geometry_of(shape)
    cls = ref.classify(inp.q.values, inp.k.values, inp.v.values, geom)
    assert list(labels) == list(cls.labels), (labels, cls.labels, cls.margins)
    assert list(labels) == list(inp.planted)
    _compare_stats(stats, cls.stats, name)
    want_full = np.stack([o.o_full for o in cls.outputs], axis=1)
    gu.assert_close(of, want_full, shape.dtype, f"{name} o_full")


@pytest.mark.parametrize("name", list(SMALL))
def test_classify_cell_proxy_small(name):
    """Classification with the deployed cell as the Spatial proxy (the
    proxy-vs-deployed comparison): labels bit-exact and statistics against
    the oracle run with the same proxy."""
    shape = SMALL[name]
    inp, labels, stats, _ = _run(shape, o_full=False, proxy_mode=hc.HC_PROXY_CELL)
    geom = ref.geometry_of(shape, proxy_mode="cell")
    cls = ref.classify(inp.q.values, inp.k.values, inp.v.values, geom)
    assert list(labels) == list(cls.labels), (labels, cls.labels, cls.margins)
    _compare_stats(stats, cls.stats, name + " cell proxy")


def test_classify_480p():
    shape = synth.SHAPES["480p"]
    inp, labels, stats, of = _run(shape)
    cls = ref.classify(inp.q.values, inp.k.values, inp.v.values, ref.geometry_of(shape))
    assert list(labels) == list(cls.labels) == list(inp.planted), cls.margins
    _compare_stats(stats, cls.stats, "480p")
    want_full = np.stack([o.o_full for o in cls.outputs], axis=1)
    gu.assert_close(of, want_full, "bf16", "480p o_full")


@pytest.mark.parametrize("name", ["720p", "1080p"])
def test_classify_full_size_matches_oracle_golden(name):
    """Full-size layers in the benchmark's launch configuration: labels
    bit-exact and per-head statistics within tolerance against the oracle's
    classification of the same seeded inputs (tests/golden/classify_<name>.json,
    written by tests/golden/make_full_size_golden.py from the oracle alone);
    the full-context output on sampled queries against the oracle."""
    shape = synth.SHAPES[name]
    gold = gu.golden(f"classify_{name}.json")
    inp = synth.make_layer(shape)
    assert gu.input_digest(inp.q.raw, inp.k.raw, inp.v.raw) == gold["inputs_sha256"], "inputs changed"
    cfg = hc.config_for(shape)
    q, k, v = (gu.to_dev(x, shape.dtype) for x in (inp.q, inp.k, inp.v))
    of = gu.torch().empty_like(q)
    labels, _, stats = hc.hc_classify(cfg, q, k, v, o_full=of)
    hc.hc_get_last_error()
    assert list(labels) == gold["labels"], (list(labels), gold["labels"], gold["margins"])
    assert gold["labels"] == list(shape.mix)
    gu.assert_stats_close(gu.to_host(stats), gold["stats"], name)
    of = gu.to_host(of)
    idx = gu.sample_queries(shape.n_q, 12, seed=shape.seed + 7)
    geom = ref.geometry_of(shape)
    for h in (0, 2, 5, 9):
        o = ref.classification_outputs(inp.q.values, inp.k.values, inp.v.values, geom, h,
                                       query_idx=idx)
        gu.assert_close(of[idx, h], o.o_full, "bf16", f"{name} o_full head {h}")


def test_classify_thresholds_are_read_from_config():
    """Raising theta above every head's similarity turns every head Global;
    lowering theta_sink below every c_sink turns every head Sink."""
    shape = SMALL["tiny_bf16"]
    inp = synth.make_layer(shape)
    q, k, v = (gu.to_dev(x, "bf16") for x in (inp.q, inp.k, inp.v))
    cfg = hc.config_for(shape, theta_sink=1.5, theta_dummy=1.5, theta_spatial=1.5)
    labels, _, _ = hc.hc_classify(cfg, q, k, v)
    assert list(labels) == [3, 3, 3, 3]
    cfg = hc.config_for(shape, theta_sink=-1.5)
    labels, _, _ = hc.hc_classify(cfg, q, k, v)
    assert list(labels) == [0, 0, 0, 0]
