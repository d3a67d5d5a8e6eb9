"""The drifting-stream generator used by the re-classification stability
measurement, checked with the oracle on a tiny layer: with no drift the
planted archetypes are recovered at every later block (window = the Sink
block plus the newest blocks), and with full drift the planted query
structure is gone (the Sink head no longer clears its gate)."""
import numpy as np

import synth
from oracle import headcast_ref as ref

SHAPE = synth.custom_shape("stream", n_heads=4, head_dim=64, frame_h=8, frame_w=8,
                           window_frames=12, dtype="fp32", seed=3)


def _classify_at(blocks, b, geom):
    ids = [0] + list(range(b - SHAPE.blocks_per_window + 2, b + 1))
    k = np.concatenate([blocks[i][1].values for i in ids])
    v = np.concatenate([blocks[i][2].values for i in ids])
    return ref.classify(blocks[b][0].values, k, v, geom)


def test_stream_without_drift_keeps_planted_labels():
    blocks = synth.make_stream(SHAPE, seed=5, n_blocks=7, drift=0.0)
    geom = ref.geometry_of(SHAPE)
    for b in (3, 4, 6):
        cls = _classify_at(blocks, b, geom)
        assert list(cls.labels) == list(SHAPE.mix), (b, cls.labels, cls.margins)
        assert np.all(np.abs(cls.margins[:, 0]) >= 0.02)


def test_stream_full_drift_breaks_the_sink_plant():
    blocks = synth.make_stream(SHAPE, seed=5, n_blocks=6, drift=1.0)
    geom = ref.geometry_of(SHAPE)
    assert list(_classify_at(blocks, 3, geom).labels) == list(SHAPE.mix)   # before drift starts
    cls = _classify_at(blocks, 5, geom)
    assert cls.labels[0] != ref.SINK, cls.stats[0]


def test_stream_is_seeded():
    a = synth.make_stream(SHAPE, seed=9, n_blocks=2)
    b = synth.make_stream(SHAPE, seed=9, n_blocks=2)
    for x, y in zip(a, b):
        for t, u in zip(x, y):
            assert np.array_equal(t.raw, u.raw)
