"""Host-side helpers of the binding: steady-state memory accounting and the
per-layer label files.  No GPU needed."""
import os

import numpy as np
import pytest

import synth

hc = pytest.importorskip("head_routed_kv_classify_b300")


@pytest.mark.parametrize("name", ["480p", "720p", "1080p"])
def test_memory_report_matches_row_counts(name):
    """Sink/Dummy heads keep one block (3F rows), Spatial/Global heads the
    21-frame window; K and V each; the buffer adds only the work list."""
    shape = synth.SHAPES[name]
    cfg = hc.config_for(shape)
    rep = hc.memory_report(cfg, shape.mix)
    F, d = shape.frame_tokens, shape.head_dim
    rows = 5 * 3 * F + 7 * 21 * F              # 2 S + 3 D one block; 4 P + 3 G the window
    assert rep["kv_bytes"] == 2 * rows * d * 2
    assert rep["monolithic_bytes"] == 2 * 21 * F * 12 * d * 2
    # the backing store adds the work list, its schedule and the split-run workspace
    assert rep["kv_bytes"] + rep["split_bytes"] <= rep["bytes"]
    assert rep["bytes"] < rep["kv_bytes"] + rep["split_bytes"] + 2 * 1024 * 1024
    # 7 of 12 heads keep the whole window: (5/7 + 7) / 12 of the monolithic bytes.
    assert abs(rep["kv_bytes"] / rep["monolithic_bytes"] - (5 * 3 / 21 + 7) / 12) < 1e-12


def test_memory_report_extremes():
    cfg = hc.make_config(12, 128, 45, 80)
    all_global = hc.memory_report(cfg, [3] * 12)
    all_dummy = hc.memory_report(cfg, [1] * 12)
    assert all_global["kv_bytes"] == all_global["monolithic_bytes"]
    assert all_dummy["kv_bytes"] * 7 == all_dummy["monolithic_bytes"]


def test_labels_round_trip(tmp_path):
    mix = synth.rollout_mix(30, 12, 4)
    path = os.path.join(tmp_path, "labels.txt")
    hc.save_labels(path, mix)
    back = hc.load_labels(path)
    assert back.dtype == np.int8 and back.shape == (30, 12)
    assert np.array_equal(back, mix)
    text = open(path).read().splitlines()
    assert text[1] == "0 " + "".join("SDPG"[a] for a in mix[0])


@pytest.mark.parametrize("body,msg", [
    ("0 SDPX\n", "unknown archetype"),
    ("0 SDPG\n1 SDP\n", "heads"),
    ("1 SDPG\n", "out of order"),
    ("# only a comment\n", "no layers"),
    ("0\n", "expected"),
])
def test_labels_rejects_malformed(tmp_path, body, msg):
    path = os.path.join(tmp_path, "bad.txt")
    with open(path, "w") as f:
        f.write(body)
    with pytest.raises(ValueError, match=msg):
        hc.load_labels(path)


def test_save_labels_rejects_non_archetypes(tmp_path):
    with pytest.raises(ValueError):
        hc.save_labels(os.path.join(tmp_path, "x.txt"), [[0, 4]])
