"""GPU parity of re-classification on a drifting stream (the stability
measurement): a 480P layer whose planted structure persists across blocks
and, after the window first fills, drifts by a fraction of its query plant
(synth.make_stream, seed 501).  At blocks 7 and 12, with drift 0.3 and 0.6,
the window of block 0 (the Sink block) plus the six newest blocks is
classified by the library and compared with the oracle's classification of
the same window (tests/golden/classify_stream.json, written by
tests/golden/make_full_size_golden.py from the oracle alone): labels
bit-exact, per-head statistics within tolerance.  At drift 0.6 the Dummy
and Spatial heads fall back to Global on both sides."""
import numpy as np
import pytest

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

hc = pytest.importorskip("head_routed_kv_classify_b300")


@pytest.fixture(scope="module")
def gold():
    return gu.golden("classify_stream.json")


@pytest.mark.parametrize("drift", [0.3, 0.6])
def test_reclassification_matches_oracle_golden(gold, drift):
    t = gu.torch()
    shape = synth.SHAPES["480p"]
    entries = [e for e in gold["entries"] if e["drift"] == drift]
    assert entries
    blocks = synth.make_stream(shape, seed=gold["seed"], n_blocks=max(e["block"] for e in entries) + 1,
                               drift=drift)
    dq = [gu.to_dev(b[0], "bf16") for b in blocks]
    dk = [gu.to_dev(b[1], "bf16") for b in blocks]
    dv = [gu.to_dev(b[2], "bf16") for b in blocks]
    cfg = hc.config_for(shape)
    for e in entries:
        ids = e["window_blocks"]
        assert ids == [0] + list(range(e["block"] - shape.blocks_per_window + 2, e["block"] + 1))
        kr = np.concatenate([blocks[i][1].raw for i in ids])
        vr = np.concatenate([blocks[i][2].raw for i in ids])
        assert gu.input_digest(blocks[e["block"]][0].raw, kr, vr) == e["inputs_sha256"], "inputs changed"
        k = t.cat([dk[i] for i in ids])
        v = t.cat([dv[i] for i in ids])
        labels, _, stats = hc.hc_classify(cfg, dq[e["block"]], k, v)
        hc.hc_get_last_error()
        what = f"drift {drift} block {e['block']}"
        assert list(labels) == e["labels"], (what, list(labels), e["labels"], e["margins"])
        gu.assert_stats_close(gu.to_host(stats), e["stats"], what)
