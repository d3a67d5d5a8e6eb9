"""Classification with the library-held workspace (hc_classify_static_scratch).

Callers such as a plugin whose host framework owns all device memory, or a
real-time loop that may not allocate after start-up, cannot hand
hc_classify a workspace.  This entry point takes its workspace from a fixed
device array inside the library instead.  The GPU test first classifies a
different layer through it (so the array holds another layer's data), then
calls it through the C ABI twice in a row on the test layer and checks each
result against hc_classify with a caller-allocated workspace, under the same
tolerances as the other parity tests, and the labels against the oracle; the
CPU test checks that a layer too large for the array is refused before
anything runs.

The file name makes pytest collect it last.
"""
import ctypes as C

import numpy as np
import pytest

import synth

hc = pytest.importorskip("head_routed_kv_classify_b300")


def _layer():
    # 23x27 grid: cells [10,13]x[10,10,7], 621 tokens per frame (ragged 128-row
    # tiles), 4 heads of d=64, 12-frame window; workspace about 7.8 MB.
    shape = synth.custom_shape("ragged", n_heads=4, head_dim=64, frame_h=23, frame_w=27,
                               window_frames=12, dtype="bf16", seed=11)
    return shape, synth.make_layer(shape)


def test_static_workspace_rejects_large_layer():
    lib = hc.load()
    cfg = hc.config_for(synth.SHAPES["480p"])
    need = hc.hc_classify_scratch_bytes(cfg)
    assert need > hc.STATIC_SCRATCH_BYTES
    st = lib.hc_classify_static_scratch(C.byref(cfg), C.c_void_p(16), C.c_void_p(16),
                                        C.c_void_p(16), cfg.window_frames, C.c_void_p(16), None,
                                        None, None, None)
    assert hc.STATUS_NAMES[st] == "HC_ERR_SIZE"
    assert b"static workspace" in lib.hc_last_error_message()


@pytest.mark.gpu
def test_static_workspace_matches_caller_workspace():
    import torch
    from oracle import headcast_ref as ref
    from tests import gpu_util as gu

    # The library-held workspace keeps whatever the previous call left in it,
    # so the first call classifies a different layer (another grid, window,
    # head count and seed): a row that the second layer's call failed to write
    # would then hold the wrong layer's data, not a correct stale value.
    other = synth.custom_shape("tiny_bf16", n_heads=4, head_dim=64, frame_h=8, frame_w=8,
                               window_frames=12, dtype="bf16", seed=10)
    oth = synth.make_layer(other)
    ocfg = hc.config_for(other)
    lab_other, _, _ = hc.hc_classify_static_scratch(ocfg, *(gu.to_dev(x, "bf16") for x in (oth.q, oth.k, oth.v)))
    assert list(lab_other) == list(oth.planted)

    shape, inp = _layer()
    cfg = hc.config_for(shape)
    assert hc.hc_classify_scratch_bytes(cfg) <= hc.STATIC_SCRATCH_BYTES
    q, k, v = (gu.to_dev(x, "bf16") for x in (inp.q, inp.k, inp.v))
    H, nq, d = shape.n_heads, shape.n_q, shape.head_dim

    o_ref = torch.empty((nq, H, d), dtype=torch.bfloat16, device="cuda")
    lab_ref, _, stats_ref = hc.hc_classify(cfg, q, k, v, o_full=o_ref)
    o_ref = gu.to_host(o_ref)
    stats_ref = stats_ref.cpu().numpy()
    cls = ref.classify(inp.q.values, inp.k.values, inp.v.values, ref.geometry_of(shape))
    assert list(lab_ref) == list(cls.labels), (lab_ref, cls.labels, cls.margins)

    labels_dev = torch.empty(H, dtype=torch.int8, device="cuda")
    stats_dev = torch.empty((H, 6), dtype=torch.float32, device="cuda")
    o_full = torch.empty((nq, H, d), dtype=torch.bfloat16, device="cuda")
    for call in range(2):
        labels_dev.fill_(-1)
        stats_dev.fill_(float("nan"))
        o_full.fill_(float("nan"))
        lab, _, _ = hc.hc_classify_static_scratch(cfg, q, k, v, labels_dev=labels_dev,
                                                  stats_dev=stats_dev, o_full=o_full)
        assert list(lab) == list(lab_ref) == list(cls.labels), (call, lab, lab_ref)
        assert list(labels_dev.cpu().numpy()) == list(lab_ref)
        np.testing.assert_allclose(stats_dev.cpu().numpy(), stats_ref, rtol=0, atol=1e-5)
        gu.assert_close(gu.to_host(o_full), o_ref, "bf16", f"static workspace call {call}")
    hc.hc_get_last_error()
