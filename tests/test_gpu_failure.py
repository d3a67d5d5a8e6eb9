"""Failure detection on the GPU without a GPU fault: with the stall test hook
on, the tensor-core attention kernel's producer stops after one key tile, the
other roles' bounded waits (2 ms) expire, every CTA drains its own work, frees
its tensor memory and returns, and hc_get_last_error reports HC_ERR_TIMEOUT.
The context stays usable: with the hook off, the same call gives the same
output as before, and the status word reads OK."""
import numpy as np
import pytest

import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

hc = pytest.importorskip("head_routed_kv_classify_b300")


def test_expired_waits_report_timeout_and_leave_the_context_usable():
    shape = synth.custom_shape("ragged", n_heads=4, head_dim=64, frame_h=23, frame_w=27,
                               window_frames=12, dtype="bf16", seed=11)
    inp = synth.make_layer(shape)
    cfg = hc.config_for(shape)
    q, k, v = (gu.to_dev(x, "bf16") for x in (inp.q, inp.k, inp.v))
    cache = hc.hc_cache_create(cfg, [3, 3, 2, 3])
    cache.restructure(k, v, 0)
    before = gu.to_host(cache.routed_attention(q))
    hc.hc_get_last_error()
    hc.hc_debug_inject_stall(True)
    try:
        cache.routed_attention(q)
        with pytest.raises(hc.HeadcastError) as err:
            hc.hc_get_last_error()
        assert err.value.name == "HC_ERR_TIMEOUT"
        # full attention goes through the same kernel and the same path
        hc.hc_full_attention(cfg, q, k, v)
        with pytest.raises(hc.HeadcastError) as err:
            hc.hc_get_last_error()
        assert err.value.name == "HC_ERR_TIMEOUT"
    finally:
        hc.hc_debug_inject_stall(False)
    after = gu.to_host(cache.routed_attention(q))
    hc.hc_get_last_error()
    assert np.array_equal(before, after)
    cache.close()
