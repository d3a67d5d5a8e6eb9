"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, and its host-only calls (config, validation, cache sizing)
behave as documented."""
import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest

import head_routed_kv_classify_b300 as hc
from head_routed_kv_classify_b300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "headcast.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return hc.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hc_[a-z_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(hc.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", hc.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_every_export_has_declared_argument_types(lib):
    """ctypes passes undeclared integer arguments as C int: a size_t or a
    64-bit value would arrive truncated."""
    for name in hc.EXPORTS:
        assert getattr(lib, name).argtypes is not None, name


def test_library_does_not_need_libcuda(lib):
    out = subprocess.run(["ldd", hc.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libcudart.so" not in out


def test_abi_version_and_strings(lib):
    assert lib.hc_abi_version() == hc.ABI_VERSION == 7
    assert lib.hc_status_string(0) == b"ok"
    assert lib.hc_status_string(7) == b"device-side wait expired"


def test_config_default_holds_ledger_constants(lib):
    cfg = hc.hc_config_default()
    assert abs(cfg.theta_sink - 0.95) < 1e-7 and abs(cfg.theta_dummy - 0.95) < 1e-7
    assert abs(cfg.theta_spatial - 0.95) < 1e-7 and abs(cfg.theta_score - 0.755) < 1e-7
    assert cfg.gamma == 5.0 and cfg.proxy_radius == 2 and (cfg.cell_h, cfg.cell_w) == (10, 10)
    assert cfg.frames_per_block == 3 and cfg.window_frames == 21
    assert cfg.proxy_mode == hc.HC_PROXY_NEIGHBOURHOOD


@pytest.mark.parametrize("field,value,status", [
    ("n_heads", 0, "HC_ERR_SHAPE"), ("n_heads", 65, "HC_ERR_SHAPE"),
    ("head_dim", 96, "HC_ERR_SHAPE"), ("frame_h", 0, "HC_ERR_SHAPE"),
    ("window_frames", 20, "HC_ERR_SHAPE"), ("dtype", 7, "HC_ERR_DTYPE"),
    ("theta_sink", float("nan"), "HC_ERR_INVALID_ARG"), ("softmax_scale", -1.0, "HC_ERR_INVALID_ARG"),
    ("cell_w", 0, "HC_ERR_INVALID_ARG"), ("proxy_radius", -1, "HC_ERR_INVALID_ARG"),
    ("proxy_mode", 2, "HC_ERR_INVALID_ARG"), ("proxy_mode", -1, "HC_ERR_INVALID_ARG"),
    ("spatial_mode", 2, "HC_ERR_INVALID_ARG"),
])
def test_config_validation(lib, field, value, status):
    cfg = hc.make_config(12, 128, 45, 80)
    hc.hc_config_validate(cfg)
    setattr(cfg, field, value)
    with pytest.raises(hc.HeadcastError) as e:
        hc.hc_config_validate(cfg)
    assert e.value.name == status
    assert lib.hc_last_error_message() != b""


def test_cache_bytes_720p(lib):
    cfg = hc.make_config(12, 128, 45, 80)
    labels = [0, 0, 1, 1, 1, 2, 2, 2, 2, 3, 3, 3]
    n = hc.hc_cache_bytes(cfg, labels)
    info = hc.hc_cache_plan_info(cfg, labels)
    F, d = 3600, 128
    rows = 5 * 3 * F + 7 * 21 * F
    assert info["bytes"] == n and info["kv_bytes"] == 2 * rows * d * 2
    assert info["rows_by_archetype"] == [2 * 3 * F, 3 * 3 * F, 4 * 21 * F, 3 * 21 * F]
    assert info["n_by_archetype"] == [2, 3, 4, 3] and info["newest_block"] == -1
    # work list, schedule and alignment on top of the K/V regions and the split workspace
    assert info["kv_bytes"] + info["split_bytes"] <= n < info["kv_bytes"] + info["split_bytes"] + 2 * 1024 * 1024
    mono = 2 * 21 * F * 12 * d * 2
    assert info["monolithic_bytes"] == mono and n < 0.66 * mono


@pytest.mark.parametrize("name,split", [("480p", True), ("720p", False), ("1080p", False)])
def test_long_key_runs_are_split_only_where_they_outlast_the_launch(lib, name, split):
    """The planner splits a Global head's key run across CTAs when one
    256-query item over the whole window is longer than an even share of the
    launch over 148 SMs (the 480P layer: 256 key tiles against about 136),
    and leaves the larger layers, whose items are shorter than that share,
    unsplit.  Split runs need a workspace of 256 rows x d fp32 per piece."""
    import synth
    shape = synth.SHAPES[name]
    info = hc.hc_cache_plan_info(hc.config_for(shape), shape.mix)
    if split:
        per_piece = 256 * (shape.head_dim + 2) * 4
        assert info["split_bytes"] >= 2 * 3 * per_piece       # >= 2 pieces per Global item
    else:
        assert info["split_bytes"] == 0
    cfg32 = hc.config_for(shape)
    cfg32.dtype = hc.HC_FP32                                  # the fp32 path never splits
    assert hc.hc_cache_plan_info(cfg32, shape.mix)["split_bytes"] == 0


@pytest.mark.parametrize("arch", [0, 1, 3])
def test_equal_items_are_split_just_enough_to_even_out_the_ctas(lib, arch):
    """A 720P layer with every head on one key run (Sink, Dummy or Global):
    12 x 43 equal items over 148 CTAs would leave 72 CTAs with one item more
    than the rest.  The planner cuts some of the items, not all, in pieces,
    so that the busiest CTA is within 2 % of the mean (and more than 5 %
    below the unsplit plan), with every piece of at least 8 key tiles."""
    import synth
    shape = synth.SHAPES["720p"]
    labels = [arch] * shape.n_heads
    info = hc.hc_cache_plan_info(hc.config_for(shape), labels)
    items = 12 * -(-shape.n_q // 256)
    assert 0 < info["n_split_runs"] < items
    assert info["n_work_items"] == items - info["n_split_runs"] + info["n_split_pieces"]
    mean = info["planned_total"] / 148
    assert info["planned_span"] <= 1.02 * mean
    tiles = -(-(shape.n_q if arch != 3 else shape.n_k) // 128)
    unsplit = -(-items // 148) * (tiles + 6)
    assert info["planned_span"] * 100 < unsplit * 95
    assert tiles // (info["n_split_pieces"] // info["n_split_runs"]) >= 8


def test_full_attention_workspace_holds_a_balanced_plan(lib):
    """The balanced full attention of a 720P layer (12 x 43 items of the
    whole 75 600-key window over 148 CTAs) splits some key runs: its
    workspace holds at least two pieces' partial outputs (256 rows x d fp32
    plus the row max and sum each).  fp32 layers need no workspace, and the
    sizes are checked like the call's."""
    import synth
    shape = synth.SHAPES["720p"]
    cfg = hc.config_for(shape)
    n = hc.hc_full_attention_ws_bytes(cfg, shape.n_q, shape.window_frames)
    assert n >= 2 * 256 * (shape.head_dim + 2) * 4
    assert n == hc.hc_full_attention_ws_bytes(cfg, shape.n_q, shape.window_frames)   # the kept plan
    cfg32 = hc.config_for(shape)
    cfg32.dtype = hc.HC_FP32
    assert hc.hc_full_attention_ws_bytes(cfg32, shape.n_q, shape.window_frames) == 0
    with pytest.raises(hc.HeadcastError) as e:
        hc.hc_full_attention_ws_bytes(cfg, shape.n_q, 0)
    assert e.value.name == "HC_ERR_SHAPE"
    p = C.c_void_p(0x10000)
    assert lib.hc_full_attention_ws(C.byref(cfg), p, p, p, shape.n_q, shape.window_frames, p, p, 256,
                                    None) == 1   # workspace too small: rejected before any launch


def test_cache_bytes_rejects_bad_labels(lib):
    cfg = hc.make_config(4, 64, 8, 8, 12)
    with pytest.raises(hc.HeadcastError) as e:
        hc.hc_cache_bytes(cfg, [0, 1, 2, 4])
    assert e.value.name == "HC_ERR_INVALID_ARG"


def test_null_arguments_rejected_before_any_cuda_call(lib):
    cfg = hc.make_config(4, 64, 8, 8, 12)
    n = C.c_size_t(0)
    assert lib.hc_classify(C.byref(cfg), None, None, None, 12, None, None, None, None, None, 0,
                           None) == 1
    assert lib.hc_cache_bytes(C.byref(cfg), None, C.byref(n)) == 1
    assert lib.hc_routed_attention(None, None, None, None) == 1
    assert lib.hc_full_attention(C.byref(cfg), None, None, None, 192, 12, None, None) == 1


def test_misaligned_pointers_rejected(lib):
    cfg = hc.make_config(4, 64, 8, 8, 12)
    p = C.c_void_p(0x1008)
    lab = np.zeros(4, np.int8)
    st = lib.hc_classify(C.byref(cfg), p, p, p, 12, C.c_void_p(0x2000), None, None, None,
                         C.c_void_p(0x3000), 1 << 30, None)
    assert st == 4
    assert lib.hc_full_attention(C.byref(cfg), p, p, p, 192, 12, p, None) == 4
    handle = C.c_void_p(0)
    assert lib.hc_cache_create(C.byref(cfg), lab.ctypes.data_as(C.c_void_p), C.c_void_p(0x1010),
                               1 << 30, C.byref(handle)) == 4


def test_classify_rejects_short_window_and_small_scratch(lib):
    cfg = hc.make_config(4, 64, 8, 8, 12)
    p = C.c_void_p(0x10000)
    assert lib.hc_classify(C.byref(cfg), p, p, p, 3, p, None, None, None, p, 1 << 30, None) == 2
    assert lib.hc_classify(C.byref(cfg), p, p, p, 12, p, None, None, None, p, 16, None) == 9
