"""The routed launch's work list, read on the host (hc_cache_plan_items) and
checked against the pathways' definitions without a GPU: every head's
queries are covered once, each item reads its own archetype's key run at the
row the cache layout puts it, split key runs are cut into whole pieces, and
the schedule is a valid longest-first deal over 148 CTAs.

Pathways [Pith review of HeadCast, major comment 2; Figure 3 caption]: Sink
heads attend to the first block, Dummy heads to the newest block, Spatial
heads to their own cell in every window frame, Global heads to the whole
window.  The cache holds each head's rows one head after another, a block
(frames_per_block frames) for Sink and Dummy heads and the window for
Spatial and Global heads; a Spatial head's window is cell-major (every frame
of cell (0, 0), then cell (0, 1), ...)."""
import collections

import numpy as np
import pytest
from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

import head_routed_kv_classify_b300 as hc
import synth
from head_routed_kv_classify_b300 import build

CTAS = 148      # the CTAs a launch is planned for (the SM count)
KEY_TILE = 128  # keys per tile of the tensor-core kernel


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return hc.load()


def n_cells(n, c):
    """Cells along an axis of n tokens: the rounded count, the last cell
    taking the remainder (ledger: "10x10 with rounded remainder")."""
    return max(1, (2 * n + c) // (2 * c))


def extents(n, c):
    k = n_cells(n, c)
    return [c] * (k - 1) + [n - (k - 1) * c]


def check_plan(cfg, labels):
    labels = list(labels)
    items = hc.hc_cache_plan_items(cfg, labels)
    info = hc.hc_cache_plan_info(cfg, labels)
    assert len(items) == info["n_work_items"]
    fh, fw, fpb, wf = cfg.frame_h, cfg.frame_w, cfg.frames_per_block, cfg.window_frames
    F = fh * fw
    nq = fpb * F
    sliding = cfg.spatial_mode == hc.HC_SPATIAL_SLIDING

    # The cache layout: head after head.
    row0, r = [], 0
    for a in labels:
        row0.append(r)
        r += nq if a in (hc.SINK, hc.DUMMY) else wf * F

    # Launch order: the main launch's CTAs in order, then the band launch's.
    order = list(zip(items["launch"], items["cta"]))
    assert order == sorted(order)
    assert np.all(items["cta"] < CTAS) and np.all(items["cta"] >= 0)
    assert set(items["launch"]) <= ({0, 1} if sliding else {0})

    # Split key runs: whole pieces, consecutive partial slots, >= 8 key tiles each.
    parts = items["part"][items["part"] >= 0]
    assert sorted(parts) == list(range(info["n_split_pieces"]))
    runs = collections.defaultdict(list)
    for w in items:
        if w["n_chunks"] > 1:
            assert w["kind"] == hc.HC_ITEM_RANGE and cfg.dtype == hc.HC_BF16
            runs[(w["head"], w["q0"], w["nq"], w["k_row0"], w["k_len"])].append(w)
        else:
            assert w["chunk"] == 0 and w["part"] == -1
    assert len(runs) == info["n_split_runs"]
    for key, pieces in runs.items():
        n = pieces[0]["n_chunks"]
        assert sorted(p["chunk"] for p in pieces) == list(range(n))
        assert all(p["n_chunks"] == n for p in pieces)
        assert len({int(p["part"]) - int(p["chunk"]) for p in pieces}) == 1
        tiles = -(-key[4] // KEY_TILE)
        assert -(-tiles // n) >= 8

    # Per head: the right key run and every query exactly once.
    whole = items[items["chunk"] == 0]
    for h, a in enumerate(labels):
        mine = whole[whole["head"] == h]
        assert len(mine) > 0
        if a in (hc.SINK, hc.DUMMY, hc.GLOBAL):
            assert np.all(mine["kind"] == hc.HC_ITEM_RANGE)
            assert np.all(mine["k_row0"] == row0[h])
            assert np.all(mine["k_len"] == (wf * F if a == hc.GLOBAL else nq))
            cover = np.zeros(nq, np.int32)
            for w in mine:
                cover[w["q0"]:w["q0"] + w["nq"]] += 1
            assert np.all(cover == 1), (h, a)
        elif not sliding:
            assert np.all(mine["kind"] == hc.HC_ITEM_CELL)
            hz, wz = extents(fh, cfg.cell_h), extents(fw, cfg.cell_w)
            ncw = len(wz)
            seen = set()
            for ci, ch in enumerate(hz):
                for cj, cw in enumerate(wz):
                    cell = ci * ncw + cj
                    cit = mine[mine["cell"] == cell]
                    # Cell-major rows: the cells before it in every frame.
                    before = sum(hz[:ci]) * fw + ch * sum(wz[:cj])
                    assert np.all(cit["k_row0"] == row0[h] + wf * before), (h, ci, cj)
                    assert np.all(cit["k_len"] == wf * ch * cw)
                    cover = np.zeros(fpb * ch * cw, np.int32)
                    for w in cit:
                        cover[w["q0"]:w["q0"] + w["nq"]] += 1
                    assert np.all(cover == 1), (h, ci, cj)
                    seen.add(cell)
            assert seen == set(int(c) for c in mine["cell"])
            # The cells' key runs tile the head's window in order.
            runs_h = sorted({(int(w["k_row0"]), int(w["k_len"])) for w in mine})
            pos = row0[h]
            for k0, kl in runs_h:
                assert k0 == pos
                pos += kl
            assert pos == row0[h] + wf * F
        elif cfg.dtype == hc.HC_BF16:
            assert np.all(mine["kind"] == hc.HC_ITEM_PATCH) and np.all(mine["launch"] == 1)
            assert np.all(mine["k_row0"] == row0[h]) and np.all(mine["k_len"] == wf * F)
            assert sorted(mine["cell"]) == list(range(len(mine)))
        else:
            assert np.all(mine["kind"] == hc.HC_ITEM_BAND) and np.all(mine["launch"] == 1)
            assert np.all(mine["k_row0"] == row0[h])
            cover = np.zeros(nq, np.int32)
            for w in mine:
                assert w["q0"] // F == (w["q0"] + w["nq"] - 1) // F   # one frame each
                cover[w["q0"]:w["q0"] + w["nq"]] += 1
            assert np.all(cover == 1), (h, a)

    # Longest-first deal: the busiest CTA exceeds the mean by less than the
    # largest item (list scheduling's bound), in key-tile steps.
    if not sliding and len(items):
        tiles = -(-items["k_len"] // KEY_TILE)
        biggest = int((-(-tiles // items["n_chunks"])).max()) + 7
        assert info["planned_span"] <= info["planned_total"] / CTAS + biggest
        assert info["planned_span"] * CTAS >= info["planned_total"]
    return items, info


@pytest.mark.parametrize("name", list(synth.SHAPES))
def test_plan_of_each_layer(name):
    shape = synth.SHAPES[name]
    check_plan(hc.config_for(shape), shape.mix)


@pytest.mark.parametrize("arch", [0, 1, 2, 3])
@pytest.mark.parametrize("name", ["480p", "720p"])
def test_plan_of_single_archetype_layers(name, arch):
    shape = synth.SHAPES[name]
    check_plan(hc.config_for(shape), [arch] * shape.n_heads)


@pytest.mark.parametrize("name", ["480p", "720p"])
def test_plan_of_sliding_spatial_layers(name):
    shape = synth.SHAPES[name]
    items, _ = check_plan(hc.config_for(shape, spatial_mode=hc.HC_SPATIAL_SLIDING), shape.mix)
    assert np.sum(items["launch"] == 1) > 0


def test_plan_items_reports_count_and_short_buffers(lib):
    import ctypes as C
    shape = synth.SHAPES["720p"]
    cfg = hc.config_for(shape)
    lab = np.asarray(shape.mix, np.int8)
    n = C.c_int32(-1)
    assert lib.hc_cache_plan_items(C.byref(cfg), lab.ctypes.data_as(C.c_void_p), None, 0, C.byref(n)) == 0
    assert n.value == hc.hc_cache_plan_info(cfg, shape.mix)["n_work_items"]
    short = np.full(n.value - 1, -7, hc.WORK_ITEM_DTYPE)
    status = lib.hc_cache_plan_items(C.byref(cfg), lab.ctypes.data_as(C.c_void_p),
                                     short.ctypes.data_as(C.c_void_p), n.value - 1, C.byref(n))
    assert hc.STATUS_NAMES[status] == "HC_ERR_SIZE"
    assert np.all(short["head"] == -7) and np.all(short["cta"] == -7)   # nothing written
    assert lib.hc_cache_plan_items(C.byref(cfg), lab.ctypes.data_as(C.c_void_p), None, 0, None) == 1
    bad = np.asarray([0, 1, 2, 5] + [0] * 8, np.int8)
    assert lib.hc_cache_plan_items(C.byref(cfg), bad.ctypes.data_as(C.c_void_p), None, 0, C.byref(n)) == 1


@st.composite
def layers(draw):
    fpb = draw(st.integers(1, 4))
    cfg = hc.make_config(draw(st.integers(1, 12)), draw(st.sampled_from([64, 128])),
                         draw(st.integers(1, 40)), draw(st.integers(1, 40)),
                         fpb * draw(st.integers(1, 8)), draw(st.sampled_from(["bf16", "fp32"])), fpb,
                         cell_h=draw(st.integers(1, 12)), cell_w=draw(st.integers(1, 12)),
                         spatial_mode=draw(st.sampled_from([hc.HC_SPATIAL_CELLS, hc.HC_SPATIAL_SLIDING])))
    labels = draw(st.lists(st.integers(0, 3), min_size=cfg.n_heads, max_size=cfg.n_heads))
    return cfg, labels


@settings(max_examples=120, deadline=None, suppress_health_check=[HealthCheck.too_slow])
@given(layers())
def test_plan_of_random_layers(layer):
    cfg, labels = layer
    try:
        items, _ = check_plan(cfg, labels)
    except hc.HeadcastError as e:
        # The only refusal: a sliding window wider than the band kernel takes.
        assert e.name == "HC_ERR_UNSUPPORTED" and cfg.spatial_mode == hc.HC_SPATIAL_SLIDING
