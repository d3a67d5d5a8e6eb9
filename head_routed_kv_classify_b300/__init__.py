"""Python binding of libheadcast.so (head-routed attention for AR video DiTs).

Argument marshalling only: every step of classification, cache maintenance
and attention runs in the library's CUDA kernels.  PyTorch supplies device
memory and streams; tensors are passed by ``data_ptr()``.  There is no CPU
fallback: if the shared library is missing, importing the compute functions
raises ``HeadcastUnavailable``.

Names mirror the C ABI in include/headcast.h:
    hc_config_default, hc_config_validate, hc_classify_scratch_bytes,
    hc_classify, hc_cache_bytes, hc_cache_create (-> Cache),
    hc_cache_restructure, hc_cache_append, hc_routed_attention,
    hc_full_attention, hc_get_last_error, hc_classify_static_scratch

Host-side helpers (no device work): memory_report (steady-state cache bytes
against the monolithic window), save_labels / load_labels (per-layer
archetype labels as text).
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libheadcast.so")

SINK, DUMMY, SPATIAL, GLOBAL = 0, 1, 2, 3
ARCHETYPES = ("sink", "dummy", "spatial", "global")
HC_BF16, HC_FP32 = 0, 1
HC_PROXY_NEIGHBOURHOOD, HC_PROXY_CELL = 0, 1
HC_SPATIAL_CELLS, HC_SPATIAL_SLIDING = 0, 1
STATUS_NAMES = {0: "HC_OK", 1: "HC_ERR_INVALID_ARG", 2: "HC_ERR_SHAPE", 3: "HC_ERR_DTYPE",
                4: "HC_ERR_ALIGN", 5: "HC_ERR_STATE", 6: "HC_ERR_CUDA", 7: "HC_ERR_TIMEOUT",
                8: "HC_ERR_UNSUPPORTED", 9: "HC_ERR_SIZE"}
MAX_HEADS = 64
ABI_VERSION = 7                   # HC_ABI_VERSION this binding is written against
STATIC_SCRATCH_BYTES = 16 << 20   # HC_STATIC_SCRATCH_BYTES

# Every symbol include/headcast.h declares.
EXPORTS = ("hc_abi_version", "hc_status_string", "hc_last_error_message", "hc_config_default",
           "hc_config_validate", "hc_classify_scratch_bytes", "hc_classify", "hc_cache_bytes",
           "hc_cache_create", "hc_cache_destroy", "hc_cache_get_info", "hc_cache_restructure",
           "hc_cache_append", "hc_routed_attention", "hc_full_attention", "hc_get_last_error",
           "hc_classify_static_scratch", "hc_debug_inject_stall", "hc_cache_plan_info",
           "hc_full_attention_ws_bytes", "hc_full_attention_ws", "hc_cache_plan_items")


class HeadcastUnavailable(RuntimeError):
    pass


class HeadcastError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{self.name}: {message}")


class HcConfig(C.Structure):
    _fields_ = [("n_heads", C.c_int32), ("head_dim", C.c_int32), ("frame_h", C.c_int32),
                ("frame_w", C.c_int32), ("frames_per_block", C.c_int32),
                ("window_frames", C.c_int32), ("dtype", C.c_int32), ("softmax_scale", C.c_float),
                ("theta_sink", C.c_float), ("theta_dummy", C.c_float),
                ("theta_spatial", C.c_float), ("theta_score", C.c_float), ("gamma", C.c_float),
                ("proxy_radius", C.c_int32), ("cell_h", C.c_int32), ("cell_w", C.c_int32),
                ("proxy_mode", C.c_int32), ("spatial_mode", C.c_int32)]

    @property
    def F(self):
        return self.frame_h * self.frame_w

    @property
    def block_tokens(self):
        return self.frames_per_block * self.F


class HcCacheInfo(C.Structure):
    _fields_ = [("newest_block", C.c_int64), ("valid_frames", C.c_int32),
                ("sink_present", C.c_int32), ("n_by_archetype", C.c_int32 * 4),
                ("rows_by_archetype", C.c_int64 * 4), ("bytes", C.c_size_t),
                ("kv_bytes", C.c_size_t), ("split_bytes", C.c_size_t),
                ("monolithic_bytes", C.c_size_t), ("n_work_items", C.c_int32),
                ("n_split_runs", C.c_int32), ("n_split_pieces", C.c_int32), ("pad_", C.c_int32),
                ("planned_span", C.c_int64), ("planned_total", C.c_int64)]

    def as_dict(self) -> dict:
        return dict(newest_block=self.newest_block, valid_frames=self.valid_frames,
                    sink_present=bool(self.sink_present),
                    n_by_archetype=list(self.n_by_archetype),
                    rows_by_archetype=list(self.rows_by_archetype), bytes=self.bytes,
                    kv_bytes=self.kv_bytes, split_bytes=self.split_bytes,
                    monolithic_bytes=self.monolithic_bytes, n_work_items=self.n_work_items,
                    n_split_runs=self.n_split_runs, n_split_pieces=self.n_split_pieces,
                    planned_span=self.planned_span, planned_total=self.planned_total)


# hc_work_item, field for field (56 bytes, 8-byte aligned).
WORK_ITEM_DTYPE = np.dtype([("head", np.int32), ("kind", np.int32), ("q0", np.int32), ("nq", np.int32),
                            ("k_row0", np.int64), ("k_len", np.int64), ("cell", np.int32),
                            ("chunk", np.int32), ("n_chunks", np.int32), ("part", np.int32),
                            ("launch", np.int32), ("cta", np.int32)], align=True)
HC_ITEM_RANGE, HC_ITEM_CELL, HC_ITEM_BAND, HC_ITEM_PATCH = 0, 1, 3, 4

_lib = None


def load(path: str = LIB_PATH):
    """Load the shared library (no GPU needed) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise HeadcastUnavailable(f"{path} is not built; run head_routed_kv_classify_b300.build")
    lib = C.CDLL(path)
    vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    cfgp = C.POINTER(HcConfig)
    sig = {
        "hc_abi_version": (i32, []),
        "hc_status_string": (C.c_char_p, [C.c_int]),
        "hc_last_error_message": (C.c_char_p, []),
        "hc_config_default": (C.c_int, [cfgp]),
        "hc_config_validate": (C.c_int, [cfgp]),
        "hc_classify_scratch_bytes": (C.c_int, [cfgp, i32, C.POINTER(sz)]),
        "hc_classify": (C.c_int, [cfgp, vp, vp, vp, i32, vp, vp, vp, vp, vp, sz, vp]),
        "hc_cache_bytes": (C.c_int, [cfgp, vp, C.POINTER(sz)]),
        "hc_cache_create": (C.c_int, [cfgp, vp, vp, sz, C.POINTER(vp)]),
        "hc_cache_destroy": (C.c_int, [vp]),
        "hc_cache_get_info": (C.c_int, [vp, C.POINTER(HcCacheInfo)]),
        "hc_cache_plan_info": (C.c_int, [cfgp, vp, C.POINTER(HcCacheInfo)]),
        "hc_cache_restructure": (C.c_int, [vp, vp, vp, i64, i32, vp]),
        "hc_cache_append": (C.c_int, [vp, i64, vp, vp, vp]),
        "hc_routed_attention": (C.c_int, [vp, vp, vp, vp]),
        "hc_full_attention": (C.c_int, [cfgp, vp, vp, vp, i32, i32, vp, vp]),
        "hc_get_last_error": (C.c_int, [vp]),
        "hc_classify_static_scratch": (C.c_int, [cfgp, vp, vp, vp, i32, vp, vp, vp, vp, vp]),
        "hc_debug_inject_stall": (C.c_int, [i32]),
        "hc_full_attention_ws_bytes": (C.c_int, [cfgp, i32, i32, C.POINTER(sz)]),
        "hc_full_attention_ws": (C.c_int, [cfgp, vp, vp, vp, i32, i32, vp, vp, sz, vp]),
        "hc_cache_plan_items": (C.c_int, [cfgp, vp, vp, i32, C.POINTER(i32)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.hc_abi_version() != ABI_VERSION:
        raise HeadcastUnavailable(f"{path} has ABI {lib.hc_abi_version()}, binding expects {ABI_VERSION}")
    _lib = lib
    return lib


def _check(status):
    if status != 0:
        msg = load().hc_last_error_message().decode(errors="replace")
        raise HeadcastError(status, msg)


# ----------------------------------------------------------------- config

def hc_config_default() -> HcConfig:
    cfg = HcConfig()
    _check(load().hc_config_default(C.byref(cfg)))
    return cfg


def make_config(n_heads, head_dim, frame_h, frame_w, window_frames=21, dtype="bf16",
                frames_per_block=3, **overrides) -> HcConfig:
    cfg = hc_config_default()
    cfg.n_heads, cfg.head_dim, cfg.frame_h, cfg.frame_w = n_heads, head_dim, frame_h, frame_w
    cfg.window_frames, cfg.frames_per_block = window_frames, frames_per_block
    cfg.dtype = {"bf16": HC_BF16, "fp32": HC_FP32}[dtype] if isinstance(dtype, str) else int(dtype)
    for k, v in overrides.items():
        setattr(cfg, k, v)
    return cfg


def config_for(shape, **overrides) -> HcConfig:
    """Config from any object with the synthetic-layer fields."""
    return make_config(shape.n_heads, shape.head_dim, shape.frame_h, shape.frame_w,
                       shape.window_frames, shape.dtype, shape.frames_per_block, **overrides)


def hc_config_validate(cfg: HcConfig):
    _check(load().hc_config_validate(C.byref(cfg)))


# ----------------------------------------------------------------- helpers

def _torch():
    import torch
    return torch


def _stream(stream):
    if stream is None:
        return C.c_void_p(_torch().cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return C.c_void_p(stream)
    return C.c_void_p(stream.cuda_stream)


def _dtype_of(cfg):
    t = _torch()
    return t.bfloat16 if cfg.dtype == HC_BF16 else t.float32


def _ptr(t, cfg=None, name="tensor", shape=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if cfg is not None and t.dtype != _dtype_of(cfg):
        raise ValueError(f"{name} has dtype {t.dtype}, config wants {_dtype_of(cfg)}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return C.c_void_p(t.data_ptr())


# ----------------------------------------------------------------- classification

def hc_classify_scratch_bytes(cfg, n_key_frames=None) -> int:
    n = C.c_size_t(0)
    nkf = cfg.window_frames if n_key_frames is None else n_key_frames
    _check(load().hc_classify_scratch_bytes(C.byref(cfg), nkf, C.byref(n)))
    return n.value


def hc_classify(cfg, q, k, v, n_key_frames=None, labels_dev=None, stats_dev=None, o_full=None,
                scratch=None, stream=None, copy_labels=True):
    """Classify every head.  Returns (labels_host int8[H] or None, labels_dev,
    stats_dev [H][6]: c_sink, c_dummy, c_spatial, P5, MSE, score)."""
    t = _torch()
    nkf = cfg.window_frames if n_key_frames is None else n_key_frames
    H, d = cfg.n_heads, cfg.head_dim
    dev = q.device
    if labels_dev is None:
        labels_dev = t.empty(H, dtype=t.int8, device=dev)
    if stats_dev is None:
        stats_dev = t.empty((H, 6), dtype=t.float32, device=dev)
    nbytes = hc_classify_scratch_bytes(cfg, nkf)
    if scratch is None:
        scratch = t.empty(nbytes, dtype=t.uint8, device=dev)
    host = np.zeros(H, dtype=np.int8) if copy_labels else None
    _check(load().hc_classify(
        C.byref(cfg), _ptr(q, cfg, "q", (cfg.block_tokens, H, d)),
        _ptr(k, cfg, "k", (nkf * cfg.F, H, d)), _ptr(v, cfg, "v", (nkf * cfg.F, H, d)), nkf,
        _ptr(labels_dev, None, "labels_dev"),
        host.ctypes.data_as(C.c_void_p) if host is not None else None,
        _ptr(stats_dev, None, "stats_dev"), _ptr(o_full, cfg, "o_full"),
        _ptr(scratch, None, "scratch"), scratch.numel() * scratch.element_size(), _stream(stream)))
    return host, labels_dev, stats_dev


def hc_classify_static_scratch(cfg, q, k, v, n_key_frames=None, labels_dev=None, stats_dev=None,
                               o_full=None, stream=None, copy_labels=True):
    """hc_classify for callers that cannot allocate device memory: the
    library supplies the workspace from a fixed device array (at most
    STATIC_SCRATCH_BYTES).  labels_dev and stats_dev must then be passed in
    by such a caller; they are only created here when omitted.  Returns
    (labels_host int8[H] or None, labels_dev, stats_dev)."""
    t = _torch()
    nkf = cfg.window_frames if n_key_frames is None else n_key_frames
    H, d = cfg.n_heads, cfg.head_dim
    dev = q.device
    if labels_dev is None:
        labels_dev = t.empty(H, dtype=t.int8, device=dev)
    if stats_dev is None:
        stats_dev = t.empty((H, 6), dtype=t.float32, device=dev)
    host = np.zeros(H, dtype=np.int8) if copy_labels else None
    _check(load().hc_classify_static_scratch(
        C.byref(cfg), _ptr(q, cfg, "q", (cfg.block_tokens, H, d)),
        _ptr(k, cfg, "k", (nkf * cfg.F, H, d)), _ptr(v, cfg, "v", (nkf * cfg.F, H, d)), nkf,
        _ptr(labels_dev, None, "labels_dev"),
        host.ctypes.data_as(C.c_void_p) if host is not None else None,
        _ptr(stats_dev, None, "stats_dev"), _ptr(o_full, cfg, "o_full"), _stream(stream)))
    return host, labels_dev, stats_dev


# ----------------------------------------------------------------- cache

def hc_cache_bytes(cfg, labels) -> int:
    lab = np.ascontiguousarray(np.asarray(labels, dtype=np.int8))
    n = C.c_size_t(0)
    _check(load().hc_cache_bytes(C.byref(cfg), lab.ctypes.data_as(C.c_void_p), C.byref(n)))
    return n.value


class Cache:
    """A restructured per-archetype cache: the library's handle plus the
    caller-owned backing buffer (a torch uint8 tensor)."""

    def __init__(self, cfg, labels, device=None, buf=None):
        t = _torch()
        self.cfg = cfg
        self.labels = np.ascontiguousarray(np.asarray(labels, dtype=np.int8))
        self.nbytes = hc_cache_bytes(cfg, self.labels)
        if buf is None:
            buf = t.empty(self.nbytes + 256, dtype=t.uint8, device=device or "cuda")
        base = buf.data_ptr()
        self._buf = buf
        self._off = (-base) % 256
        handle = C.c_void_p(0)
        _check(load().hc_cache_create(C.byref(cfg), self.labels.ctypes.data_as(C.c_void_p),
                                      C.c_void_p(base + self._off),
                                      buf.numel() - self._off, C.byref(handle)))
        self.handle = handle

    def close(self):
        if self.handle:
            load().hc_cache_destroy(self.handle)
            self.handle = C.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def info(self) -> dict:
        inf = HcCacheInfo()
        _check(load().hc_cache_get_info(self.handle, C.byref(inf)))
        return inf.as_dict()

    def restructure(self, k_win, v_win, first_block_id=0, n_blocks=None, stream=None):
        cfg = self.cfg
        nb = k_win.shape[0] // cfg.block_tokens if n_blocks is None else n_blocks
        shape = (nb * cfg.block_tokens, cfg.n_heads, cfg.head_dim)
        _check(load().hc_cache_restructure(self.handle, _ptr(k_win, cfg, "k_win", shape),
                                           _ptr(v_win, cfg, "v_win", shape), first_block_id, nb,
                                           _stream(stream)))

    def append(self, block_id, k_blk, v_blk, stream=None):
        cfg = self.cfg
        shape = (cfg.block_tokens, cfg.n_heads, cfg.head_dim)
        _check(load().hc_cache_append(self.handle, block_id, _ptr(k_blk, cfg, "k_blk", shape),
                                      _ptr(v_blk, cfg, "v_blk", shape), _stream(stream)))

    def routed_attention(self, q, o=None, stream=None):
        cfg = self.cfg
        shape = (cfg.block_tokens, cfg.n_heads, cfg.head_dim)
        if o is None:
            o = _torch().empty(shape, dtype=_dtype_of(cfg), device=q.device)
        _check(load().hc_routed_attention(self.handle, _ptr(q, cfg, "q", shape),
                                          _ptr(o, cfg, "o", shape), _stream(stream)))
        return o


def hc_cache_create(cfg, labels, device=None, buf=None) -> Cache:
    return Cache(cfg, labels, device, buf)


def hc_routed_attention(cache: Cache, q, o=None, stream=None):
    return cache.routed_attention(q, o, stream)


def hc_full_attention_ws_bytes(cfg, n_q_tokens, n_key_frames) -> int:
    n = C.c_size_t(0)
    _check(load().hc_full_attention_ws_bytes(C.byref(cfg), n_q_tokens, n_key_frames, C.byref(n)))
    return n.value


def hc_full_attention(cfg, q, k, v, o=None, n_key_frames=None, stream=None, scratch=None, balanced=True):
    """Full attention of every head over the key window.  bf16 layers use the
    balanced schedule (hc_full_attention_ws; `scratch` is created when
    omitted) unless balanced=False, which calls hc_full_attention."""
    nkf = k.shape[0] // cfg.F if n_key_frames is None else n_key_frames
    H, d = cfg.n_heads, cfg.head_dim
    nq = q.shape[0]
    if o is None:
        o = _torch().empty((nq, H, d), dtype=_dtype_of(cfg), device=q.device)
    args = (C.byref(cfg), _ptr(q, cfg, "q", (nq, H, d)), _ptr(k, cfg, "k", (nkf * cfg.F, H, d)),
            _ptr(v, cfg, "v", (nkf * cfg.F, H, d)), nq, nkf, _ptr(o, cfg, "o", (nq, H, d)))
    if balanced and cfg.dtype == HC_BF16 and nq > 0:
        nbytes = hc_full_attention_ws_bytes(cfg, nq, nkf)
        if scratch is None:
            scratch = _torch().empty(max(nbytes, 256), dtype=_torch().uint8, device=q.device)
        _check(load().hc_full_attention_ws(*args, _ptr(scratch, None, "scratch"),
                                           scratch.numel() * scratch.element_size(), _stream(stream)))
    else:
        _check(load().hc_full_attention(*args, _stream(stream)))
    return o


def hc_debug_inject_stall(enable: bool):
    """Test hook: while enabled, tensor-core attention launches stall their
    K/V producer after one tile so that the bounded device waits expire and
    hc_get_last_error reports HC_ERR_TIMEOUT (outputs undefined)."""
    _check(load().hc_debug_inject_stall(1 if enable else 0))


def hc_get_last_error(stream=None):
    _check(load().hc_get_last_error(_stream(stream)))


# ----------------------------------------------------------------- host-side helpers

def hc_cache_plan_info(cfg, labels) -> dict:
    """What hc_cache_create would reserve for these labels (host only)."""
    lab = np.ascontiguousarray(np.asarray(labels, dtype=np.int8))
    inf = HcCacheInfo()
    _check(load().hc_cache_plan_info(C.byref(cfg), lab.ctypes.data_as(C.c_void_p), C.byref(inf)))
    return inf.as_dict()


def hc_cache_plan_items(cfg, labels) -> np.ndarray:
    """The routed work list hc_cache_create would write for these labels
    (host only), in launch order, as a structured array of WORK_ITEM_DTYPE."""
    lab = np.ascontiguousarray(np.asarray(labels, dtype=np.int8))
    lib, n = load(), C.c_int32(0)
    _check(lib.hc_cache_plan_items(C.byref(cfg), lab.ctypes.data_as(C.c_void_p), None, 0, C.byref(n)))
    out = np.zeros(n.value, WORK_ITEM_DTYPE)
    _check(lib.hc_cache_plan_items(C.byref(cfg), lab.ctypes.data_as(C.c_void_p),
                                   out.ctypes.data_as(C.c_void_p), n.value, C.byref(n)))
    return out


def memory_report(cfg, labels) -> dict:
    """Steady-state KV-cache footprint of one layer for these labels against
    the monolithic [window][H][d] K/V cache, as the library plans it
    (hc_cache_plan_info, host only).  `ratio` compares the K/V regions with
    the monolithic cache; `bytes` is the whole backing store (K/V regions,
    work list and schedule, and the split-run workspace).
    [Pith review of HeadCast, Figure 9 caption / Appendix C: memory of the
    restructured cache.]"""
    info = hc_cache_plan_info(cfg, labels)
    rows = {ARCHETYPES[a]: int(info["rows_by_archetype"][a]) for a in range(4)}
    return {"bytes": info["bytes"], "kv_bytes": info["kv_bytes"], "split_bytes": info["split_bytes"],
            "monolithic_bytes": info["monolithic_bytes"],
            "ratio": info["kv_bytes"] / info["monolithic_bytes"], "rows_by_archetype": rows}


_LETTERS = "SDPG"


def save_labels(path, labels):
    """Write per-layer archetype labels ([layers][heads] ints 0..3) as text:
    a comment line, then one line per layer: the layer index and one letter
    per head (S Sink, D Dummy, P Spatial, G Global)."""
    lab = np.atleast_2d(np.asarray(labels, dtype=np.int64))
    if lab.size == 0 or lab.min() < 0 or lab.max() > 3:
        raise ValueError("labels must be archetypes 0..3")
    with open(path, "w") as f:
        f.write(f"# headcast head archetypes: {lab.shape[0]} layers x {lab.shape[1]} heads; "
                "S=Sink D=Dummy P=Spatial G=Global\n")
        for layer, row in enumerate(lab):
            f.write(f"{layer} {''.join(_LETTERS[int(a)] for a in row)}\n")


def load_labels(path) -> np.ndarray:
    """Read labels written by save_labels: int8 [layers][heads].  Raises
    ValueError on a malformed file (unknown letter, ragged rows, layers out
    of order or missing)."""
    rows = []
    with open(path) as f:
        for n, line in enumerate(f, 1):
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if len(parts) != 2 or not parts[0].isdigit():
                raise ValueError(f"{path}:{n}: expected '<layer> <letters>'")
            if int(parts[0]) != len(rows):
                raise ValueError(f"{path}:{n}: layer {parts[0]} out of order (expected {len(rows)})")
            if any(c not in _LETTERS for c in parts[1]):
                raise ValueError(f"{path}:{n}: unknown archetype letter in {parts[1]!r}")
            if rows and len(parts[1]) != len(rows[0]):
                raise ValueError(f"{path}:{n}: {len(parts[1])} heads, earlier layers have {len(rows[0])}")
            rows.append([_LETTERS.index(c) for c in parts[1]])
    if not rows:
        raise ValueError(f"{path}: no layers")
    return np.array(rows, dtype=np.int8)
