"""Helpers for the GPU parity tests: move seeded synthetic inputs to the
device in their storage dtype, bring outputs back, and compare with the
oracle under the stated tolerances."""
import hashlib
import json
import os

import numpy as np

import synth

# Outputs of bf16 I/O with fp32 accumulation versus the fp64 oracle.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
# fp32 I/O (tiny layer): fp32 accumulation with fp32 probabilities.
MAX_ABS_F32 = 1e-4
MEAN_ABS_F32 = 1e-5


def torch():
    import torch as t
    return t


def to_dev(x: synth.Tensor3, dtype: str):
    t = torch()
    if dtype == "bf16":
        return t.from_numpy(x.raw.view(np.int16).copy()).view(t.bfloat16).cuda()
    return t.from_numpy(np.ascontiguousarray(x.raw)).cuda()


def to_host(t_):
    t = torch()
    return t_.detach().to(t.float32).cpu().numpy().astype(np.float64)


def tolerances(dtype):
    return (MAX_ABS, MEAN_ABS) if dtype == "bf16" else (MAX_ABS_F32, MEAN_ABS_F32)


def assert_close(got, want, dtype, what=""):
    mx_tol, mean_tol = tolerances(dtype)
    err = np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err.max() <= mx_tol and err.mean() <= mean_tol, (
        f"{what}: max-abs {err.max():.3e} (tol {mx_tol}), mean-abs {err.mean():.3e} (tol {mean_tol})")
    return err.max(), err.mean()


def sample_queries(n, k, seed):
    rng = np.random.default_rng(seed)
    if k >= n:
        return np.arange(n)
    idx = rng.choice(n, size=k, replace=False)
    idx[:2] = [0, n - 1]                       # always include both ends
    return np.sort(idx)


def per_cell_row_sample(shape, seed, cell_h=10, cell_w=10):
    """Block-local query tokens: one query (seeded column) for every frame of
    the block and every frame row of every deployed cell, so that every cell
    of a Spatial head, and every row inside it, is checked."""
    rng = np.random.default_rng(seed)
    F, W = shape.frame_tokens, shape.frame_w

    def axis(n, c):
        k = max(1, int(n / c + 0.5))
        return [(i * c, c if i < k - 1 else n - c * (k - 1)) for i in range(k)]
    out = []
    for h0, hz in axis(shape.frame_h, cell_h):
        for w0, wz in axis(shape.frame_w, cell_w):
            for f in range(shape.frames_per_block):
                for hh in range(h0, h0 + hz):
                    out.append(f * F + hh * W + w0 + int(rng.integers(wz)))
    return np.array(sorted(out), dtype=np.int64)


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def input_digest(q_raw, k_raw, v_raw):
    """SHA-256 of the raw input bytes, as the golden files record them."""
    return {n: hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()
            for n, a in (("q", q_raw), ("k", k_raw), ("v", v_raw))}


# Per-head statistics of the GPU (fp32 per-token values from bf16-probability
# outputs) against the fp64 oracle: the mean cosines, P5 and the score to
# 2e-3, the MSE to 5 % + 1e-5.
STAT_ATOL = 2e-3


def assert_stats_close(got, want, what):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    for h in range(want.shape[0]):
        for j in (0, 1, 2, 3, 5):
            assert abs(got[h, j] - want[h, j]) <= STAT_ATOL, (what, h, j, got[h], want[h])
        assert abs(got[h, 4] - want[h, 4]) <= 0.05 * abs(want[h, 4]) + 1e-5, (what, h, got[h], want[h])
