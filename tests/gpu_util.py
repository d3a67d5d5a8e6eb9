"""Helpers for the GPU parity tests: move seeded synthetic inputs to the
device in their storage dtype, bring outputs back, and compare with the
oracle under the stated tolerances."""
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
