"""Parity measures between a bf16 CUDA result and the float64 oracle.

Acceptance (the stated tolerance for bf16 outputs):
  * max |gpu - ref| <= 2e-2 (absolute, over all elements);
  * median of |gpu - ref| / max(|ref|, 1e-6) <= 4e-3;
  * no NaN / Inf where the oracle is finite.
"""
import numpy as np
import torch

MAX_ABS = 2e-2
MEDIAN_REL = 4e-3


def to_f64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def errors(gpu, ref):
    g = to_f64(gpu)
    r = to_f64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    fin = np.isfinite(r)
    bad_nonfinite = int(np.sum(~np.isfinite(g) & fin))
    d = np.abs(g[fin] - r[fin])
    rel = d / np.maximum(np.abs(r[fin]), 1e-6)
    return dict(max_abs=float(d.max()) if d.size else 0.0,
                median_rel=float(np.median(rel)) if rel.size else 0.0,
                nonfinite=bad_nonfinite)


def assert_parity(gpu, ref, what="", max_abs=MAX_ABS, median_rel=MEDIAN_REL):
    e = errors(gpu, ref)
    assert e["nonfinite"] == 0, f"{what}: {e['nonfinite']} non-finite outputs where the oracle is finite"
    assert e["max_abs"] <= max_abs, f"{what}: max|err| {e['max_abs']:.3e} > {max_abs}"
    assert e["median_rel"] <= median_rel, f"{what}: median rel {e['median_rel']:.3e} > {median_rel}"
    return e


def fails_parity(gpu, ref, max_abs=MAX_ABS, median_rel=MEDIAN_REL):
    e = errors(gpu, ref)
    return e["nonfinite"] > 0 or e["max_abs"] > max_abs or e["median_rel"] > median_rel
