"""Parity measures between a bf16 / fp16 CUDA result and the float64 oracle.

Acceptance (the stated tolerance for bf16 outputs):
  * max |gpu - ref| <= 2e-2 (absolute, over all elements);
  * median of |gpu - ref| / max(|ref|, 1e-6) <= 4e-3;
  * no NaN / Inf where the oracle is finite.

fp16 outputs must meet that bar and a tighter one derived from fp16's unit
roundoff u = 2^-11 (the stated tolerance is for bf16 only):
  * the output rounding costs at most half an ulp, <= 2^-10 for |out| < 4
    (outputs are convex combinations of N(0,1) values times a gate in (0, 1));
  * P enters the P.V product rounded to fp16 (relative error <= u each), which
    moves an output by at most u * sum_j p_j |V_j| / l <= u * max|V| ~ 2.4e-3
    for N(0,1) values (|V| < 5);
  * scores, sums and accumulation are fp32 (errors near 2^-24, negligible);
  so max |err| <= 5e-3 (FP16_MAX_ABS), and the median relative error, which
  the output rounding dominates (<= u), is held to 1e-3 (FP16_MEDIAN_REL).
"""
import numpy as np
import torch

MAX_ABS = 2e-2
MEDIAN_REL = 4e-3
FP16_MAX_ABS = 5e-3
FP16_MEDIAN_REL = 1e-3


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


def assert_parity_dtype(gpu, ref, what=""):
    """assert_parity at the stated bar, plus the fp16 bar for fp16 results."""
    e = assert_parity(gpu, ref, what)
    if isinstance(gpu, torch.Tensor) and gpu.dtype == torch.float16:
        e = assert_parity(gpu, ref, what + " (fp16 bar)", FP16_MAX_ABS, FP16_MEDIAN_REL)
    return e


def assert_nonfinite_parity(gpu, ref, what="", max_abs=MAX_ABS, median_rel=MEDIAN_REL):
    """Non-finite inputs: NaN, +Inf and -Inf sit exactly where the oracle has them,
    and the finite elements meet the parity bar."""
    g = to_f64(gpu)
    r = to_f64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    for name, f in (("NaN", np.isnan), ("+Inf", lambda a: a == np.inf),
                    ("-Inf", lambda a: a == -np.inf)):
        diff = int(np.sum(f(g) != f(r)))
        assert diff == 0, f"{what}: {name} pattern differs in {diff} elements"
    fin = np.isfinite(r)
    if fin.any():
        d = np.abs(g[fin] - r[fin])
        rel = d / np.maximum(np.abs(r[fin]), 1e-6)
        assert d.max() <= max_abs, f"{what}: max|err| {d.max():.3e}"
        assert np.median(rel) <= median_rel, f"{what}: median rel {np.median(rel):.3e}"
