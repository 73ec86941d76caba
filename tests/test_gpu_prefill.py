"""Prefill on the GPU (tcgen05 kernel through the C ABI) against the float64 oracle."""
import numpy as np
import pytest
import torch

import gqa_head_gated_gb300 as G
import oracle
from synth import inputs as S
from tests.parity import assert_parity, errors, fails_parity, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run(x, gate=True, lse=False):
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    r = G.prefill(q, k, v, g if gate else None, kv_offset=x.kv_offset, return_lse=lse)
    assert G.last_device_status() == 0
    return r


def ref(x, gate=True):
    return oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g) if gate else None,
                          kv_offset=x.kv_offset)


def test_tiny_prefill_workload():
    x = S.tiny_prefill()
    out, lse = run(x, lse=True)
    r_out, r_lse = ref(x)
    assert_parity(out, r_out, "tiny prefill")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)


CASES = [
    # B, Hq, Hkv, Lq, Lkv, kv_offset
    (1, 1, 1, 1, 1, 0),
    (1, 2, 2, 37, 37, 0),
    (1, 4, 4, 129, 129, 0),         # GQA 1: 128 rows per tile, ragged tail
    (2, 8, 4, 200, 200, 0),         # GQA 2
    (1, 24, 4, 300, 300, 0),        # GQA 6: 21 rows x 6 heads per tile (2 padding rows)
    (1, 16, 2, 257, 400, 143),      # GQA 8 with an offset
    (2, 24, 2, 45, 300, 255),       # GQA 12 (10 rows per tile)
    (1, 32, 1, 70, 100, 30),        # GQA 32 (4 rows per tile)
    (1, 128, 1, 5, 9, 3),           # GQA 128 (1 row per tile)
    (1, 8, 8, 640, 1000, 360),      # several K/V tiles, ragged everywhere
    (2, 15, 3, 100, 100, 0),        # GQA 5: 25 rows x 5 heads = 125 packed rows per tile
    (1, 21, 3, 77, 160, 83),        # GQA 7: 18 rows x 7 heads = 126, with an offset
]


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lkv,off", CASES)
def test_prefill_shapes(B, Hq, Hkv, Lq, Lkv, off):
    x = S.make_prefill(B, Hq, Hkv, Lq, Lkv=Lkv, kv_offset=off, seed=100 + Lq)
    out, lse = run(x, lse=True)
    r_out, r_lse = ref(x)
    assert_parity(out, r_out, f"prefill {B,Hq,Hkv,Lq,Lkv,off}")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)


def test_prefill_ungated():
    x = S.make_prefill(1, 12, 2, 150, seed=5)
    out = run(x, gate=False)
    assert_parity(out, ref(x, gate=False)[0], "ungated")


def test_prefill_gate_precision_outliers():
    """Score outliers (1% of keys x8) and large gates."""
    x = S.make_prefill(1, 8, 2, 384, seed=6, outlier_frac=0.01, g_std=6.0)
    assert_parity(run(x), ref(x)[0], "outliers")


def test_never_seen_keys_are_never_read():
    """Keys past kv_offset + Lq - 1 (no row sees them) may hold NaN / Inf: the output
    is bit-identical."""
    x = S.make_prefill(1, 8, 2, 100, Lkv=300, kv_offset=50, seed=7)
    a = run(x)
    x.k[:, :, 150:] = float("nan")
    x.v[:, :, 150:] = float("inf")
    b = run(x)
    assert torch.equal(a, b)


def test_masked_future_keys_bit_exact():
    """Perturbing keys a row does not see (but later rows do) leaves that row bit for
    bit unchanged."""
    x = S.make_prefill(1, 24, 4, 256, seed=8)
    a = run(x)
    x.k[:, :, 200:] = (x.k[:, :, 200:].float() * -3 + 1).to(torch.bfloat16)
    x.v[:, :, 200:] = (x.v[:, :, 200:].float() * 5).to(torch.bfloat16)
    b = run(x)
    assert torch.equal(a[:, :, :200], b[:, :, :200])
    assert not torch.equal(a[:, :, 200:], b[:, :, 200:])


def test_chunked_equals_whole():
    """A prompt run in chunks with kv_offset equals the whole-prompt run bit for bit: a
    row's arithmetic depends on its own scores and on the key tiles from key 0, not on
    which row tile or CTA computes it (other rows' lazy rescales multiply it by exactly
    1, and the keys it does not see add exact zeros)."""
    x = S.make_prefill(1, 16, 2, 700, seed=9)
    whole = run(x)
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    parts = []
    for c0, c1 in [(0, 128), (128, 129), (129, 512), (512, 700)]:
        parts.append(G.prefill(q[:, :, c0:c1].contiguous(), k[:, :, :c1].contiguous(),
                               v[:, :, :c1].contiguous(), g[:, :, c0:c1].contiguous(), kv_offset=c0))
    chunked = torch.cat(parts, dim=2)
    assert torch.equal(chunked, whole), errors(chunked, whole.float())


def test_one_key_too_far_control():
    """Control: the oracle with one extra visible key per row must fail parity against
    the GPU output (the checker can see a masking error)."""
    x = S.make_prefill(1, 8, 2, 64, Lkv=72, seed=10)    # a spare key past the prompt
    out = run(x)
    orig = oracle.attention.prefill_visible
    try:
        oracle.attention.prefill_visible = lambda i, off: off + i + 2
        bad = ref(x)[0]
    finally:
        oracle.attention.prefill_visible = orig
    assert fails_parity(out, bad)


def test_lost_tile_edge_control():
    """Control: an oracle that drops the last partial key tile (keys past a multiple
    of 128) must fail parity on a ragged prompt."""
    x = S.make_prefill(1, 4, 2, 200, seed=11)
    out = run(x)
    orig = oracle.attention.prefill_visible
    try:
        oracle.attention.prefill_visible = lambda i, off: min(off + i + 1, 128)
        bad = ref(x)[0]
    finally:
        oracle.attention.prefill_visible = orig
    assert fails_parity(out, bad)


def test_empty_prompt_is_noop():
    q = torch.empty(1, 4, 0, 256, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(1, 2, 4, 256, dtype=torch.bfloat16, device=DEV)
    out = G.prefill(q, k, k, q, kv_offset=4)
    assert out.shape == (1, 4, 0, 256)


def _sampled_rows(Hq, Lq, n, seed):
    rng = np.random.default_rng(seed)
    rows = set()
    for h in range(Hq):
        rows.add((0, h, Lq - 1))
        rows.add((0, h, 0))
    while len(rows) < min(n, Hq * Lq):
        rows.add((0, int(rng.integers(Hq)), int(rng.integers(Lq))))
    return sorted(rows)


@pytest.mark.parametrize("name", ["prefill_27b", "chunked_prefill_35b"])
def test_full_size_workloads_sampled(name):
    """The 8192-row and the 2048-row-at-offset-30720 workloads at full size, in the
    bench's launch configuration, checked on sampled rows the oracle computes one by one
    (every head's first and last row plus random rows)."""
    x = S.WORKLOADS[name]()
    out, lse = run(x, lse=True)
    assert torch.isfinite(out).all()
    B, Hq, Lq, _ = x.q.shape
    rows = _sampled_rows(Hq, Lq, 160, 1)
    r_out, r_lse = oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g),
                                  kv_offset=x.kv_offset, rows=rows)
    got = torch.stack([out[b, h, i] for b, h, i in rows])
    assert_parity(got, r_out, name)
    got_lse = np.array([float(lse[b, h, i]) for b, h, i in rows])
    np.testing.assert_allclose(got_lse, r_lse, rtol=0, atol=2e-3)


def _random_shapes(n, seed):
    """Seeded random prefill shapes: batch 1-2, 1-4 KV heads, GQA 1-12 (the third
    page's 24 / 2 model among them), prompt 1-300 rows at an offset of 0-200."""
    rng = np.random.default_rng(seed)
    shapes = [(1, 24, 2, 97, 97 + 61, 61)]                 # GQA 12, 24 / 2 heads
    while len(shapes) < n:
        B = int(rng.integers(1, 3))
        Hkv = int(rng.integers(1, 5))
        gqa = int(rng.integers(1, 13))
        Lq = int(rng.integers(1, 301))
        off = int(rng.integers(0, 201))
        shapes.append((B, Hkv * gqa, Hkv, Lq, Lq + off, off))
    return shapes


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lkv,off", _random_shapes(10, 2024))
def test_prefill_random_shapes(B, Hq, Hkv, Lq, Lkv, off):
    x = S.make_prefill(B, Hq, Hkv, Lq, Lkv=Lkv, kv_offset=off, seed=Lq * 7 + Hq)
    out, lse = run(x, lse=True)
    r_out, r_lse = ref(x)
    assert_parity(out, r_out, f"prefill random {B,Hq,Hkv,Lq,Lkv,off}")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)
