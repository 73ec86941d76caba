"""Prefill at the lengths where the kernels change shape, against the float64 oracle.

  * The prefill call sends a prompt to CTA pairs once its last row sees 2048 keys or
    more (kv_offset + Lq >= 2048) and to single CTAs below that: prompts whose last
    row sees 2047, 2048 and 2049 keys, from a zero offset and from one that leaves a
    single row, land on the expected kernel and match the oracle.
  * Prompts of 8191 and 8193 rows end one key before and one key past the 64th
    128-key tile.
  Both in bf16 and in fp16 (the fp16 results also meet the fp16 bar).
  * A 3000-row prompt run in chunks whose last rows see 1024, 2047, 2048 and 3000
    keys (single CTAs for the first two, pairs for the rest) equals the whole-prompt
    run bit for bit, in bf16 and fp16, with key outliers that make rows rescale; so
    do a prompt cut into 16-row and into 32-row chunks, whose seams are those of the
    pages' prompt-row frames."""
import numpy as np
import pytest
import torch

import gqa_head_gated_gb300 as G
import oracle
from synth import inputs as S
from tests.parity import assert_parity_dtype, errors, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
SINGLE = "attn_tc_kernel<prefill,bf16>"
PAIR = "attn_pair_kernel<prefill,bf16>"
DTYPES = [torch.bfloat16, torch.float16]
IDS = ["bf16", "fp16"]


def _names(dtype):
    sfx = "fp16>" if dtype == torch.float16 else "bf16>"
    return "attn_tc_kernel<prefill," + sfx, "attn_pair_kernel<prefill," + sfx


def _rows(Hq, Lq, n, seed, extra=()):
    """Every head's first and last row, the given row indices in head 0 and the last
    head, then seeded random rows up to n."""
    rng = np.random.default_rng(seed)
    rows = {(0, h, i) for h in range(Hq) for i in (0, Lq - 1)}
    rows |= {(0, h, i) for h in (0, Hq - 1) for i in extra if 0 <= i < Lq}
    while len(rows) < min(n, Hq * Lq):
        rows.add((0, int(rng.integers(Hq)), int(rng.integers(Lq))))
    return sorted(rows)


def _check_sampled(x, out, lse, rows, what):
    r_out, r_lse = oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g),
                                  kv_offset=x.kv_offset, rows=rows)
    got = torch.stack([out[b, h, i] for b, h, i in rows])
    assert_parity_dtype(got, r_out, what)
    got_lse = np.array([float(lse[b, h, i]) for b, h, i in rows])
    np.testing.assert_allclose(got_lse, r_lse, rtol=0, atol=2e-3)


def _run(x):
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    out, lse = G.prefill(q, k, v, g, kv_offset=x.kv_offset, return_lse=True)
    torch.cuda.synchronize()
    assert G.last_device_status() == 0
    return out, lse, G.launch_log(1)[0]["kernel"]


@pytest.mark.parametrize("Lq,off", [(2047, 0), (2048, 0), (2049, 0),
                                    (1, 2046), (1, 2047), (300, 1748), (301, 1748)])
@pytest.mark.parametrize("dtype", DTYPES, ids=IDS)
def test_pair_routing_threshold(dtype, Lq, off):
    single, pair = _names(dtype)
    x = S.make_prefill(1, 8, 1, Lq, kv_offset=off, seed=Lq + off, dtype=dtype)
    out, lse, kernel = _run(x)
    assert out.dtype == dtype
    assert kernel == (pair if off + Lq >= 2048 else single), kernel
    rows = _rows(8, Lq, 48, Lq, extra=(15, 16, 31, 32, Lq - 2, Lq - 17))
    _check_sampled(x, out, lse, rows, f"Lq {Lq} at offset {off}")


@pytest.mark.parametrize("Lq", [8191, 8193])
@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (4, 4)], ids=["gqa8", "gqa1"])
@pytest.mark.parametrize("dtype", DTYPES, ids=IDS)
def test_long_prompt_key_tile_edge(dtype, Lq, Hq, Hkv):
    x = S.make_prefill(1, Hq, Hkv, Lq, seed=Lq * Hq, dtype=dtype)
    out, lse, kernel = _run(x)
    assert kernel == _names(dtype)[1], kernel
    assert torch.isfinite(out).all()
    rows = _rows(Hq, Lq, 40, Lq, extra=(127, 128, 8063, 8064, 8190, 8191, 8192))
    _check_sampled(x, out, lse, rows, f"Lq {Lq}, {Hq}/{Hkv} heads")


def _chunked(x, cuts):
    """The prompt in chunks [c0, c1) at kv_offset c0; K / V hold the whole prompt (a
    chunk's rows see keys 0..c0 + i of them).  Returns the rows and the kernels."""
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    parts, kernels = [], []
    for c0, c1 in cuts:
        parts.append(G.prefill(q[:, :, c0:c1].contiguous(), k, v, g[:, :, c0:c1].contiguous(),
                               kv_offset=c0))
        kernels.append(G.launch_log(1)[0]["kernel"])
    torch.cuda.synchronize()
    assert G.last_device_status() == 0
    return torch.cat(parts, dim=2), kernels


@pytest.mark.parametrize("dtype", DTYPES, ids=IDS)
def test_chunked_equals_whole_across_pair_threshold(dtype):
    single, pair = _names(dtype)
    x = S.make_prefill(1, 16, 2, 3000, seed=31, outlier_frac=0.01, dtype=dtype)
    whole, _, kernel = _run(x)
    assert kernel == pair, kernel
    chunked, kernels = _chunked(x, [(0, 1024), (1024, 2047), (2047, 2048), (2048, 3000)])
    assert kernels == [single, single, pair, pair], kernels
    assert torch.equal(chunked, whole), errors(chunked, whole.float())
    rows = _rows(16, 3000, 48, 31, extra=(1023, 1024, 2046, 2047, 2048))
    r_out, _ = oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g), kv_offset=0,
                              rows=rows)
    got = torch.stack([chunked[b, h, i] for b, h, i in rows])
    assert_parity_dtype(got, r_out, "chunked across the pair threshold")


@pytest.mark.parametrize("step", [16, 32])
@pytest.mark.parametrize("dtype", DTYPES, ids=IDS)
def test_prompt_row_frames_equal_whole(dtype, step):
    """A 2300-row prompt cut into frames of 16 or 32 rows (the first ones on single
    CTAs, the frames whose last row sees 2048 keys or more on CTA pairs) equals the
    whole-prompt run bit for bit."""
    single, pair = _names(dtype)
    x = S.make_prefill(1, 24, 4, 2300, seed=33, outlier_frac=0.01, dtype=dtype)
    whole, _, _ = _run(x)
    cuts = [(c, min(c + step, 2300)) for c in range(0, 2300, step)]
    chunked, kernels = _chunked(x, cuts)
    assert set(kernels) == {single, pair}, set(kernels)
    assert torch.equal(chunked, whole), errors(chunked, whole.float())
