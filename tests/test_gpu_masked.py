"""General masks (gqa_attn_masked, the dense SDPA consumer of the DS4Server issue113
README) on the GPU against the float64 oracle: bool and additive (fp32, bf16, fp16)
masks of several broadcast shapes and strides, with and without the causal rule,
chunk-local masks under head chunking, and the accept / reject table of mask head
counts."""
import os

import numpy as np
import pytest
import torch

import gqa_head_gated_gb300 as G
import oracle
from synth import inputs as S
from tests.parity import assert_parity_dtype, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _inputs(B, Hq, Hkv, Lq, Lkv, seed, dtype=torch.bfloat16):
    return S.make_prefill(B, Hq, Hkv, Lq, Lkv=Lkv, kv_offset=Lkv - Lq, seed=seed, dtype=dtype)


def _run(x, mask, causal=False, kv_offset=None, chunking=True, lse=True):
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    m = None if mask is None else mask.to(DEV)
    r = G.masked(q, k, v, g, m, causal=causal, kv_offset=kv_offset, head_chunking=chunking,
                 return_lse=lse)
    assert G.last_device_status() == 0
    return r


def _ref(x, mask, causal=False, kv_offset=None, chunking=True):
    m = None
    if mask is not None:
        m = mask.numpy() if mask.dtype == torch.bool else to_f64(mask)
    return oracle.sdpa_masked(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g), m,
                              causal=causal, kv_offset=kv_offset, head_chunking=chunking)


def _check(x, mask, what, **kw):
    out, lse = _run(x, mask, **kw)
    r_out, r_lse = _ref(x, mask, **kw)
    assert_parity_dtype(out, r_out, what)
    fin = np.isfinite(r_lse)
    assert np.array_equal(np.isfinite(to_f64(lse)), fin), what
    np.testing.assert_allclose(to_f64(lse)[fin], r_lse[fin], rtol=0, atol=2e-3)
    return out, r_out


def _gen(seed):
    return torch.Generator().manual_seed(seed)


@pytest.mark.parametrize("causal", [False, True])
def test_bool_full_head_mask(causal):
    x = _inputs(2, 8, 2, 150, 300, seed=70)
    m = torch.rand(2, 8, 150, 300, generator=_gen(70)) < 0.7
    m[0, 3, 17] = False                                   # a row that keeps no key
    out, _ = _check(x, m, f"bool 4-D causal={causal}", causal=causal)
    assert torch.all(out[0, 3, 17] == 0)


def test_bool_2d_mask_document_blocks():
    """Block-diagonal (packed documents) bool mask [Lq, Lkv], broadcast over batch and
    heads, with the causal rule."""
    L = 400
    doc = torch.arange(L) // 97
    m = doc[:, None] == doc[None, :]
    x = _inputs(1, 24, 4, L, L, seed=71)
    _check(x, m, "document mask", causal=True, kv_offset=0)


@pytest.mark.parametrize("mdtype", [torch.float32, torch.bfloat16, torch.float16])
def test_additive_masks(mdtype):
    """Additive biases N(0, 2) with some -inf, as [1,1,Lq,Lkv] (fp32 / bf16 / fp16)."""
    x = _inputs(1, 16, 2, 200, 333, seed=72)
    a = torch.randn(1, 1, 200, 333, generator=_gen(72)) * 2
    a[torch.rand(1, 1, 200, 333, generator=_gen(73)) < 0.2] = float("-inf")
    _check(x, a.to(mdtype), f"additive {mdtype}")


def test_key_padding_mask_and_strided_view():
    """A per-batch key-padding mask [B,1,1,Lkv] and a non-contiguous (transposed)
    additive mask."""
    x = _inputs(2, 12, 3, 130, 260, seed=74)
    pad = torch.ones(2, 1, 1, 260, dtype=torch.bool)
    pad[0, ..., 200:] = False
    pad[1, ..., :5] = False
    _check(x, pad, "key padding")
    at = (torch.randn(260, 130, generator=_gen(75)) * 3).t()       # strides (1, 130)
    assert not at.is_contiguous()
    _check(x, at, "transposed additive")


def test_no_mask_full_attention_and_causal():
    """No mask: every key (non-causal), or the causal rule alone at an offset."""
    x = _inputs(1, 8, 8, 140, 500, seed=76)
    _check(x, None, "full attention")
    _check(x, None, "causal at offset", causal=True, kv_offset=300)


def test_all_true_causal_mask_is_prefill_bit_for_bit():
    """An all-True bool mask with the causal rule runs the same arithmetic as the
    plain prefill: the outputs are identical bit for bit."""
    x = _inputs(1, 24, 4, 300, 300, seed=77)
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    ones = torch.ones(300, 300, dtype=torch.bool, device=DEV)
    a = G.masked(q, k, v, g, ones, causal=True, kv_offset=0)
    b = G.prefill(q, k, v, g, kv_offset=0)
    assert torch.equal(a, b)


def test_chunk_local_mask():
    """4 rows x GQA 16 under head chunking: chunks of 8 heads, an 8-head mask applies
    per chunk; the same tiled to 32 heads without chunking gives the same output."""
    x = _inputs(1, 32, 2, 4, 900, seed=78)
    local = torch.rand(1, 8, 4, 900, generator=_gen(78)) < 0.6
    out, _ = _check(x, local, "chunk-local", chunking=True)
    full = torch.cat([local] * 4, dim=1)
    out2, _ = _run(x, full, chunking=False)
    assert torch.equal(out, out2)


def test_fp16_masked():
    x = _inputs(1, 16, 2, 160, 400, seed=79, dtype=torch.float16)
    a = (torch.randn(160, 400, generator=_gen(79)) * 2).to(torch.float16)
    _check(x, a, "fp16 additive", causal=True, kv_offset=240)


def _rules():
    rows = []
    for line in open(os.path.join(ROOT, "tests", "golden", "mask_head_rules.txt")):
        f = line.split("#")[0].split()
        if f:
            rows.append((int(f[0]), int(f[1]), int(f[2]), int(f[3]), f[4] == "on", f[5]))
    return rows


@pytest.mark.parametrize("rule", _rules(), ids=lambda r: "r{}g{}k{}m{}{}".format(
    r[0], r[1], r[2], r[3], "on" if r[4] else "off"))
def test_head_rule_table_through_the_kernel(rule):
    """Every row of the table: accepted masks match the oracle, refused masks raise
    GQA_ERR_INVALID_ARG (and the oracle refuses them too)."""
    rows, gqa, hkv, hm, chunking, expect = rule
    x = _inputs(1, gqa * hkv, hkv, rows, 40, seed=80 + rows + gqa + hm)
    m = torch.rand(1, hm, rows, 40, generator=_gen(hm)) < 0.7
    m[..., 0] = True
    if expect == "ok":
        _check(x, m, f"rule {rule}", chunking=chunking)
    else:
        with pytest.raises(G.GqaError) as e:
            _run(x, m, chunking=chunking)
        assert e.value.code == 1
        with pytest.raises(ValueError):
            _ref(x, m, chunking=chunking)


def test_masked_keys_with_nonfinite_k_are_ignored():
    """K rows excluded by a bool mask may hold NaN / Inf: the output is unchanged bit
    for bit (the kernel excludes the score, it never uses it)."""
    x = _inputs(1, 8, 2, 130, 260, seed=81)
    m = torch.ones(130, 260, dtype=torch.bool)
    m[:, 100:110] = False
    a, _ = _run(x, m)
    x.k[:, :, 100:110] = float("nan")
    x.k[:, 1, 105] = float("inf")
    b, _ = _run(x, m)
    assert torch.equal(a, b)


@pytest.mark.parametrize("mdtype", [torch.bool, torch.float32, torch.bfloat16, torch.float16])
def test_staged_mask_rows_match_direct_loads(mdtype):
    """A mask with one head whose rows start on 16-byte boundaries is staged in shared
    memory by the kernel's mask warp (here a [Lq, 333] view of a [Lq, 352] tensor, so
    the last 16-byte chunk of each row is partly past the mask); the same values in
    rows that are not 16-byte aligned are read directly by the softmax threads. Both
    match the oracle and each other bit for bit, causal and not."""
    Lq, Lkv, wide = 190, 333, 352
    x = _inputs(1, 24, 4, Lq, Lkv, seed=90)              # GQA 6: 21 query rows per tile
    if mdtype == torch.bool:
        base = torch.rand(Lq, wide, generator=_gen(90)) < 0.7
    else:
        base = torch.randn(Lq, wide, generator=_gen(90)) * 2
        base[torch.rand(Lq, wide, generator=_gen(91)) < 0.15] = float("-inf")
        base = base.to(mdtype)
    staged = base[:, :Lkv]
    odd = torch.empty(Lq, Lkv + 1, dtype=mdtype)[:, :Lkv]
    odd.copy_(staged)
    assert staged.stride(0) * staged.element_size() % 16 == 0
    assert odd.stride(0) * odd.element_size() % 16 != 0
    for causal in (False, True):
        out_s, _ = _check(x, staged, f"staged {mdtype} causal={causal}", causal=causal)
        out_d, _ = _run(x, odd, causal=causal)
        assert torch.equal(out_s, out_d), f"staged vs direct {mdtype} causal={causal}"


def test_staged_masks_per_batch_and_key_padding():
    """Staged mask rows with a batch stride: a per-batch [B,1,Lq,Lkv] bf16 bias and a
    per-batch key-padding bool mask [B,1,1,Lkv] (row stride 0), both with 16-byte
    aligned rows, against the oracle."""
    B, Lq, Lkv = 2, 150, 272
    x = _inputs(B, 16, 2, Lq, Lkv, seed=92)               # GQA 8: 16 query rows per tile
    bias = (torch.randn(B, 1, Lq, Lkv, generator=_gen(92)) * 2).to(torch.bfloat16)
    _check(x, bias, "per-batch staged bias", causal=True)
    pad = torch.ones(B, 1, 1, Lkv, dtype=torch.bool)
    pad[0, ..., 230:] = False
    pad[1, ..., :7] = False
    _check(x, pad, "staged key padding")


def _random_masked(n, seed):
    """Seeded random mask cases: broadcast shape, element type, causal rule and sizes
    (key counts that do and do not give 16-byte aligned rows)."""
    rng = np.random.default_rng(seed)
    kinds = [torch.bool, torch.float32, torch.bfloat16, torch.float16]
    shapes = ["2d", "1x1", "bx1", "full", "keypad"]
    out = []
    while len(out) < n:
        Hkv = int(rng.integers(1, 4))
        gqa = int(rng.integers(1, 9))
        B = int(rng.integers(1, 3))
        Lq = int(rng.integers(1, 200))
        Lkv = Lq + int(rng.integers(0, 300))
        if rng.random() < 0.5:
            Lkv = max(16, (Lkv // 16) * 16)          # aligned rows for every element type
            Lq = min(Lq, Lkv)
        out.append((B, Hkv * gqa, Hkv, Lq, Lkv, shapes[int(rng.integers(len(shapes)))],
                    kinds[int(rng.integers(len(kinds)))], bool(rng.random() < 0.5)))
    return out


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lkv,shape,mdtype,causal", _random_masked(10, 314))
def test_random_masks(B, Hq, Hkv, Lq, Lkv, shape, mdtype, causal):
    x = _inputs(B, Hq, Hkv, Lq, Lkv, seed=Lq + Lkv + Hq)
    dims = {"2d": (Lq, Lkv), "1x1": (1, 1, Lq, Lkv), "bx1": (B, 1, Lq, Lkv),
            "full": (B, Hq, Lq, Lkv), "keypad": (B, 1, 1, Lkv)}[shape]
    gen = _gen(Lq * 3 + Lkv)
    if mdtype == torch.bool:
        m = torch.rand(dims, generator=gen) < 0.8
    else:
        m = torch.randn(dims, generator=gen) * 2
        m[torch.rand(dims, generator=gen) < 0.1] = float("-inf")
        m = m.to(mdtype)
    # a full-head mask is refused under head chunking (few rows, many heads per group)
    _check(x, m, f"random mask {B, Hq, Hkv, Lq, Lkv, shape, mdtype, causal}", causal=causal,
           chunking=shape != "full")
