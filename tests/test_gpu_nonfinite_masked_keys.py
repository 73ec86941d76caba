"""Non-finite V and K values at keys that some rows of a call do not see while other
rows of the same tile, block or split do (TensorFold PR #1009, second comment:
a masked key's infinite value times probability 0 gives NaN).  Keys a row does not
see are excluded from its sums, never weighted by 0, on every kernel:

* prompt rows (tcgen05 prefill): the causal diagonal of a row tile, GQA 1 / 6 / 8,
  planted keys in one and in both of the two key tiles a diagonal can straddle;
* chain verify on the tcgen05 split kernel and on the mma.sync split kernel
  (balanced shares, and fixed splits whose boundary falls inside the new keys);
* tree verify on both split kernels;
* general masks (bool and additive, staged and per-head mask rows).

For each case, bf16 and fp16: every output element no planted value can reach is
bit for bit the clean run's; NaN, +Inf and -Inf sit exactly where the float64
oracle (which evaluates every row over exactly its visible keys) puts them, and
the finite elements meet the parity bar.
"""
import numpy as np
import pytest
import torch

import gqa_head_gated_gb300 as G
import oracle
from synth import inputs as S
from tests.parity import assert_nonfinite_parity, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
DTYPES = [torch.bfloat16, torch.float16]
VALUE = {"v_inf": float("inf"), "v_ninf": float("-inf"), "v_nan": float("nan"),
         "k_nan": float("nan")}


def _plant(k, v, plants):
    """k, v: [Hkv, keys, 256] views of one sequence; plants: (kind, kv_head, key, col)."""
    for kind, gk, key, col in plants:
        (k if kind == "k_nan" else v)[gk, key, col] = VALUE[kind]


def _affected(sees, plants, n_rows_shape):
    """Elements a plant can reach: sees(row_index, kv_head, key) -> bool over the
    rows of `n_rows_shape` (a tuple of index ranges ending in the query head axis is
    handled by the caller); returns a bool array [*shape, 256]."""
    aff = np.zeros(n_rows_shape + (256,), dtype=bool)
    for idx in np.ndindex(*n_rows_shape):
        for kind, gk, key, col in plants:
            if sees(idx, gk, key):
                if kind == "k_nan":
                    aff[idx] = True
                else:
                    aff[idx + (col,)] = True
    return aff


def _check(out, clean, ref, aff, what):
    assert not np.isfinite(ref).all(), f"{what}: no plant reached the output"
    assert_nonfinite_parity(out, ref, what)
    keep = torch.from_numpy(~aff).to(out.device)
    assert torch.equal(out[keep], clean[keep]), f"{what}: an element no plant reaches changed"


# ----------------------------------------------------------------------------- prefill
PREFILL = {
    # GQA 6 (21 rows per tile) at an offset: diagonals of row tiles 5, 8 (straddling the
    # key tiles 256.. and 384..), 11 and the last, partial tile
    "gqa6": ((1, 24, 4, 300, 500, 200),
             [("v_inf", 1, 370, 10), ("v_nan", 1, 386, 20), ("v_ninf", 2, 312, 30),
              ("k_nan", 3, 450, 7), ("v_inf", 0, 499, 255), ("v_ninf", 0, 498, 255)]),
    # GQA 1 (128 rows per tile): partial keys fill whole key tiles
    "gqa1": ((1, 4, 4, 300, 300, 0),
             [("v_nan", 0, 5, 0), ("v_inf", 1, 127, 64), ("v_ninf", 2, 130, 128),
              ("v_inf", 3, 250, 200), ("k_nan", 3, 299, 3), ("v_nan", 0, 200, 100)]),
    # GQA 8 (16 rows per tile) at offset 143
    "gqa8": ((1, 16, 2, 257, 400, 143),
             [("v_inf", 0, 150, 1), ("v_ninf", 0, 151, 2), ("v_nan", 1, 399, 3),
              ("k_nan", 1, 300, 4)]),
    # GQA 1 at offset 64: the first row tile's diagonal spans keys 65..191 and its
    # second key tile runs to key 255, so 180 planted keys are hidden from some of its
    # rows (more than 128 in one CTA)
    "gqa1_many": ((1, 4, 4, 256, 320, 64),
                  [("v_nan" if k % 3 else "v_inf", 0, k, k % 256) for k in range(65, 245)]),
}


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
@pytest.mark.parametrize("case", sorted(PREFILL))
def test_prefill_partially_masked_keys(case, dtype):
    (B, Hq, Hkv, Lq, Lkv, off), plants = PREFILL[case]
    x = S.make_prefill(B, Hq, Hkv, Lq, Lkv=Lkv, kv_offset=off, seed=80, dtype=dtype)
    q, g = x.q.to(DEV), x.g.to(DEV)
    clean = G.prefill(q, x.k.to(DEV), x.v.to(DEV), g, kv_offset=off)
    _plant(x.k[0], x.v[0], plants)
    out, lse = G.prefill(q, x.k.to(DEV), x.v.to(DEV), g, kv_offset=off, return_lse=True)
    assert G.last_device_status() == 0
    ref, r_lse = oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g),
                                kv_offset=off)
    gqa = Hq // Hkv
    aff = _affected(lambda idx, gk, key: idx[1] // gqa == gk and key <= off + idx[2],
                    plants, (B, Hq, Lq))
    _check(out, clean, ref, aff, f"prefill {case}")
    assert_nonfinite_parity(lse, r_lse, f"prefill lse {case}", max_abs=2e-3, median_rel=1.0)


# Key outliers (2 % of the keys x8) lift rows' maxima past the fp16 rescale threshold
# (15 log2 units) again and again, so the cleaning pass rescales O while it cleans:
# single CTAs (500 keys) and CTA pairs (2100 keys).
RESCALING = {
    "single_cta": ((1, 16, 2, 300, 500, 200),
                   [("v_inf", 0, 205, 3), ("v_nan", 1, 330, 40), ("v_ninf", 1, 499, 255),
                    ("k_nan", 0, 420, 9)]),
    "cta_pair": ((1, 16, 2, 600, 2100, 1500),
                 [("v_inf", 0, 1510, 3), ("v_nan", 1, 1800, 40), ("v_ninf", 1, 2099, 255),
                  ("k_nan", 0, 1950, 9), ("v_nan", 0, 1501, 128)]),
}


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
@pytest.mark.parametrize("case", sorted(RESCALING))
def test_prefill_rescaling_rows_partially_masked_keys(case, dtype):
    (B, Hq, Hkv, Lq, Lkv, off), plants = RESCALING[case]
    x = S.make_prefill(B, Hq, Hkv, Lq, Lkv=Lkv, kv_offset=off, seed=81, dtype=dtype,
                       outlier_frac=0.02)
    q, g = x.q.to(DEV), x.g.to(DEV)
    clean = G.prefill(q, x.k.to(DEV), x.v.to(DEV), g, kv_offset=off)
    kernel = G.launch_log(1)[0]["kernel"]
    assert kernel.startswith("attn_pair_kernel" if case == "cta_pair" else "attn_tc_kernel"), kernel
    _plant(x.k[0], x.v[0], plants)
    out = G.prefill(q, x.k.to(DEV), x.v.to(DEV), g, kv_offset=off)
    assert G.last_device_status() == 0
    ref, _ = oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g), kv_offset=off)
    gqa = Hq // Hkv
    aff = _affected(lambda idx, gk, key: idx[1] // gqa == gk and key <= off + idx[2],
                    plants, (B, Hq, Lq))
    _check(out, clean, ref, aff, f"prefill with rescales {case}")


# ----------------------------------------------------------------------------- verify
VERIFY = {
    # 8 / 16 new rows x GQA 8: tcgen05 split kernel
    "tc": ((3, 16, 2, [8, 16, 1], [3000, 700, 129], 3100),
           [(0, "v_inf", 1, 2994, 3), (0, "v_nan", 0, 2999, 100), (1, "v_ninf", 1, 690, 200),
            (1, "k_nan", 0, 699, 1), (1, "v_inf", 0, 685, 50)]),
    # 2 / 2 / 1 new rows x GQA 8 (16 packed rows): mma.sync kernel, balanced shares
    "mma": ((3, 16, 2, [2, 2, 1], [3000, 700, 129], 3100),
            [(0, "v_inf", 1, 2997, 3), (0, "v_nan", 0, 2999, 100), (1, "v_ninf", 1, 699, 200),
             (0, "k_nan", 1, 2998, 9)]),
    # 2 / 2 new rows x GQA 6 (12 packed rows in a 16-row block)
    "mma_gqa6": ((2, 24, 4, [2, 2], [1500, 900], 1600),
                 [(0, "v_inf", 3, 1497, 77), (0, "v_ninf", 2, 1499, 78), (1, "v_nan", 1, 898, 79),
                  (1, "k_nan", 0, 899, 80)]),
}


def _verify_sees(x, masks=None):
    """sees((t, h), kv_head, (b, key)) for the packed rows of a decode case."""
    cu = x.cu_rows.tolist()
    lens = x.kv_lens.tolist()
    gqa = x.q.shape[1] // x.k_cache.shape[1]
    seq_of = {t: b for b in range(len(lens)) for t in range(cu[b], cu[b + 1])}

    def sees(idx, gk, bkey):
        t, h = idx
        b, key = bkey
        if seq_of[t] != b or h // gqa != gk:
            return False
        r, i = cu[b + 1] - cu[b], t - cu[b]
        base = lens[b] - r
        if masks is None:
            return key < base + i + 1
        return key < base or (key < lens[b] and (masks[t] >> (key - base)) & 1)
    return sees


def _plant_decode(x, plants):
    for b, kind, gk, key, col in plants:
        _plant(x.k_cache[b], x.v_cache[b], [(kind, gk, key, col)])


def _decode_args(x):
    return (x.q.to(DEV), x.k_cache.to(DEV), x.v_cache.to(DEV), x.g.to(DEV), x.kv_lens.to(DEV),
            x.cu_rows.to(DEV))


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
@pytest.mark.parametrize("case", sorted(VERIFY))
def test_chain_verify_partially_masked_keys(case, dtype):
    (B, Hq, Hkv, rows, lens, Lcap), plants = VERIFY[case]
    x = S.make_decode(B, Hq, Hkv, rows, lens, Lcap=Lcap, seed=81, dtype=dtype)
    kw = dict(max_rows=max(rows), max_kv_len=max(lens))
    clean = G.decode(*_decode_args(x), **kw)
    _plant_decode(x, plants)
    out, lse = G.decode(*_decode_args(x), return_lse=True, **kw)
    assert G.last_device_status() == 0
    ref, r_lse = oracle.decode(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache), to_f64(x.g),
                               lens, x.cu_rows.tolist())
    sees = _verify_sees(x)
    aff = _affected(lambda idx, gk, bk: sees(idx, gk, bk),
                    [(kind, gk, (b, key), col) for b, kind, gk, key, col in plants],
                    tuple(x.q.shape[:2]))
    _check(out, clean, ref, aff, f"chain verify {case}")
    assert_nonfinite_parity(lse, r_lse, f"verify lse {case}", max_abs=2e-3, median_rel=1.0)


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
def test_chain_verify_rescaling_rows_partially_masked_keys(dtype):
    """The tcgen05 verify case with 2 % of the cached keys scaled x8 (rows rescale, and
    keys far below a row's maximum round to an fp16 P of 0), the same plants plus a
    +Inf value at an early key every row sees."""
    (B, Hq, Hkv, rows, lens, Lcap), plants = VERIFY["tc"]
    plants = plants + [(0, "v_inf", 1, 100, 7)]
    x = S.make_decode(B, Hq, Hkv, rows, lens, Lcap=Lcap, seed=83, dtype=dtype)
    gen = torch.Generator().manual_seed(83)
    for b in range(B):
        for gk in range(Hkv):
            pos = torch.randperm(lens[b], generator=gen)[:max(1, lens[b] // 50)]
            pos = pos[pos != 100]
            x.k_cache[b, gk, pos] = (x.k_cache[b, gk, pos].float() * 8).to(dtype)
    kw = dict(max_rows=max(rows), max_kv_len=max(lens))
    clean = G.decode(*_decode_args(x), **kw)
    assert any(r["kernel"].startswith("attn_tc_kernel<split") for r in G.launch_log(2))
    _plant_decode(x, plants)
    out = G.decode(*_decode_args(x), **kw)
    assert G.last_device_status() == 0
    ref, _ = oracle.decode(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache), to_f64(x.g),
                           lens, x.cu_rows.tolist())
    sees = _verify_sees(x)
    aff = _affected(lambda idx, gk, bk: sees(idx, gk, bk),
                    [(kind, gk, (b, key), col) for b, kind, gk, key, col in plants],
                    tuple(x.q.shape[:2]))
    _check(out, clean, ref, aff, "chain verify with rescales")


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
@pytest.mark.parametrize("tc", [True, False], ids=["tcgen05", "mma"])
def test_split_boundary_inside_new_keys(tc, dtype):
    """Fixed splits whose boundary falls among the new keys (split 1024 on the tcgen05
    kernel, 64 on the mma.sync kernel), through gqa_attn_decode_split then the merge."""
    if tc:
        x = S.make_decode(1, 16, 2, [16], [1030], Lcap=1100, seed=82, dtype=dtype)
        split, plants = 1024, [(0, "v_inf", 0, 1020, 5), (0, "v_nan", 1, 1027, 6),
                               (0, "v_ninf", 1, 1015, 7)]
    else:
        x = S.make_decode(1, 8, 2, [4], [130], Lcap=140, seed=83, dtype=dtype)
        split, plants = 64, [(0, "v_inf", 0, 127, 5), (0, "v_nan", 1, 129, 6),
                             (0, "v_ninf", 1, 128, 7)]
    n_splits = -(-int(x.kv_lens.max()) // split)

    def run():
        q, kc, vc, g, kv, cu = _decode_args(x)
        o, l = G.decode_split(q, kc, vc, kv, cu, max_rows=max(x.rows),
                              max_kv_len=int(x.kv_lens.max()), num_splits=n_splits,
                              split_keys=split)
        return G.lse_merge(o, l, g.reshape(-1, 256)).reshape(x.q.shape)
    clean = run()
    _plant_decode(x, plants)
    out = run()
    assert G.last_device_status() == 0
    ref, _ = oracle.decode(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache), to_f64(x.g),
                           x.kv_lens.tolist(), x.cu_rows.tolist())
    sees = _verify_sees(x)
    aff = _affected(lambda idx, gk, bk: sees(idx, gk, bk),
                    [(kind, gk, (b, key), col) for b, kind, gk, key, col in plants],
                    tuple(x.q.shape[:2]))
    _check(out, clean, ref, aff, f"split boundary tc={tc}")


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
@pytest.mark.parametrize("case", ["tc", "mma"])
def test_tree_verify_partially_masked_keys(case, dtype):
    (B, Hq, Hkv, rows, lens, Lcap), plants = VERIFY[case]
    x = S.make_decode(B, Hq, Hkv, rows, lens, Lcap=Lcap, seed=84, dtype=dtype)
    masks = S.random_tree_masks(rows, 85)
    tm = torch.tensor([m - (1 << 64) if m >= 1 << 63 else m for m in masks], dtype=torch.int64,
                      device=DEV)
    kw = dict(max_rows=max(rows), max_kv_len=max(lens))
    clean = G.verify_tree(*_decode_args(x), tm, **kw)
    _plant_decode(x, plants)
    out = G.verify_tree(*_decode_args(x), tm, **kw)
    assert G.last_device_status() == 0
    ref, _ = oracle.decode_tree(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache),
                                to_f64(x.g), lens, x.cu_rows.tolist(), masks)
    sees = _verify_sees(x, masks)
    aff = _affected(lambda idx, gk, bk: sees(idx, gk, bk),
                    [(kind, gk, (b, key), col) for b, kind, gk, key, col in plants],
                    tuple(x.q.shape[:2]))
    _check(out, clean, ref, aff, f"tree verify {case}")


# ----------------------------------------------------------------------------- masks
def _mask(kind, Lq, Lkv, Hq, seed):
    gen = torch.Generator().manual_seed(seed)
    if kind == "bool_2d":                       # one mask head: rows staged in shared memory
        return torch.rand(Lq, Lkv, generator=gen) < 0.6
    if kind == "bool_per_head":                 # a mask head per query head: direct loads
        return torch.rand(1, Hq, Lq, Lkv, generator=gen) < 0.6
    if kind == "bias_bf16":                     # additive, -inf excludes
        a = torch.randn(Lq, Lkv, generator=gen) * 2
        a[torch.rand(Lq, Lkv, generator=gen) < 0.3] = float("-inf")
        return a.to(torch.bfloat16)
    raise ValueError(kind)


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("kind", ["bool_2d", "bool_per_head", "bias_bf16"])
def test_general_mask_partially_masked_keys(kind, causal, dtype):
    B, Hq, Hkv, Lq, Lkv = 1, 16, 2, 150, 320        # 2-D mask rows 16-byte aligned: staged
    x = S.make_prefill(B, Hq, Hkv, Lq, Lkv=Lkv, kv_offset=Lkv - Lq, seed=86, dtype=dtype)
    m = _mask(kind, Lq, Lkv, Hq, 86)
    plants = [("v_inf", 0, 3, 11), ("v_nan", 0, 140, 12), ("v_ninf", 1, 200, 13),
              ("k_nan", 1, 319, 14), ("v_inf", 1, 17, 15), ("v_nan", 0, 260, 255)]
    q, g, md = x.q.to(DEV), x.g.to(DEV), m.to(DEV)
    off = Lkv - Lq
    clean = G.masked(q, x.k.to(DEV), x.v.to(DEV), g, md, causal=causal)
    _plant(x.k[0], x.v[0], plants)
    out = G.masked(q, x.k.to(DEV), x.v.to(DEV), g, md, causal=causal)
    assert G.last_device_status() == 0
    mnp = m.numpy() if m.dtype == torch.bool else to_f64(m)
    ref, _ = oracle.sdpa_masked(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g), mnp,
                                causal=causal)
    keep = mnp if m.dtype == torch.bool else (mnp != -np.inf)
    keep = np.broadcast_to(keep, (B, Hq, Lq, Lkv))
    gqa = Hq // Hkv

    def sees(idx, gk, key):
        b, h, i = idx
        return h // gqa == gk and bool(keep[b, h, i, key]) and (not causal or key <= off + i)
    aff = _affected(sees, plants, (B, Hq, Lq))
    _check(out, clean, ref, aff, f"mask {kind} causal={causal}")
