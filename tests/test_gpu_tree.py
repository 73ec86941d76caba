"""Tree-masked draft verify on the GPU (both split kernels) against the float64
oracle."""
import numpy as np
import pytest
import torch

import gqa_head_gated_gb300 as G
import oracle
from synth import inputs as S
from tests.parity import assert_parity, fails_parity, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def as_tensor(masks):
    # masks are < 2^64; store the bit pattern in int64
    return torch.tensor([m - (1 << 64) if m >= 1 << 63 else m for m in masks],
                        dtype=torch.int64, device=DEV)


def run_tree(x, masks, lse=False):
    r = G.verify_tree(x.q.to(DEV), x.k_cache.to(DEV), x.v_cache.to(DEV), x.g.to(DEV),
                      x.kv_lens.to(DEV), x.cu_rows.to(DEV), as_tensor(masks),
                      max_rows=max(x.rows), max_kv_len=int(x.kv_lens.max()), return_lse=lse)
    assert G.last_device_status() == 0
    return r


def ref_tree(x, masks):
    return oracle.decode_tree(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache), to_f64(x.g),
                              x.kv_lens.tolist(), x.cu_rows.tolist(), masks)


CASES = [
    # Hq, Hkv, rows, kv_lens: more than 16 packed rows per group take the tcgen05 kernel
    (16, 2, [8, 3, 16, 1], [3000, 700, 9000, 129]),     # tcgen05 (16 x 8 = 128)
    (8, 4, [5, 12], [2000, 4100]),                       # tcgen05 (12 x 2 = 24)
    (4, 4, [64, 7], [5000, 64]),                         # tcgen05, a 64-row tree
    (24, 4, [9, 2, 4], [300, 8200, 1000]),               # tcgen05 (9 x 6 = 54)
    (8, 4, [5, 8], [2000, 4100]),                        # mma.sync (8 x 2 = 16)
    (24, 4, [2, 2, 1], [300, 8200, 1000]),               # mma.sync (2 x 6 = 12)
]


@pytest.mark.parametrize("Hq,Hkv,rows,kv", CASES)
def test_tree_verify_matches_oracle(Hq, Hkv, rows, kv):
    x = S.make_decode(len(rows), Hq, Hkv, rows, kv, Lcap=max(kv) + 33, seed=sum(kv) + 1)
    masks = S.random_tree_masks(rows, sum(rows))
    out, lse = run_tree(x, masks, lse=True)
    r_out, r_lse = ref_tree(x, masks)
    assert_parity(out, r_out, f"tree {Hq, Hkv, rows, kv}")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)


@pytest.mark.parametrize("Hq,Hkv,rows,kv", [(16, 2, [8, 16], [3000, 9000]),
                                            (8, 4, [5, 12], [2000, 4100])])
def test_chain_masks_equal_chain_verify(Hq, Hkv, rows, kv):
    """Chain masks (row i sees new rows 0..i) reproduce gqa_attn_decode bit for bit on
    the same kernel path."""
    x = S.make_decode(len(rows), Hq, Hkv, rows, kv, seed=7)
    tree = run_tree(x, oracle.chain_masks(rows))
    chain = G.decode(x.q.to(DEV), x.k_cache.to(DEV), x.v_cache.to(DEV), x.g.to(DEV),
                     x.kv_lens.to(DEV), x.cu_rows.to(DEV), max_rows=max(rows),
                     max_kv_len=max(kv))
    assert torch.equal(tree, chain)


def test_ignoring_the_tree_control():
    """Control: the oracle's chain result must fail parity against a branching tree's
    GPU output (the masks reach the kernels)."""
    rows, kv = [16, 8], [3000, 5000]
    x = S.make_decode(2, 16, 2, rows, kv, seed=9)
    masks = S.random_tree_masks(rows, 3)
    out = run_tree(x, masks)
    chain_ref = ref_tree(x, oracle.chain_masks(rows))[0]
    assert fails_parity(out, chain_ref)


def test_tree_padding_never_read():
    """NaN cache padding past kv_len leaves the tree outputs finite and unchanged."""
    rows, kv = [16, 3], [1000, 2000]
    x = S.make_decode(2, 16, 2, rows, kv, Lcap=2200, seed=11, pad_value=0.0)
    masks = S.random_tree_masks(rows, 4)
    a = run_tree(x, masks)
    x.k_cache[0, :, 1000:] = float("nan")
    x.v_cache[0, :, 1000:] = float("nan")
    b = run_tree(x, masks)
    assert torch.equal(a, b)


def _random_verify(n, seed):
    """Seeded random verify batches: 1-4 sequences of 0-40 new rows (0-64 for one of
    them), GQA 1-12 over 1-4 KV heads, kv lengths from the rows up to 6,000; both
    kernels are hit (the path follows max rows x GQA)."""
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        Hkv = int(rng.integers(1, 5))
        gqa = int(rng.integers(1, 13))
        B = int(rng.integers(1, 5))
        rows = [int(rng.integers(0, 41)) for _ in range(B)]
        if rng.random() < 0.3:
            rows[0] = int(rng.integers(41, 65))
        if max(rows) == 0:
            rows[0] = 1
        kv = [r + int(rng.integers(0, 6001)) for r in rows]
        kv = [max(k, 1) for k in kv]
        out.append((Hkv * gqa, Hkv, rows, kv))
    return out


@pytest.mark.parametrize("Hq,Hkv,rows,kv", _random_verify(8, 77) + [
    (4, 2, [3, 8, 0, 5], [100, 5000, 0, 37]),        # mma.sync path, a sequence with no rows
    (6, 3, [1, 1, 1], [1, 4097, 300])])               # decode rows, a one-key sequence
def test_random_tree_and_chain_verify(Hq, Hkv, rows, kv):
    x = S.make_decode(len(rows), Hq, Hkv, rows, kv, Lcap=max(kv) + 17, seed=sum(kv) + Hq)
    masks = S.random_tree_masks(rows, sum(rows) + 5)
    out, lse = run_tree(x, masks, lse=True)
    r_out, r_lse = ref_tree(x, masks)
    assert_parity(out, r_out, f"random tree {Hq, Hkv, rows, kv}")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)
    chain = G.decode(x.q.to(DEV), x.k_cache.to(DEV), x.v_cache.to(DEV), x.g.to(DEV),
                     x.kv_lens.to(DEV), x.cu_rows.to(DEV), max_rows=max(rows),
                     max_kv_len=int(x.kv_lens.max()))
    r_chain = oracle.decode(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache), to_f64(x.g),
                            x.kv_lens.tolist(), x.cu_rows.tolist())[0]
    assert_parity(chain, r_chain, f"random chain {Hq, Hkv, rows, kv}")
