"""KV-cache append and keep on the GPU, bit for bit against the oracle."""
import numpy as np
import pytest
import torch

import gqa_head_gated_gb300 as G
import oracle
from synth import inputs as S
from tests.parity import to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _caches(B, Hkv, Lcap, seed):
    gen = torch.Generator().manual_seed(seed)
    k = torch.randn(B, Hkv, Lcap, 256, generator=gen).to(torch.bfloat16)
    v = torch.randn(B, Hkv, Lcap, 256, generator=gen).to(torch.bfloat16)
    return k, v


def test_append_bit_exact():
    B, Hkv, Lcap = 4, 2, 300
    kc, vc = _caches(B, Hkv, Lcap, 1)
    rows, lens = [3, 0, 17, 1], [10, 5, 283, 0]
    cu = [0, 3, 3, 20, 21]
    gen = torch.Generator().manual_seed(2)
    kn = torch.randn(21, Hkv, 256, generator=gen).to(torch.bfloat16)
    vn = torch.randn(21, Hkv, 256, generator=gen).to(torch.bfloat16)
    dk, dv = kc.to(DEV), vc.to(DEV)
    G.kv_append(kn.to(DEV), vn.to(DEV), torch.tensor(lens, dtype=torch.int32, device=DEV), dk, dv,
                torch.tensor(cu, dtype=torch.int32, device=DEV))
    assert G.last_device_status() == 0
    rk, rv = oracle.kv_append(to_f64(kc), to_f64(vc), to_f64(kn), to_f64(vn), lens, cu)
    assert np.array_equal(to_f64(dk), rk) and np.array_equal(to_f64(dv), rv)
    # control: an append one row late is caught
    late_k, _ = oracle.kv_append(to_f64(kc), to_f64(vc), to_f64(kn), to_f64(vn),
                                 [x + 1 for x in lens[:2]] + lens[2:], cu)
    assert not np.array_equal(to_f64(dk), late_k)


def test_append_one_row_per_sequence_and_range_error():
    B, Hkv, Lcap = 3, 4, 64
    kc, vc = _caches(B, Hkv, Lcap, 3)
    gen = torch.Generator().manual_seed(4)
    kn = torch.randn(B, Hkv, 256, generator=gen).to(torch.bfloat16)
    vn = torch.randn(B, Hkv, 256, generator=gen).to(torch.bfloat16)
    dk, dv = kc.to(DEV), vc.to(DEV)
    G.kv_append(kn.to(DEV), vn.to(DEV), torch.tensor([0, 63, 10], dtype=torch.int32, device=DEV),
                dk, dv)
    assert G.last_device_status() == 0
    rk, rv = oracle.kv_append(to_f64(kc), to_f64(vc), to_f64(kn), to_f64(vn), [0, 63, 10],
                              [0, 1, 2, 3])
    assert np.array_equal(to_f64(dk), rk) and np.array_equal(to_f64(dv), rv)
    G.kv_append(kn.to(DEV), vn.to(DEV), torch.tensor([0, 64, 10], dtype=torch.int32, device=DEV),
                dk, dv)                              # sequence 1 is full: skipped, recorded
    assert G.last_device_status() == 6


def test_keep_bit_exact_in_place():
    B, Hkv, Lcap = 4, 2, 40
    kc, vc = _caches(B, Hkv, Lcap, 5)
    lens, cu = [20, 6, 39, 8], [0, 6, 7, 19, 19]
    keep = [[1, 2, 4], [], [0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11], []]
    flat = [i for kk in keep for i in kk]
    cuk = [0]
    for kk in keep:
        cuk.append(cuk[-1] + len(kk))
    dk, dv = kc.to(DEV), vc.to(DEV)
    out_lens = torch.zeros(B, dtype=torch.int32, device=DEV)
    G.kv_keep(dk, dv, torch.tensor(lens, dtype=torch.int32, device=DEV),
              torch.tensor(cu, dtype=torch.int32, device=DEV),
              torch.tensor(flat, dtype=torch.int32, device=DEV),
              torch.tensor(cuk, dtype=torch.int32, device=DEV), out_lens)
    assert G.last_device_status() == 0
    rk, rv, nl = oracle.kv_keep(to_f64(kc), to_f64(vc), lens, cu, keep)
    assert np.array_equal(to_f64(dk), rk) and np.array_equal(to_f64(dv), rv)
    assert out_lens.tolist() == nl


def test_keep_rejects_unsorted_list():
    kc, vc = _caches(1, 1, 16, 6)
    dk, dv = kc.to(DEV), vc.to(DEV)
    i32 = lambda xs: torch.tensor(xs, dtype=torch.int32, device=DEV)
    G.kv_keep(dk, dv, i32([10]), i32([0, 4]), i32([2, 1]), i32([0, 2]))
    assert G.last_device_status() == 6
    assert torch.equal(dk.cpu(), kc) and torch.equal(dv.cpu(), vc)


def test_append_verify_keep_decode_round_trip():
    """Drafts appended, verified over a tree, the accepted path kept: the next decode
    step equals the one over a cache where only the accepted rows were ever appended."""
    Hq, Hkv, Lcap = 16, 2, 4096
    x = S.make_decode(2, Hq, Hkv, [1, 1], [3000, 1500], Lcap=Lcap, seed=8, pad_value=0.0)
    kc, vc = x.k_cache.to(DEV), x.v_cache.to(DEV)
    lens0 = [3000, 1500]
    rows = [6, 4]
    gen = torch.Generator().manual_seed(9)
    kd = torch.randn(10, Hkv, 256, generator=gen).to(torch.bfloat16).to(DEV)
    vd = torch.randn(10, Hkv, 256, generator=gen).to(torch.bfloat16).to(DEV)
    qd = torch.randn(10, Hq, 256, generator=gen).to(torch.bfloat16).to(DEV)
    gd = (torch.randn(10, Hq, 256, generator=gen) * 2).to(torch.bfloat16).to(DEV)
    cu = torch.tensor([0, 6, 10], dtype=torch.int32, device=DEV)
    i32 = lambda xs: torch.tensor(xs, dtype=torch.int32, device=DEV)
    G.kv_append(kd, vd, i32(lens0), kc, vc, cu)
    masks = S.random_tree_masks(rows, 10)
    G.verify_tree(qd, kc, vc, gd, i32([3006, 1504]), cu,
                  torch.tensor(masks, dtype=torch.int64, device=DEV), max_rows=6, max_kv_len=3006)
    keep = [[0, 2, 5], [1, 3]]
    lens1 = torch.zeros(2, dtype=torch.int32, device=DEV)
    G.kv_keep(kc, vc, i32([3006, 1504]), cu, i32([0, 2, 5, 1, 3]), i32([0, 3, 5]), lens1)
    assert lens1.tolist() == [3003, 1502]
    # the same cache built by appending only the accepted rows
    kc2, vc2 = x.k_cache.to(DEV), x.v_cache.to(DEV)
    acc = [0, 2, 5, 6 + 1, 6 + 3]
    G.kv_append(kd[acc].contiguous(), vd[acc].contiguous(), i32(lens0), kc2, vc2, i32([0, 3, 5]))
    assert G.last_device_status() == 0
    for b, n in enumerate([3003, 1502]):            # each sequence up to its new length
        assert torch.equal(kc[b, :, :n], kc2[b, :, :n]) and torch.equal(vc[b, :, :n], vc2[b, :, :n])
    q1 = torch.randn(2, Hq, 256, generator=gen).to(torch.bfloat16).to(DEV)
    a = G.decode(q1, kc, vc, None, lens1, None, max_rows=1, max_kv_len=3003)
    b = G.decode(q1, kc2, vc2, None, lens1, None, max_rows=1, max_kv_len=3003)
    assert torch.equal(a, b)
