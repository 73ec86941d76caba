"""FP16 entry points (the `_f16` twins of the C ABI) on the GPU against the float64
oracle: prefill on the tcgen05 kernel, decode / chain verify / tree verify on both
split kernels, the LSE merge.  The d-inference page ships FP16 and BF16 symbols of
its head_dim-256 kernel (PR #640, "Summary"); the oracle is the same float64
definition, fed the exact fp16 values."""
import numpy as np
import pytest
import torch

import gqa_head_gated_gb300 as G
import oracle
from synth import inputs as S
from tests.parity import assert_parity_dtype, errors, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
F16 = torch.float16


def prefill_run(x, lse=False):
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    r = G.prefill(q, k, v, g, kv_offset=x.kv_offset, return_lse=lse)
    assert G.last_device_status() == 0
    return r


def prefill_ref(x):
    return oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g),
                          kv_offset=x.kv_offset)


@pytest.mark.parametrize("B,Hq,Hkv,Lq,Lkv,off", [
    (1, 2, 2, 37, 37, 0),
    (1, 4, 4, 129, 129, 0),
    (1, 24, 4, 300, 300, 0),
    (1, 16, 2, 257, 400, 143),
    (2, 24, 2, 45, 300, 255),
    (1, 128, 1, 5, 9, 3),
    (1, 8, 8, 640, 1000, 360),
])
def test_prefill_fp16_shapes(B, Hq, Hkv, Lq, Lkv, off):
    x = S.make_prefill(B, Hq, Hkv, Lq, Lkv=Lkv, kv_offset=off, seed=300 + Lq, dtype=F16)
    out, lse = prefill_run(x, lse=True)
    assert out.dtype == F16
    r_out, r_lse = prefill_ref(x)
    assert_parity_dtype(out, r_out, f"fp16 prefill {B, Hq, Hkv, Lq, Lkv, off}")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)


def test_prefill_fp16_rescale_stress():
    """Keys scaled x8 (2% of rows) give score spreads of tens of log2 units, so the
    running maximum jumps past the rescale threshold again and again.  fp16 P must
    stay finite: the tcgen05 kernel rescales once the maximum grows by 15 (P <= 2^15,
    below fp16's 65504); with bf16's threshold of 32 P would reach 2^32 and overflow
    fp16."""
    x = S.make_prefill(1, 8, 2, 700, seed=31, outlier_frac=0.02, dtype=F16)
    out = prefill_run(x)
    assert torch.isfinite(out).all()
    assert_parity_dtype(out, prefill_ref(x)[0], "fp16 rescale stress")


def test_prefill_fp16_matches_bf16_to_rounding():
    """The same draws rounded to fp16 and to bf16 give outputs that agree to bf16's
    resolution (the kernels differ only in element type)."""
    a = prefill_run(S.make_prefill(1, 16, 2, 200, seed=32))
    b = prefill_run(S.make_prefill(1, 16, 2, 200, seed=32, dtype=F16))
    e = errors(b, a.float())
    assert e["max_abs"] <= 3e-2 and e["median_rel"] <= 1e-2, e


def test_prefill_chunked_35b_fp16_sampled():
    """The 2048-row chunk at kv_offset 30720 in fp16, full size, on sampled rows."""
    x = S.chunked_prefill_35b(dtype=F16)
    out, lse = prefill_run(x, lse=True)
    assert torch.isfinite(out).all()
    rng = np.random.default_rng(2)
    rows = sorted({(0, int(rng.integers(16)), int(rng.integers(2048))) for _ in range(96)}
                  | {(0, h, 2047) for h in range(16)})
    r_out, r_lse = oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g),
                                  kv_offset=x.kv_offset, rows=rows)
    got = torch.stack([out[b, h, i] for b, h, i in rows])
    assert_parity_dtype(got, r_out, "chunked 35B fp16")
    np.testing.assert_allclose(np.array([float(lse[b, h, i]) for b, h, i in rows]), r_lse,
                               rtol=0, atol=2e-3)


def dev(x):
    return (x.q.to(DEV), x.k_cache.to(DEV), x.v_cache.to(DEV), x.g.to(DEV), x.kv_lens.to(DEV),
            x.cu_rows.to(DEV))


def decode_ref(x):
    return oracle.decode(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache), to_f64(x.g),
                         x.kv_lens.tolist(), x.cu_rows.tolist())


def test_decode_27b_fp16_workload():
    """16 sequences, one row each, 24/4 heads, kv lengths up to 32768 (NaN padding):
    the bench's decode workload in fp16."""
    x = S.decode_27b(dtype=F16)
    q, kc, vc, g, kv, _ = dev(x)
    out, lse = G.decode(q, kc, vc, g, kv, None, max_rows=1, max_kv_len=int(x.kv_lens.max()),
                        return_lse=True)
    assert G.last_device_status() == 0 and out.dtype == F16
    r_out, r_lse = decode_ref(x)
    assert_parity_dtype(out, r_out, "decode 27B fp16")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)


@pytest.mark.parametrize("Hq,Hkv,rows,kv", [
    (24, 4, [1, 1, 1], [8191, 300, 129]),       # mma.sync split
    (16, 2, [3, 4, 8], [3, 100, 4097]),          # tcgen05 split (64 packed rows)
    (16, 2, [16, 32], [40, 3000]),               # tcgen05 split (256 packed rows)
    (12, 1, [5, 2], [700, 5]),                   # tcgen05 split (60 packed rows)
    (16, 2, [2, 1], [700, 5]),                   # mma.sync (16 packed rows)
])
def test_decode_fp16_sweep(Hq, Hkv, rows, kv):
    x = S.make_decode(len(rows), Hq, Hkv, rows, kv, Lcap=max(kv) + 5, seed=sum(kv) + 3,
                      dtype=F16)
    q, kc, vc, g, kvd, cu = dev(x)
    out, lse = G.decode(q, kc, vc, g, kvd, cu, max_rows=max(rows), max_kv_len=max(kv),
                        return_lse=True)
    assert G.last_device_status() == 0
    r_out, r_lse = decode_ref(x)
    assert_parity_dtype(out, r_out, f"decode fp16 {Hq, Hkv, rows, kv}")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)


@pytest.mark.parametrize("Hq,Hkv,rows,kv", [(16, 2, [8, 32, 1], [3000, 9000, 129]),
                                         (24, 4, [11, 2], [4097, 700])])
def test_fp16_tc_and_mma_split_paths(Hq, Hkv, rows, kv):
    """Both split kernels in fp16 (split sizes 1024: tcgen05, 1088: mma.sync), merged
    by the fp16 merge, against the oracle."""
    x = S.make_decode(len(rows), Hq, Hkv, rows, kv, seed=sum(kv) + 4, dtype=F16)
    q, kc, vc, g, kvd, cu = dev(x)
    mk = max(kv)
    ref = decode_ref(x)[0]
    for C in (1024, 1088):
        op, lp = G.decode_split(q, kc, vc, kvd, cu, max_rows=max(rows), max_kv_len=mk,
                                num_splits=(mk + C - 1) // C, split_keys=C)
        out = G.lse_merge(op, lp, g).view_as(q)
        assert out.dtype == F16
        assert_parity_dtype(out, ref, f"fp16 split C={C}")
    assert G.last_device_status() == 0


def as_tensor(masks):
    return torch.tensor([m - (1 << 64) if m >= 1 << 63 else m for m in masks],
                        dtype=torch.int64, device=DEV)


@pytest.mark.parametrize("Hq,Hkv,rows,kv", [(16, 2, [8, 3, 16, 1], [3000, 700, 9000, 129]),
                                         (24, 4, [9, 2, 4], [300, 8200, 1000])])
def test_tree_verify_fp16(Hq, Hkv, rows, kv):
    x = S.make_decode(len(rows), Hq, Hkv, rows, kv, Lcap=max(kv) + 33, seed=sum(kv) + 5,
                      dtype=F16)
    masks = S.random_tree_masks(rows, sum(rows) + 1)
    q, kc, vc, g, kvd, cu = dev(x)
    out, lse = G.verify_tree(q, kc, vc, g, kvd, cu, as_tensor(masks), max_rows=max(rows),
                             max_kv_len=max(kv), return_lse=True)
    assert G.last_device_status() == 0 and out.dtype == F16
    r_out, r_lse = oracle.decode_tree(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache),
                                      to_f64(x.g), x.kv_lens.tolist(), x.cu_rows.tolist(), masks)
    assert_parity_dtype(out, r_out, f"tree fp16 {Hq, Hkv, rows, kv}")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)


def test_merge_fp16_against_oracle():
    gen = torch.Generator().manual_seed(33)
    Sn, N = 5, 200
    o = torch.randn(Sn, N, 256, generator=gen)
    l = torch.randn(Sn, N, generator=gen) * 3
    empty = torch.rand(Sn, N, generator=gen) < 0.3
    l[empty] = float("-inf")
    o[empty] = float("nan")
    gate = (torch.randn(N, 256, generator=gen) * 2).to(F16)
    out, lse = G.lse_merge(o.to(DEV), l.to(DEV), gate.to(DEV), return_lse=True)
    assert out.dtype == F16
    r_out, r_lse = oracle.lse_merge(o.double().numpy(), l.double().numpy(), to_f64(gate))
    assert_parity_dtype(out, r_out, "merge fp16")
    fin = np.isfinite(r_lse)
    np.testing.assert_allclose(to_f64(lse)[fin], r_lse[fin], rtol=0, atol=1e-5)


def test_kv_append_keep_fp16_bit_exact():
    """Append and keep copy 16-bit elements, so fp16 caches round-trip bit for bit."""
    x = S.make_decode(2, 8, 2, [3, 2], [10, 7], Lcap=16, seed=34, pad_value=0.0, dtype=F16)
    gen = torch.Generator().manual_seed(35)
    kn = torch.randn(5, 2, 256, generator=gen).to(F16)
    vn = torch.randn(5, 2, 256, generator=gen).to(F16)
    kc, vc = x.k_cache.to(DEV), x.v_cache.to(DEV)
    G.kv_append(kn.to(DEV), vn.to(DEV), x.kv_lens.to(DEV), kc, vc, x.cu_rows.to(DEV))
    assert G.last_device_status() == 0
    rk, rv = oracle.kv_append(x.k_cache.numpy().view(np.uint16), x.v_cache.numpy().view(np.uint16),
                              kn.numpy().view(np.uint16), vn.numpy().view(np.uint16),
                              x.kv_lens.tolist(), x.cu_rows.tolist())
    assert np.array_equal(kc.cpu().numpy().view(np.uint16), rk)
    assert np.array_equal(vc.cpu().numpy().view(np.uint16), rv)
