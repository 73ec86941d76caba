"""Non-finite inputs on the GPU, bf16 and fp16 (the TensorFold attention contract's
gate 1 plants NaN / Inf inputs and compares with float64 gated attention).

* Positions no row sees (prompt keys past the last row, cache rows past kv_len)
  and K of keys masked for a row: outputs of the rows that do not see them are
  bit for bit those of the clean run.
* Values that rows see -- a NaN query element, +-Inf / NaN in the value or key of
  a key every row of the call sees, infinite or NaN gates: NaN, +Inf and -Inf sit
  exactly where the float64 oracle puts them, and the finite elements meet the
  parity bar.  The planted keys lie before the rows' own positions, so no row of
  the call multiplies them by a probability of 0 (0 * Inf would be NaN where
  float64 excludes the key).
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
NAN, INF = float("nan"), float("inf")


def plant(kind, q, k, v, g, key, g_kv=0):
    """Plants one kind of non-finite value.  q, g: [..., rows, 256] indexed by a
    leading (row) tuple below; k, v: [Hkv, keys, 256] views of one sequence."""
    if kind == "q_nan":
        q[0][3, 17] = NAN
        q[1][0, 200] = NAN
    elif kind == "v_inf":
        v[g_kv, key, 10] = INF
        v[g_kv, key + 1, 20] = -INF
        v[g_kv, key + 2, 30] = NAN
    elif kind == "k_inf":
        k[g_kv, key, 5] = INF
    elif kind == "k_nan":
        k[g_kv, key, 99] = NAN
    elif kind == "g_nonfinite":
        g[0][1, 3] = -INF
        g[0][1, 4] = INF
        g[1][2, 5] = NAN
    else:
        raise ValueError(kind)


KINDS = ["q_nan", "v_inf", "k_inf", "k_nan", "g_nonfinite"]


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
@pytest.mark.parametrize("kind", KINDS)
def test_prefill_visible_nonfinite(kind, dtype):
    """A 300-row chunk at kv_offset 200 (24/4 heads): keys 0..199 are seen by every
    row; the plants sit at keys 50..52 of KV head 1."""
    x = S.make_prefill(1, 24, 4, 300, Lkv=500, kv_offset=200, seed=50, dtype=dtype)
    # q, g rows are (head, row) pairs: pass [B=0][h] views
    plant(kind, [x.q[0, 0], x.q[0, 7]], x.k[0], x.v[0], [x.g[0, 6], x.g[0, 23]], key=50,
          g_kv=1)
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    out, lse = G.prefill(q, k, v, g, kv_offset=200, return_lse=True)
    assert G.last_device_status() == 0
    r_out, r_lse = oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g),
                                  kv_offset=200)
    assert not np.isfinite(r_out).all()          # the plant reached the output
    assert_nonfinite_parity(out, r_out, f"prefill {kind}")
    assert_nonfinite_parity(lse, r_lse, f"prefill lse {kind}", max_abs=2e-3, median_rel=1.0)


def _decode_case(dtype, tc):
    if tc:      # 16 x 8 packed rows per group: tcgen05 split kernel
        return S.make_decode(3, 16, 2, [8, 16, 1], [3000, 700, 129], Lcap=3100, seed=51,
                             dtype=dtype)
    # 6 packed rows per group: mma.sync split kernel
    return S.make_decode(3, 24, 4, [1, 1, 1], [5000, 700, 129], Lcap=5100, seed=52,
                         dtype=dtype)


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
@pytest.mark.parametrize("tc", [True, False], ids=["tcgen05", "mma"])
@pytest.mark.parametrize("kind", KINDS)
def test_decode_visible_nonfinite(kind, tc, dtype):
    """Decode / chain verify; the plants sit at keys 60..62 of sequence 0's KV head
    1 (before its new rows, seen by all of them)."""
    x = _decode_case(dtype, tc)
    plant(kind, [x.q[0], x.q[1]], x.k_cache[0], x.v_cache[0], [x.g[0], x.g[2]], key=60,
          g_kv=1)
    q, kc, vc, g, kv, cu = (t.to(DEV) for t in (x.q, x.k_cache, x.v_cache, x.g, x.kv_lens,
                                                 x.cu_rows))
    out, lse = G.decode(q, kc, vc, g, kv, cu, max_rows=max(x.rows),
                        max_kv_len=int(x.kv_lens.max()), return_lse=True)
    assert G.last_device_status() == 0
    r_out, r_lse = oracle.decode(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache),
                                 to_f64(x.g), x.kv_lens.tolist(), x.cu_rows.tolist())
    assert not np.isfinite(r_out).all()
    assert_nonfinite_parity(out, r_out, f"decode {kind}")
    assert_nonfinite_parity(lse, r_lse, f"decode lse {kind}", max_abs=2e-3, median_rel=1.0)


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
@pytest.mark.parametrize("tc", [True, False], ids=["tcgen05", "mma"])
def test_tree_visible_nonfinite(tc, dtype):
    """Tree verify with +-Inf / NaN values at keys every new row sees."""
    x = _decode_case(dtype, tc)
    plant("v_inf", None, x.k_cache[0], x.v_cache[0], None, key=60, g_kv=1)
    masks = S.random_tree_masks(x.rows, 53)
    tm = torch.tensor([m - (1 << 64) if m >= 1 << 63 else m for m in masks], dtype=torch.int64,
                      device=DEV)
    q, kc, vc, g, kv, cu = (t.to(DEV) for t in (x.q, x.k_cache, x.v_cache, x.g, x.kv_lens,
                                                 x.cu_rows))
    out = G.verify_tree(q, kc, vc, g, kv, cu, tm, max_rows=max(x.rows),
                        max_kv_len=int(x.kv_lens.max()))
    assert G.last_device_status() == 0
    r_out, _ = oracle.decode_tree(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache),
                                  to_f64(x.g), x.kv_lens.tolist(), x.cu_rows.tolist(), masks)
    assert_nonfinite_parity(out, r_out, "tree v_inf")


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
def test_prefill_unseen_and_masked_keys(dtype):
    """NaN / Inf past the last row's position change nothing; a NaN key at position
    kv_offset + 40 turns exactly the rows that see it NaN and leaves rows 0..39
    bit for bit unchanged."""
    x = S.make_prefill(1, 16, 2, 100, Lkv=300, kv_offset=50, seed=54, dtype=dtype)
    q, g = x.q.to(DEV), x.g.to(DEV)
    clean = G.prefill(q, x.k.to(DEV), x.v.to(DEV), g, kv_offset=50)
    k2, v2 = x.k.clone(), x.v.clone()
    k2[:, :, 150:] = NAN
    v2[:, :, 150:] = -INF
    k2[:, 1, 90, 7] = NAN                        # seen by rows 40.. of KV head 1's heads
    out = G.prefill(q, k2.to(DEV), v2.to(DEV), g, kv_offset=50)
    assert G.last_device_status() == 0
    assert torch.equal(out[:, :8], clean[:, :8])        # KV head 0's heads: untouched
    assert torch.equal(out[:, 8:, :40], clean[:, 8:, :40])
    assert torch.isnan(out[:, 8:, 40:]).all()


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
@pytest.mark.parametrize("tc", [True, False], ids=["tcgen05", "mma"])
def test_decode_unseen_padding(tc, dtype):
    """Cache rows past kv_len hold +Inf, -Inf or NaN: outputs are bit-identical."""
    outs = []
    for pad in (0.0, NAN, INF, -INF):
        x = _decode_case(dtype, tc)
        for b, L in enumerate(x.kv_lens.tolist()):
            x.k_cache[b, :, L:] = pad
            x.v_cache[b, :, L:] = pad
        q, kc, vc, g, kv, cu = (t.to(DEV) for t in (x.q, x.k_cache, x.v_cache, x.g, x.kv_lens,
                                                     x.cu_rows))
        outs.append(G.decode(q, kc, vc, g, kv, cu, max_rows=max(x.rows),
                             max_kv_len=int(x.kv_lens.max())))
    assert G.last_device_status() == 0
    assert torch.isfinite(outs[0]).all()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


@pytest.mark.parametrize("dtype", DTYPES, ids=["bf16", "fp16"])
def test_merge_nonfinite_parts(dtype):
    """A NaN lse part poisons its row; +Inf lse gives NaN; a -inf part's NaN O row is
    never read."""
    o = torch.ones(3, 3, 256)
    l = torch.tensor([[0.1, 0.2, 0.3], [NAN, -INF, INF], [0.5, 0.5, 0.5]])
    o[1, 1] = NAN
    out, lse = G.lse_merge(o.to(DEV), l.to(DEV), None, return_lse=True, dtype=dtype)
    r_out, r_lse = oracle.lse_merge(o.double().numpy(), l.double().numpy())
    assert_nonfinite_parity(out, r_out, "merge")
    assert_nonfinite_parity(lse, r_lse, "merge lse", max_abs=1e-5, median_rel=1.0)


@pytest.mark.parametrize("dtype,tc", [(torch.bfloat16, True), (torch.bfloat16, False),
                                      (torch.float16, True)],
                         ids=["bf16-tcgen05", "bf16-mma", "fp16-tcgen05"])
def test_visible_inf_at_low_probability_key(dtype, tc):
    """+Inf in V at a key every row sees whose probability is 2^-46 of the row
    maximum's (key 60 = -u against key 50 = u, every query row of the group = u):
    float64's p is tiny but positive, so that column is +Inf.  An fp16 P rounds such
    a probability to 0; the tensor-memory kernel's fp16 cleaning pass still gives
    +Inf.  (The cp.async kernel in fp16 gives NaN there, a stated limit; bf16 P keeps
    probabilities down to 126 log2 units below the maximum.)"""
    x = _decode_case(dtype, tc)
    gqa = x.q.shape[1] // x.k_cache.shape[1]
    r0, r1 = int(x.cu_rows[0]), int(x.cu_rows[1])
    u = x.q[r0, gqa].clone()                              # sequence 0, KV head 1
    x.q[r0:r1, gqa:2 * gqa] = u
    x.k_cache[0, 1, 50] = u
    x.k_cache[0, 1, 60] = -u
    x.v_cache[0, 1, 60, 5] = INF
    q, kc, vc, g, kv, cu = (t.to(DEV) for t in (x.q, x.k_cache, x.v_cache, x.g, x.kv_lens,
                                                 x.cu_rows))
    out = G.decode(q, kc, vc, g, kv, cu, max_rows=max(x.rows), max_kv_len=int(x.kv_lens.max()))
    assert G.last_device_status() == 0
    r_out, _ = oracle.decode(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache), to_f64(x.g),
                             x.kv_lens.tolist(), x.cu_rows.tolist())
    assert np.isposinf(r_out[r0:r1, gqa:2 * gqa, 5]).all()
    assert_nonfinite_parity(out, r_out, "visible +Inf at a low-probability key")
