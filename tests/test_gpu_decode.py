"""Decode / chain verify and the LSE merge on the GPU, through the C ABI, against the
float64 oracle."""
import numpy as np
import pytest
import torch

import gqa_head_gated_gb300 as G
import oracle
from synth import inputs as S
from tests.parity import MAX_ABS, MEDIAN_REL, assert_parity, errors, fails_parity, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def dev(x):
    return (x.q.to(DEV), x.k_cache.to(DEV), x.v_cache.to(DEV), x.g.to(DEV), x.kv_lens.to(DEV),
            x.cu_rows.to(DEV))


def run(x, gate=True, lse=False, one_row=False):
    q, kc, vc, g, kv, cu = dev(x)
    r = G.decode(q, kc, vc, g if gate else None, kv, None if one_row else cu,
                 max_rows=max(x.rows) if x.rows else 1, max_kv_len=int(x.kv_lens.max()),
                 return_lse=lse)
    assert G.last_device_status() == 0
    return r


def ref(x, gate=True):
    return oracle.decode(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache),
                         to_f64(x.g) if gate else None, x.kv_lens.tolist(), x.cu_rows.tolist())


def test_decode_27b_workload():
    """16 sequences, one row each, kv lengths 1987..32233 in a 32768-key cache whose
    padding is NaN; the bench's launch configuration."""
    x = S.decode_27b()
    out, lse = run(x, lse=True, one_row=True)
    r_out, r_lse = ref(x)
    assert_parity(out, r_out, "decode 27B")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)


def test_verify_35b_workload():
    """8 sequences with 1..32 verify rows, kv lengths 4271..45513 in a 65536-key cache."""
    x = S.verify_35b()
    out, lse = run(x, lse=True)
    r_out, r_lse = ref(x)
    assert_parity(out, r_out, "verify 35B")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)


SWEEP = [
    # Hq, Hkv, rows, kv_lens
    (4, 4, [1, 1, 1], [1, 2, 3]),
    (8, 2, [1, 1, 1, 1], [127, 128, 129, 63]),
    (24, 4, [1, 1], [8190, 8191]),
    (24, 4, [1, 1], [8192, 8193]),
    (16, 2, [3, 4, 8], [3, 100, 4097]),
    (16, 2, [16, 32], [40, 1000]),
    (12, 1, [5, 2], [700, 5]),                # GQA 12: 60 packed rows (tcgen05)
    (16, 2, [2, 1, 2], [900, 50, 3000]),      # 16 packed rows: the mma.sync kernel's largest
    (32, 4, [32, 7], [300, 3000]),            # GQA 8 x 32 rows = 256 packed rows
    (6, 6, [64], [2000]),                     # 64 rows, GQA 1
    (16, 1, [9, 0, 1], [500, 0, 33]),         # a sequence with no rows
]


@pytest.mark.parametrize("Hq,Hkv,rows,kv", SWEEP)
def test_decode_sweep(Hq, Hkv, rows, kv):
    x = S.make_decode(len(rows), Hq, Hkv, rows, kv, Lcap=max(kv) + 7, seed=sum(kv) + Hq)
    out, lse = run(x, lse=True)
    r_out, r_lse = ref(x)
    assert_parity(out, r_out, f"decode {Hq,Hkv,rows,kv}")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)


def test_decode_ungated():
    x = S.make_decode(3, 8, 2, [1, 2, 3], [10, 200, 3000], seed=12)
    assert_parity(run(x, gate=False), ref(x, gate=False)[0], "ungated")


def test_padding_and_future_keys_bit_exact():
    """Cache padding (NaN vs other garbage) never changes an output; perturbing the
    keys of later verify rows leaves earlier rows bit for bit unchanged."""
    x = S.make_decode(2, 16, 2, [4, 8], [900, 5000], Lcap=5100, seed=13)
    a = run(x)
    x.k_cache[0, :, 900:] = 7.0
    x.v_cache[1, :, 5000:] = float("-inf")
    b = run(x)
    assert torch.equal(a, b)
    # sequence 1 rows: kv_len 5000, 8 rows at positions 4992..4999; perturb 4996..4999
    x.k_cache[1, :, 4996:5000] = (x.k_cache[1, :, 4996:5000].float() * 3).to(torch.bfloat16)
    x.v_cache[1, :, 4996:5000] = (x.v_cache[1, :, 4996:5000].float() - 2).to(torch.bfloat16)
    c = run(x)
    t0 = 4
    assert torch.equal(a[:t0 + 4], c[:t0 + 4])
    assert not torch.equal(a[t0 + 4:], c[t0 + 4:])


def test_verify_row_equals_decode_row():
    """Row i of an r-row verify equals a one-row decode at kv_len - r + i + 1."""
    r, L = 8, 3000
    x = S.make_decode(1, 16, 2, [r], [L], seed=14)
    full = run(x)
    for i in [0, 3, 7]:
        y = S.DecodeInputs(x.q[i:i + 1].clone(), x.k_cache, x.v_cache, x.g[i:i + 1].clone(),
                           torch.tensor([L - r + i + 1], dtype=torch.int32),
                           torch.tensor([0, 1], dtype=torch.int32), 0)
        one = run(y, one_row=True)
        # 8 rows x 8 heads run on the tcgen05 kernel, one row on the mma.sync kernel:
        # the two agree within the parity tolerance.
        e = errors(one, full[i:i + 1].float())
        assert e["max_abs"] <= MAX_ABS and e["median_rel"] <= MEDIAN_REL, e


def test_split_then_merge_equals_decode():
    """The exposed split + merge (fixed splits) and the one-call decode (balanced
    shares on this path) agree within rounding; the split + merge result does not
    depend on who launches the merge."""
    x = S.make_decode(4, 24, 4, [1, 2, 1, 3], [5000, 70, 12000, 900], seed=15)
    out = run(x)
    q, kc, vc, g, kv, cu = dev(x)
    op, lp = G.decode_split(q, kc, vc, kv, cu, max_rows=3, max_kv_len=12000)
    merged = G.lse_merge(op, lp, g)
    e = errors(merged.view_as(out), out.float())
    assert e["max_abs"] <= 4e-3, e
    # any split count gives the same result within tolerance
    op2, lp2 = G.decode_split(q, kc, vc, kv, cu, max_rows=3, max_kv_len=12000, num_splits=1,
                              split_keys=12032)
    merged2 = G.lse_merge(op2, lp2, g)
    assert (merged2.float() - merged.float()).abs().max().item() <= 4e-3
    assert G.last_device_status() == 0


@pytest.mark.parametrize("Hq,Hkv,rows,kv", [(16, 2, [8, 32, 1], [3000, 9000, 129]),
                                         (24, 4, [11, 2], [4097, 700]),
                                         (64, 1, [2, 1], [1000, 5000])])
def test_tc_and_mma_split_paths_agree(Hq, Hkv, rows, kv):
    """Groups of more than 16 packed rows take the tcgen05 split kernel when the split size
    is a multiple of 128 and the mma.sync kernel otherwise: both match the oracle and
    each other."""
    x = S.make_decode(len(rows), Hq, Hkv, rows, kv, seed=sum(kv))
    q, kc, vc, g, kvd, cu = dev(x)
    mk = max(kv)
    outs = []
    for C in (1024, 1088):        # 1024 = 8 x 128: tcgen05; 1088 = 17 x 64: mma.sync
        S_ = (mk + C - 1) // C
        op, lp = G.decode_split(q, kc, vc, kvd, cu, max_rows=max(rows), max_kv_len=mk,
                                num_splits=S_, split_keys=C)
        outs.append(G.lse_merge(op, lp, g).view_as(q))
    assert G.last_device_status() == 0
    ref = oracle.decode(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache), to_f64(x.g),
                        x.kv_lens.tolist(), x.cu_rows.tolist())[0]
    for o in outs:
        assert_parity(o, ref, f"split path {Hq, Hkv, rows, kv}")
    e = errors(outs[0], outs[1].float())
    assert e["max_abs"] <= MAX_ABS and e["median_rel"] <= MEDIAN_REL, e


def test_tc_split_padded_last_tile_repeated():
    """The tcgen05 split zeroes the V rows past kv_len of a sequence's last tile
    before releasing P.  A split of four 128-key tiles whose last one is padded with
    NaN, run repeatedly: every partial stays finite and the result matches the
    oracle (the zeroing must wait for that tile to land, not an earlier one)."""
    x = S.make_decode(2, 16, 2, [1, 3], [21627, 4271], Lcap=8192 * 3, seed=27)
    q, kc, vc, g, kvd, cu = dev(x)
    C = 1280                      # split 3 of sequence 1 = keys 3840..4270, tiles 30..33
    S_ = (21627 + C - 1) // C
    ref = oracle.decode(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache), to_f64(x.g),
                        x.kv_lens.tolist(), x.cu_rows.tolist())[0]
    for _ in range(10):
        op, lp = G.decode_split(q, kc, vc, kvd, cu, max_rows=32, max_kv_len=21627,
                                num_splits=S_, split_keys=C)
        live = torch.isfinite(lp)
        assert torch.isfinite(op[live]).all()
        assert_parity(G.lse_merge(op, lp, g).view_as(q), ref, "padded last tile")
    assert G.last_device_status() == 0


def test_merge_against_oracle():
    """Random normalised parts, some empty (lse -inf, O full of NaN that must not be
    read)."""
    gen = torch.Generator().manual_seed(16)
    Sn, N = 7, 300
    o = torch.randn(Sn, N, 256, generator=gen)
    l = torch.randn(Sn, N, generator=gen) * 3
    empty = torch.rand(Sn, N, generator=gen) < 0.3
    l[empty] = float("-inf")
    o[empty] = float("nan")
    l[:, 5] = float("-inf")                          # a row with no key at all
    gate = (torch.randn(N, 256, generator=gen) * 2).to(torch.bfloat16)
    out, lse = G.lse_merge(o.to(DEV), l.to(DEV), gate.to(DEV), return_lse=True)
    r_out, r_lse = oracle.lse_merge(o.double().numpy(), l.double().numpy(), to_f64(gate))
    assert_parity(out, r_out, "merge")
    assert torch.all(out[5] == 0) and lse[5].item() == float("-inf")
    fin = np.isfinite(r_lse)
    np.testing.assert_allclose(to_f64(lse)[fin], r_lse[fin], rtol=0, atol=1e-5)


def test_merge_dropping_a_chunk_control():
    """Control: a merge that drops the last part must fail parity."""
    gen = torch.Generator().manual_seed(17)
    o = torch.randn(4, 64, 256, generator=gen)
    l = torch.randn(4, 64, generator=gen)
    out = G.lse_merge(o.to(DEV), l.to(DEV))
    bad, _ = oracle.lse_merge(o[:3].double().numpy(), l[:3].double().numpy())
    assert fails_parity(out, bad)


def test_empty_decode_is_noop():
    q = torch.empty(0, 8, 256, dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros(2, 2, 8, 256, dtype=torch.bfloat16, device=DEV)
    kv = torch.tensor([0, 0], dtype=torch.int32, device=DEV)
    cu = torch.tensor([0, 0, 0], dtype=torch.int32, device=DEV)
    out = G.decode(q, kc, kc, q, kv, cu, max_rows=1, max_kv_len=1)
    assert out.shape == (0, 8, 256)


def test_device_range_error_is_recorded():
    """A kv length beyond the cache is caught on the device: the sequence is skipped
    and the status word says so; the context stays usable."""
    x = S.make_decode(2, 8, 2, [1, 1], [10, 20], Lcap=32, seed=18)
    q, kc, vc, g, kv, cu = dev(x)
    kv_bad = torch.tensor([10, 40], dtype=torch.int32, device=DEV)
    G.decode(q, kc, vc, g, kv_bad, None, max_rows=1, max_kv_len=32)
    assert G.last_device_status() == 6
    assert G.last_device_status() == 0
    out = G.decode(q, kc, vc, g, kv, None, max_rows=1, max_kv_len=20)
    assert_parity(out, ref(x)[0], "after range error")


@pytest.mark.parametrize("Hq,Hkv,rows,kv", [(24, 4, [1, 1, 1, 1], [5000, 70, 12000, 900]),
                                         (16, 2, [8, 32, 1], [3000, 9000, 129])])
def test_one_call_decode_any_workspace_contents(Hq, Hkv, rows, kv):
    """The one-call decode launches its merge as a programmatic dependent of the split
    kernel (the merge waits for the split grid before reading the parts): on both
    split kernels, with a workspace full of 0xFF bytes (every part slot the merge
    reads must have been written), and called repeatedly, it gives the same bits as
    with a zeroed workspace."""
    x = S.make_decode(len(rows), Hq, Hkv, rows, kv, seed=sum(kv) + 7)
    q, kc, vc, g, kvd, cu = dev(x)
    B, T = len(rows), q.shape[0]
    need = G.decode_workspace_size(B, T, Hq, Hkv, max(rows), max(kv))
    ref = G.decode(q, kc, vc, g, kvd, cu, max_rows=max(rows), max_kv_len=max(kv),
                   workspace=torch.zeros(need, dtype=torch.uint8, device=DEV))
    ws = torch.full((need,), 255, dtype=torch.uint8, device=DEV)
    for _ in range(3):
        out = G.decode(q, kc, vc, g, kvd, cu, max_rows=max(rows), max_kv_len=max(kv),
                       workspace=ws)
        assert torch.equal(out, ref)
    assert G.last_device_status() == 0
    assert_parity(out, oracle.decode(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache),
                                     to_f64(x.g), x.kv_lens.tolist(), x.cu_rows.tolist())[0],
                  "one-call decode")


@pytest.mark.parametrize("lens", [
    [60000] + [1] * 40,                       # one sequence holds almost every key
    [1, 2, 3, 5, 8, 13, 21, 34, 55, 89, 144, 233, 377, 610, 987, 1597, 2584, 4181, 6765],
    [32] * 256,                               # the largest batch the balanced table takes
    [100, 7000] * 130,                        # 260 sequences: fixed splits instead
])
def test_balanced_shares_extreme_lengths(lens):
    """The one-call decode on the mma.sync path cuts all sequences' key tiles into equal
    shares per CTA; a share may span sequences and a sequence many shares (up to the
    part capacity).  Extreme length mixes against the oracle, with NaN cache padding."""
    B = len(lens)
    x = S.make_decode(B, 8, 2, [1] * B, lens, Lcap=max(lens) + 3, seed=B + max(lens))
    out, lse = run(x, lse=True, one_row=True)
    r_out, r_lse = ref(x)
    assert_parity(out, r_out, f"balanced {B} seqs")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)


@pytest.mark.parametrize("rows,lens", [
    ([8, 1, 32, 3], [24000, 9, 200, 3000]),          # one range dwarfs the rest
    ([16] * 12, [130 + 2777 * i for i in range(12)]), # a ladder over 12 sequences
    ([64, 2], [70, 64000]),                           # 64 rows over a short cache
])
def test_tcgen05_path_extreme_lengths(rows, lens):
    """Verify rows on the tcgen05 split kernel (more than 16 packed rows per group) with
    extreme length mixes, chain and tree masks, against the oracle."""
    B = len(rows)
    x = S.make_decode(B, 16, 2, rows, lens, Lcap=max(lens) + 5, seed=sum(lens) % 1000)
    out, lse = run(x, lse=True)
    r_out, r_lse = ref(x)
    assert_parity(out, r_out, f"tcgen05 path {rows}")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)
    masks = S.random_tree_masks(rows, 3)
    q, kc, vc, g, kvd, cu = dev(x)
    tm = torch.tensor([m - (1 << 64) if m >= 1 << 63 else m for m in masks], dtype=torch.int64,
                      device=DEV)
    t_out = G.verify_tree(q, kc, vc, g, kvd, cu, tm, max_rows=max(rows), max_kv_len=max(lens))
    assert G.last_device_status() == 0
    t_ref = oracle.decode_tree(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache), to_f64(x.g),
                               x.kv_lens.tolist(), x.cu_rows.tolist(), masks)[0]
    assert_parity(t_out, t_ref, f"tcgen05 path tree {rows}")
