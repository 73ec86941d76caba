"""gqa_attn_prefill_pair: the prefill computed by CTA pairs (tcgen05 .cta_group::2;
two CTAs of a cluster take two row tiles of a KV group and share every K/V tile).

Checked against the float64 oracle at the parity bar on shapes that cover an odd
number of row tiles (the last pair's second tile is empty), GQA 1 / 3 / 5 / 6 / 7 /
8 / 16 / 32 / 128, an offset, several batches, a gate-less call and lse; against
gqa_attn_prefill (the one-CTA form) within the same bar; and with NaN / Inf V values
at keys that some rows of a pair do not see (the cleaning pass in pair form), where
every element no planted value can reach keeps the clean run's bits and the
non-finite pattern is the oracle's."""
import numpy as np
import pytest
import torch

import gqa_head_gated_gb300 as G
import oracle
from synth import inputs as S
from tests.parity import assert_nonfinite_parity, assert_parity, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"

SHAPES = {
    "gqa6_odd_tiles": (1, 24, 4, 300, 0),      # 15 row tiles: the last pair has one
    "gqa1": (1, 4, 4, 300, 0),
    "gqa8_offset_b2": (2, 16, 2, 257, 143),
    "gqa16_short": (1, 16, 1, 9, 0),           # one row tile: its pair partner is empty
    "gqa6_one_key_tile": (1, 24, 4, 128, 0),
    # packings with empty MMA rows (128 not a multiple of GQA) and GQA 32 / 128
    "gqa3": (1, 6, 2, 260, 0),                 # R = 42, 126 packed rows
    "gqa5_offset": (1, 10, 2, 131, 60),        # R = 25, 125 packed rows
    "gqa7": (1, 7, 1, 200, 0),                 # R = 18, 126 packed rows
    "gqa32_b3": (3, 64, 2, 19, 5),             # R = 4
    "gqa128": (1, 128, 1, 37, 0),              # R = 1: 37 row tiles, 19 pairs
}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_pair_prefill_matches_oracle(name):
    B, Hq, Hkv, Lq, off = SHAPES[name]
    x = S.make_prefill(B, Hq, Hkv, Lq, Lkv=Lq + off, kv_offset=off, seed=21)
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    out, lse = G.prefill_pair(q, k, v, g, kv_offset=off, return_lse=True)
    assert G.last_device_status() == 0
    assert G.launch_log(1)[0]["kernel"] == "attn_pair_kernel<prefill,bf16>"
    ref, r_lse = oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g), kv_offset=off)
    assert_parity(out, ref, f"pair {name}")
    assert_parity(lse, r_lse, f"pair lse {name}", max_abs=2e-3, median_rel=1.0)
    one = G.prefill(q, k, v, g, kv_offset=off)
    assert_parity(out, to_f64(one), f"pair vs one-CTA {name}")


def test_pair_prefill_without_gate():
    x = S.make_prefill(1, 24, 4, 200, seed=22)
    q, k, v = (t.to(DEV) for t in (x.q, x.k, x.v))
    out = G.prefill_pair(q, k, v, None)
    assert G.last_device_status() == 0
    ref, _ = oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), None, kv_offset=0)
    assert_parity(out, ref, "pair, no gate")


def test_pair_prefill_nonfinite_values_at_partially_masked_keys():
    """NaN / Inf V elements at keys that some rows of a pair see and others do not
    (its diagonal spans both CTAs' rows), and one NaN K value: the cleaning pass."""
    B, Hq, Hkv, Lq, off = 1, 24, 4, 300, 64
    x = S.make_prefill(B, Hq, Hkv, Lq, Lkv=Lq + off, kv_offset=off, seed=23)
    q, g = x.q.to(DEV), x.g.to(DEV)
    clean = G.prefill_pair(q, x.k.to(DEV), x.v.to(DEV), g, kv_offset=off)
    plants = [("v", 0, 80, 3, float("nan")), ("v", 1, 100, 200, float("inf")),
              ("v", 2, 140, 128, float("-inf")), ("v", 3, 330, 255, float("nan")),
              ("k", 3, 200, 9, float("nan"))]
    for kind, gk, key, col, val in plants:
        (x.k if kind == "k" else x.v)[0, gk, key, col] = val
    out = G.prefill_pair(q, x.k.to(DEV), x.v.to(DEV), g, kv_offset=off)
    assert G.last_device_status() == 0
    ref, _ = oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g), kv_offset=off)
    assert not np.isfinite(ref).all()
    assert_nonfinite_parity(out, ref, "pair non-finite")
    gqa = Hq // Hkv
    aff = np.zeros((B, Hq, Lq, 256), dtype=bool)
    for kind, gk, key, col, _ in plants:
        for h in range(gk * gqa, (gk + 1) * gqa):
            rows = np.arange(Lq)[off + np.arange(Lq) >= key]
            if kind == "k":
                aff[0, h, rows, :] = True
            else:
                aff[0, h, rows, col] = True
    keep = torch.from_numpy(~aff).to(DEV)
    assert torch.equal(out[keep], clean[keep])


def test_pair_masked_future_keys_bit_exact():
    """Perturbing keys a row does not see (but later rows of its pair do) leaves that
    row bit for bit unchanged on CTA pairs too; 1000 rows put key 600 inside a pair."""
    x = S.make_prefill(1, 24, 4, 1000, seed=24)
    q, g = x.q.to(DEV), x.g.to(DEV)
    a = G.prefill_pair(q, x.k.to(DEV), x.v.to(DEV), g)
    x.k[:, :, 600:] = (x.k[:, :, 600:].float() * -3 + 1).to(torch.bfloat16)
    x.v[:, :, 600:] = (x.v[:, :, 600:].float() * 5).to(torch.bfloat16)
    b = G.prefill_pair(q, x.k.to(DEV), x.v.to(DEV), g)
    assert G.last_device_status() == 0
    assert torch.equal(a[:, :, :600], b[:, :, :600])
    assert not torch.equal(a[:, :, 600:], b[:, :, 600:])


def test_pair_long_prompt_routing_matches_oracle_sampled():
    """gqa_attn_prefill on a prompt long enough for CTA pairs (3000 rows at an offset of
    500 keys): sampled rows against the oracle, and the same bits as forcing the pair."""
    B, Hq, Hkv, Lq, off = 1, 16, 2, 3000, 500
    x = S.make_prefill(B, Hq, Hkv, Lq, Lkv=Lq + off, kv_offset=off, seed=25)
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    out = G.prefill(q, k, v, g, kv_offset=off)
    assert G.launch_log(1)[0]["kernel"] == "attn_pair_kernel<prefill,bf16>"
    forced = G.prefill_pair(q, k, v, g, kv_offset=off)
    assert torch.equal(out, forced)
    gen = np.random.default_rng(25)
    rows = [(0, int(h), int(i)) for h, i in zip(gen.integers(0, Hq, 48), gen.integers(0, Lq, 48))]
    rows += [(0, 0, 0), (0, Hq - 1, Lq - 1), (0, 3, 1535), (0, 9, 1536)]
    ref, _ = oracle.prefill(to_f64(x.q), to_f64(x.k), to_f64(x.v), to_f64(x.g), kv_offset=off,
                            rows=rows)
    got = torch.stack([out[b_, h, i] for b_, h, i in rows])
    assert_parity(got, ref, "routed pair, sampled rows")
