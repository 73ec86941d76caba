"""Pins for the float64 oracle: checks against things other than the oracle itself.

* brute force in 40-digit arithmetic on tiny inputs (tests/brute.py);
* a library routine (torch scaled_dot_product_attention in float64, explicit
  boolean mask, GQA by repeat_interleave);
* closed forms: one visible key, G = 0 halves the output, a large gate passes it
  through, equal keys give the mean of the visible values, a dominant score picks
  its value row;
* invariants: masked and padded keys never change a row, chunked prefill equals
  whole prefill, verify rows equal prefill rows at the same positions, head
  chunks equal the unchunked group, an LSE merge of any key partition equals the
  unsplit row;
* the head-chunk plan against the worked example the DS4Server issue113 README
  prints (tests/golden/head_chunk_plan.txt);
* non-finite inputs (the TensorFold attention contract's gate 1 plants them and
  compares with float64): what IEEE arithmetic of the formula fixes -- a NaN
  query row is NaN, an Inf value under a positive probability is Inf in that
  column only, an Inf score poisons exactly the rows whose score is +Inf and
  drops the key where it is -Inf (checked by brute force over the other keys),
  a -Inf gate gives 0, a NaN merge part gives a NaN row, non-finite values
  in positions no row sees change nothing, and non-finite K/V of a key that
  earlier rows of the call do not see and later rows do leave the earlier rows
  bitwise unchanged (excluded, not weighted by 0) while the later rows carry the
  IEEE result;
* general masks: brute force over the kept keys (bool) and with exact biases
  (additive), torch's scaled_dot_product_attention with bool and float masks,
  2-D == expanded 4-D, all-True + causal == prefill, additive -inf == False, a
  row shift moves only lse, chunk-local == tiled full-head, and the accept /
  reject table of mask head counts derived from the DS4Server README's rule
  (tests/golden/mask_head_rules.txt).

Each check is a function returning an error string (empty when it holds) so that
test_oracle_mutants.py can run the same checks against oracles with planted
mistakes.
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from synth import make_decode, make_prefill
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(t):
    return t.to(torch.float64).numpy()


def _cmp(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return f"{what}: shape {a.shape} vs {b.shape}"
    if not np.all(np.isfinite(a) == np.isfinite(b)):
        return f"{what}: finiteness differs"
    fin = np.isfinite(a)
    if not fin.any():
        return ""
    err = np.max(np.abs(a[fin] - b[fin]) / np.maximum(1.0, np.abs(b[fin])))
    return "" if err <= tol else f"{what}: max err {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------------------
# checks (each takes the oracle module so mutants can be substituted)
# ---------------------------------------------------------------------------

def check_brute_prefill(ora):
    x = make_prefill(2, 4, 2, 4, Lkv=7, kv_offset=3, seed=11)
    Q, K, V, G = (f64(t) for t in (x.q, x.k, x.v, x.g))
    out, lse = ora.prefill(Q, K, V, G, kv_offset=3)
    ref = brute.prefill(Q, K, V, G, 3)
    for (b, h, i), (o, l) in ref.items():
        e = _cmp(out[b, h, i], [float(v) for v in o], 1e-12, f"prefill out {(b, h, i)}")
        e = e or _cmp(lse[b, h, i], float(l), 1e-12, f"prefill lse {(b, h, i)}")
        if e:
            return e
    return ""


def check_brute_prefill_ungated(ora):
    x = make_prefill(1, 2, 1, 3, seed=12)
    Q, K, V = (f64(t) for t in (x.q, x.k, x.v))
    out, _ = ora.prefill(Q, K, V, None, kv_offset=0)
    ref = brute.prefill(Q, K, V, None, 0)
    for (b, h, i), (o, _) in ref.items():
        e = _cmp(out[b, h, i], [float(v) for v in o], 1e-12, f"ungated {(b, h, i)}")
        if e:
            return e
    return ""


def check_brute_decode(ora):
    # ragged rows (0 rows for one sequence), NaN cache padding, GQA 2
    x = make_decode(3, 4, 2, rows=[1, 0, 3], kv_lens=[5, 2, 6], Lcap=8, seed=13)
    Q, Kc, Vc, G = (f64(t) for t in (x.q, x.k_cache, x.v_cache, x.g))
    out, lse = ora.decode(Q, Kc, Vc, G, x.kv_lens.tolist(), x.cu_rows.tolist())
    ref = brute.decode(Q, Kc, Vc, G, x.kv_lens.tolist(), x.rows)
    for (t, h), (o, l) in ref.items():
        e = _cmp(out[t, h], [float(v) for v in o], 1e-12, f"decode out {(t, h)}")
        e = e or _cmp(lse[t, h], float(l), 1e-12, f"decode lse {(t, h)}")
        if e:
            return e
    return ""


def check_library_sdpa(ora):
    """torch SDPA in float64 with an explicit causal/offset boolean mask."""
    B, Hq, Hkv, Lq, off = 2, 6, 2, 9, 5
    x = make_prefill(B, Hq, Hkv, Lq, kv_offset=off, seed=14)
    q, k, v, g = (t.to(torch.float64) for t in (x.q, x.k, x.v, x.g))
    Lkv = off + Lq
    mask = torch.arange(Lkv)[None, :] <= (off + torch.arange(Lq))[:, None]
    kk = k.repeat_interleave(Hq // Hkv, dim=1)
    vv = v.repeat_interleave(Hq // Hkv, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=mask,
                                                           scale=1.0 / 16.0)
    ref = (ref * torch.sigmoid(g)).numpy()
    out, _ = ora.prefill(q.numpy(), k.numpy(), v.numpy(), g.numpy(), kv_offset=off)
    return _cmp(out, ref, 1e-12, "sdpa")


def check_one_key(ora):
    """Lkv = 1: out = V0 * sigmoid(G), lse = the single score."""
    x = make_prefill(1, 3, 1, 1, seed=15)
    Q, K, V, G = (f64(t) for t in (x.q, x.k, x.v, x.g))
    out, lse = ora.prefill(Q, K, V, G, 0)
    want = V[0, 0, 0][None, :] / (1.0 + np.exp(-G[0, :, 0]))
    s = (Q[0, :, 0] @ K[0, 0, 0]) / 16.0
    return _cmp(out[0, :, 0], want, 1e-15, "one key") or _cmp(lse[0, :, 0], s, 1e-15, "one key lse")


def check_gate_zero_half(ora):
    """G = 0: sigmoid(0) = 1/2 exactly, so the output is exactly half the ungated one."""
    x = make_prefill(1, 4, 2, 6, seed=16)
    Q, K, V = (f64(t) for t in (x.q, x.k, x.v))
    gated, _ = ora.prefill(Q, K, V, np.zeros_like(Q), 0)
    plain, _ = ora.prefill(Q, K, V, None, 0)
    return "" if np.array_equal(gated, plain * 0.5) else "G=0 is not half"


def check_gate_large_passthrough(ora):
    """G = +40: sigmoid rounds to 1 in float64; G = -40: the output is ~4e-18 of it."""
    x = make_prefill(1, 4, 2, 6, seed=17)
    Q, K, V = (f64(t) for t in (x.q, x.k, x.v))
    plain, _ = ora.prefill(Q, K, V, None, 0)
    hi, _ = ora.prefill(Q, K, V, np.full_like(Q, 40.0), 0)
    lo, _ = ora.prefill(Q, K, V, np.full_like(Q, -40.0), 0)
    e = _cmp(hi, plain, 1e-15, "G=+40")
    if e:
        return e
    return "" if np.max(np.abs(lo)) <= 1e-16 * max(1.0, np.max(np.abs(plain))) else "G=-40 not ~0"


def check_equal_keys_mean(ora):
    """All keys equal: every visible key has the same score, out = mean of the
    visible V rows times the gate."""
    x = make_prefill(1, 2, 1, 5, Lkv=8, kv_offset=3, seed=18)
    Q, K, V, G = (f64(t) for t in (x.q, x.k, x.v, x.g))
    K[:] = K[:, :, :1]
    out, _ = ora.prefill(Q, K, V, G, 3)
    for h in range(2):
        for i in range(5):
            want = V[0, 0, :3 + i + 1].mean(axis=0) / (1.0 + np.exp(-G[0, h, i]))
            e = _cmp(out[0, h, i], want, 1e-14, f"equal keys {(h, i)}")
            if e:
                return e
    return ""


def check_dominant_key(ora):
    """A key whose score exceeds the others by ~1000 (exp would overflow without
    the max shift) picks its V row exactly."""
    x = make_prefill(1, 1, 1, 1, Lkv=6, kv_offset=5, seed=19)
    Q, K, V, G = (f64(t) for t in (x.q, x.k, x.v, x.g))
    Q[:] = 0.0
    Q[0, 0, 0, 0] = 16.0 * 1000.0
    K[:] = 0.0
    K[0, 0, 3, 0] = 1.0                 # score 1000 for key 3, 0 for the rest
    out, lse = ora.prefill(Q, K, V, None, 5)
    e = _cmp(out[0, 0, 0], V[0, 0, 3], 1e-15, "dominant key")
    return e or _cmp(lse[0, 0, 0], 1000.0, 1e-15, "dominant lse")


def check_masked_keys_ignored(ora):
    """Keys a row does not see (future keys, cache padding) never change it: bit
    for bit under finite perturbation of future keys and NaN padding."""
    x = make_prefill(1, 4, 2, 10, Lkv=14, kv_offset=2, seed=20)
    Q, K, V, G = (f64(t) for t in (x.q, x.k, x.v, x.g))
    base, _ = ora.prefill(Q, K, V, G, 2)
    K2, V2 = K.copy(), V.copy()
    K2[:, :, 8:] += 3.0                 # keys 8..13: rows 0..5 do not see them
    V2[:, :, 8:] *= -7.0
    K2[:, :, 12:] = np.nan              # keys 12, 13: no row sees them
    V2[:, :, 12:] = np.inf
    pert, _ = ora.prefill(Q, K2, V2, G, 2)
    if not np.array_equal(base[:, :, :6], pert[:, :, :6]):
        return "masked future keys changed a row"
    y = make_decode(2, 4, 2, rows=[2, 1], kv_lens=[5, 3], Lcap=9, seed=21, pad_value=0.0)
    Qd, Kd, Vd, Gd = (f64(t) for t in (y.q, y.k_cache, y.v_cache, y.g))
    a, _ = ora.decode(Qd, Kd, Vd, Gd, [5, 3], y.cu_rows.tolist())
    Kd[0, :, 5:] = np.nan
    Vd[1, :, 3:] = np.nan
    b, _ = ora.decode(Qd, Kd, Vd, Gd, [5, 3], y.cu_rows.tolist())
    return "" if np.array_equal(a, b) else "cache padding changed a row"


def check_chunked_prefill(ora):
    """Any chunking of the prompt rows with kv_offset equals the whole prompt."""
    x = make_prefill(1, 4, 2, 12, seed=22)
    Q, K, V, G = (f64(t) for t in (x.q, x.k, x.v, x.g))
    whole, wl = ora.prefill(Q, K, V, G, 0)
    for c0, c1 in [(0, 5), (5, 6), (6, 12)]:
        part, pl = ora.prefill(Q[:, :, c0:c1], K[:, :, :c1], V[:, :, :c1], G[:, :, c0:c1], c0)
        e = _cmp(part, whole[:, :, c0:c1], 1e-13, f"chunk {c0}:{c1}")
        e = e or _cmp(pl, wl[:, :, c0:c1], 1e-13, f"chunk lse {c0}:{c1}")
        if e:
            return e
    return ""


def check_verify_equals_prefill(ora):
    """r verify rows at kv_len are prompt rows at kv_offset = kv_len - r."""
    r, L = 4, 9
    y = make_decode(1, 4, 2, rows=[r], kv_lens=[L], Lcap=11, seed=23)
    Qd, Kd, Vd, Gd = (f64(t) for t in (y.q, y.k_cache, y.v_cache, y.g))
    dec, dl = ora.decode(Qd, Kd, Vd, Gd, [L], [0, r])
    pre, pl = ora.prefill(Qd.transpose(1, 0, 2)[None], Kd[:, :, :L], Vd[:, :, :L],
                          Gd.transpose(1, 0, 2)[None], L - r)
    return (_cmp(dec, pre[0].transpose(1, 0, 2), 1e-13, "verify vs prefill")
            or _cmp(dl, pl[0].T, 1e-13, "verify vs prefill lse"))


def check_head_chunks(ora):
    """Head-chunked evaluation (chunks of min(GQA, 32/rows), remainder kept) equals
    the unchunked group.  rows*GQA = 4*12 > 32 gives chunks 8 + 4."""
    y = make_decode(2, 24, 2, rows=[4, 2], kv_lens=[9, 6], Lcap=10, seed=24)
    Qd, Kd, Vd, Gd = (f64(t) for t in (y.q, y.k_cache, y.v_cache, y.g))
    a, al = ora.decode(Qd, Kd, Vd, Gd, [9, 6], y.cu_rows.tolist())
    b, bl = ora.decode_head_chunked(Qd, Kd, Vd, Gd, [9, 6], y.cu_rows.tolist())
    return _cmp(b, a, 1e-13, "head chunks") or _cmp(bl, al, 1e-13, "head chunks lse")


def check_merge_partition(ora):
    """An LSE merge of the parts of any key partition equals the unsplit row."""
    y = make_decode(1, 4, 2, rows=[3], kv_lens=[23], Lcap=23, seed=25)
    Qd, Kd, Vd, Gd = (f64(t) for t in (y.q, y.k_cache, y.v_cache, y.g))
    full, fl = ora.decode(Qd, Kd, Vd, Gd, [23], [0, 3])
    cuts = [0, 4, 5, 13, 21, 30]        # the last part is empty for every row
    N = 3 * 4
    parts = np.zeros((len(cuts) - 1, N, 256))
    lses = np.zeros((len(cuts) - 1, N))
    for s in range(len(cuts) - 1):
        a, b = cuts[s], cuts[s + 1]
        for t in range(3):
            lim = ora.verify_visible(t, 3, 23)
            n_keys = max(0, min(b, lim) - a)
            for h in range(4):
                g = ora.kv_head_of(h, 4, 2)
                o, l = ora.attend_rows(Qd[t, h][None], Kd[0, g, a:], Vd[0, g, a:], None, [n_keys])
                parts[s, t * 4 + h] = o[0]
                lses[s, t * 4 + h] = l[0]
    out, lse = ora.lse_merge(parts, lses, Gd.reshape(N, 256))
    return (_cmp(out, full.reshape(N, 256), 1e-12, "merge")
            or _cmp(lse, fl.reshape(N), 1e-12, "merge lse"))


def check_merge_empty_row(ora):
    """A row whose parts are all empty is zeros with lse -inf; an empty part among
    live ones carries weight 0 even when its O holds NaN."""
    parts = np.zeros((3, 2, 256))
    parts[1, 1] = np.nan
    lses = np.array([[-np.inf, 0.5], [-np.inf, -np.inf], [-np.inf, 0.5]])
    parts[0, 1] = 1.0
    parts[2, 1] = 3.0
    out, lse = ora.lse_merge(parts, lses)
    if not (np.all(out[0] == 0) and lse[0] == -np.inf):
        return "empty row"
    e = _cmp(out[1], np.full(256, 2.0), 1e-15, "equal weights")
    return e or _cmp(lse[1], 0.5 + math.log(2.0), 1e-15, "equal weights lse")


def _load_plan_golden():
    cases = []
    with open(os.path.join(GOLDEN, "head_chunk_plan.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            rows, gqa, plan = line.split(None, 2)
            cases.append((int(rows), int(gqa), [int(c) for c in plan.split(",")]))
    return cases


def check_plan_golden(ora):
    for rows, gqa, plan in _load_plan_golden():
        got = ora.head_chunk_plan(rows, gqa)
        if got != plan:
            return f"plan({rows},{gqa}) = {got}, page says {plan}"
    return ""


def _tree_masks(rows, seed):
    """Random token trees: new row i's parent is a random earlier row (or none);
    the mask holds the row and its ancestors."""
    rng = np.random.default_rng(seed)
    masks = []
    for r in rows:
        anc = []
        for i in range(r):
            par = int(rng.integers(-1, i)) if i else -1
            m = (1 << i) | (anc[par] if par >= 0 else 0)
            anc.append(m)
            masks.append(m)
    return masks


def check_brute_tree(ora):
    x = make_decode(2, 4, 2, rows=[4, 3], kv_lens=[7, 5], Lcap=8, seed=31)
    Q, Kc, Vc, G = (f64(t) for t in (x.q, x.k_cache, x.v_cache, x.g))
    masks = _tree_masks([4, 3], 5)
    masks[1] = 0b10                                  # a row that does not see row 0
    out, lse = ora.decode_tree(Q, Kc, Vc, G, x.kv_lens.tolist(), x.cu_rows.tolist(), masks)
    ref = brute.decode_tree(Q, Kc, Vc, G, x.kv_lens.tolist(), [4, 3], masks)
    for (t, h), (o, l) in ref.items():
        e = _cmp(out[t, h], [float(v) for v in o], 1e-12, f"tree out {(t, h)}")
        e = e or _cmp(lse[t, h], float(l), 1e-12, f"tree lse {(t, h)}")
        if e:
            return e
    return ""


def check_tree_chain_is_decode(ora):
    """Chain masks (row i sees new rows 0..i) give the chain-verify result."""
    y = make_decode(3, 8, 2, rows=[3, 1, 5], kv_lens=[9, 4, 12], Lcap=13, seed=32)
    Q, Kc, Vc, G = (f64(t) for t in (y.q, y.k_cache, y.v_cache, y.g))
    a, al = ora.decode(Q, Kc, Vc, G, y.kv_lens.tolist(), y.cu_rows.tolist())
    b, bl = ora.decode_tree(Q, Kc, Vc, G, y.kv_lens.tolist(), y.cu_rows.tolist(),
                            ora.chain_masks([3, 1, 5]))
    return _cmp(b, a, 1e-13, "chain tree") or _cmp(bl, al, 1e-13, "chain tree lse")


def check_tree_storage_permutation(ora):
    """Storing the new rows' keys in another order, with the mask bits renamed to
    match, changes no output: only the visible set matters."""
    r, L = 5, 11
    y = make_decode(1, 4, 1, rows=[r], kv_lens=[L], Lcap=L, seed=33)
    Q, Kc, Vc, G = (f64(t) for t in (y.q, y.k_cache, y.v_cache, y.g))
    masks = _tree_masks([r], 7)
    a, _ = ora.decode_tree(Q, Kc, Vc, G, [L], [0, r], masks)
    perm = [3, 0, 4, 1, 2]                           # new row k stored at slot perm[k]
    base = L - r
    K2, V2 = Kc.copy(), Vc.copy()
    for k in range(r):
        K2[0, :, base + perm[k]] = Kc[0, :, base + k]
        V2[0, :, base + perm[k]] = Vc[0, :, base + k]
    m2 = [sum(1 << perm[k] for k in range(r) if (m >> k) & 1) for m in masks]
    b, _ = ora.decode_tree(Q, K2, V2, G, [L], [0, r], m2)
    return _cmp(b, a, 1e-12, "tree permutation")


def check_kv_append_brute(ora):
    """Append against an element-by-element loop; rows already in the cache, other
    sequences and positions past the new rows are untouched."""
    rng = np.random.default_rng(41)
    B, Hkv, Lcap, D = 3, 2, 12, 256
    Kc = rng.standard_normal((B, Hkv, Lcap, D))
    Vc = rng.standard_normal((B, Hkv, Lcap, D))
    rows, lens = [2, 0, 3], [4, 7, 9]
    cu = [0, 2, 2, 5]
    Kn = rng.standard_normal((5, Hkv, D))
    Vn = rng.standard_normal((5, Hkv, D))
    K2, V2 = ora.kv_append(Kc, Vc, Kn, Vn, lens, cu)
    for b in range(B):
        for g in range(Hkv):
            for pos in range(Lcap):
                i = pos - lens[b]
                if 0 <= i < rows[b]:
                    wk, wv = Kn[cu[b] + i, g], Vn[cu[b] + i, g]
                else:
                    wk, wv = Kc[b, g, pos], Vc[b, g, pos]
                if not (np.array_equal(K2[b, g, pos], wk) and np.array_equal(V2[b, g, pos], wv)):
                    return f"append wrong at {(b, g, pos)}"
    return ""


def check_kv_keep_brute(ora):
    """Keep against an element-by-element loop, including keeping every row (no
    change), keeping none, and a kept set whose destinations overlap its sources."""
    rng = np.random.default_rng(42)
    B, Hkv, Lcap, D = 3, 2, 16, 256
    Kc = rng.standard_normal((B, Hkv, Lcap, D))
    Vc = rng.standard_normal((B, Hkv, Lcap, D))
    lens, cu = [10, 6, 15], [0, 5, 6, 12]
    keep = [[1, 2, 4], [], [0, 1, 2, 3, 4, 5]]
    K2, V2, nl = ora.kv_keep(Kc, Vc, lens, cu, keep)
    for b in range(B):
        r = cu[b + 1] - cu[b]
        base = lens[b] - r
        if nl[b] != base + len(keep[b]):
            return "kept length"
        for g in range(Hkv):
            for pos in range(Lcap):
                k = pos - base
                src = base + keep[b][k] if 0 <= k < len(keep[b]) else pos
                if not (np.array_equal(K2[b, g, pos], Kc[b, g, src]) and
                        np.array_equal(V2[b, g, pos], Vc[b, g, src])):
                    return f"keep wrong at {(b, g, pos)}"
    return ""


def check_append_then_chain_verify(ora):
    """Appending the new rows' K/V and running chain verify equals attending over the
    old keys plus the new rows' own keys: the append lands where verify reads."""
    y = make_decode(1, 4, 2, rows=[3], kv_lens=[8], Lcap=8, seed=43)
    Q, Kc, Vc, G = (f64(t) for t in (y.q, y.k_cache, y.v_cache, y.g))
    Kn, Vn = Kc[0, :, 5:8].swapaxes(0, 1).copy(), Vc[0, :, 5:8].swapaxes(0, 1).copy()
    blank_k, blank_v = Kc.copy(), Vc.copy()
    blank_k[:, :, 5:] = 0.0
    blank_v[:, :, 5:] = 0.0
    K2, V2 = ora.kv_append(blank_k, blank_v, Kn, Vn, [5], [0, 3])
    a, _ = ora.decode(Q, K2, V2, G, [8], [0, 3])
    b, _ = ora.decode(Q, Kc, Vc, G, [8], [0, 3])
    return "" if np.array_equal(a, b) else "append then verify differs"


# ---------------------------------------------------------------------------
# non-finite inputs
# ---------------------------------------------------------------------------

def _same_except(a, b, mask):
    """a equals b bit for bit outside `mask` (a boolean array of a's shape)."""
    return np.array_equal(np.where(mask, 0.0, a), np.where(mask, 0.0, b))


def check_nonfinite_q_row(ora):
    """A NaN query row gives NaN out and lse for that row; other rows unchanged."""
    x = make_prefill(1, 4, 2, 6, Lkv=9, kv_offset=3, seed=40)
    Q, K, V, G = (f64(t) for t in (x.q, x.k, x.v, x.g))
    a, la = ora.prefill(Q, K, V, G, 3)
    Q[0, 1, 2, 7] = np.nan
    b, lb = ora.prefill(Q, K, V, G, 3)
    if not (np.isnan(b[0, 1, 2]).all() and np.isnan(lb[0, 1, 2])):
        return "NaN query row is not NaN"
    m = np.zeros(a.shape, bool)
    m[0, 1, 2] = True
    return "" if _same_except(b, a, m) else "NaN query row changed another row"


def check_nonfinite_v_column(ora):
    """+Inf and -Inf in two columns of a key every row sees: every row of the KV
    group is +Inf / -Inf in exactly those columns (p > 0, gate > 0); NaN in a
    third column is NaN there; other heads and columns are unchanged."""
    x = make_prefill(1, 4, 2, 5, Lkv=8, kv_offset=3, seed=41)
    Q, K, V, G = (f64(t) for t in (x.q, x.k, x.v, x.g))
    a, la = ora.prefill(Q, K, V, G, 3)
    V[0, 1, 0, 10] = np.inf
    V[0, 1, 2, 20] = -np.inf
    V[0, 1, 1, 30] = np.nan
    b, lb = ora.prefill(Q, K, V, G, 3)
    grp = b[0, 2:4]                        # heads 2, 3 read KV head 1
    if not (np.all(grp[..., 10] == np.inf) and np.all(grp[..., 20] == -np.inf)
            and np.all(np.isnan(grp[..., 30]))):
        return "Inf/NaN value column did not propagate"
    m = np.zeros(a.shape, bool)
    m[0, 2:4, :, [10, 20, 30]] = True
    if not _same_except(b, a, m):
        return "Inf value changed other columns"
    return "" if np.array_equal(la, lb) else "Inf value changed lse"


def check_nonfinite_k_sign(ora):
    """K[key 0, d] = +Inf: rows whose q_d > 0 score +Inf (NaN row); rows with
    q_d < 0 score -Inf on key 0, which drops out -- checked by brute force over
    keys 1..lim."""
    y = make_decode(1, 4, 2, rows=[3], kv_lens=[6], Lcap=8, seed=42, pad_value=0.0)
    Q, Kc, Vc, G = (f64(t) for t in (y.q, y.k_cache, y.v_cache, y.g))
    d = 5
    Kc[0, :, 0, d] = np.inf
    out, lse = ora.decode(Q, Kc, Vc, G, [6], [0, 3])
    seen_neg = 0
    for t in range(3):
        lim = 6 - 3 + t + 1
        for h in range(4):
            g = h // 2
            if Q[t, h, d] > 0:
                if not (np.isnan(out[t, h]).all() and np.isnan(lse[t, h])):
                    return "+Inf score did not give a NaN row"
            else:
                seen_neg += 1
                o, l = brute._row(Q[t, h], [Kc[0, g, j] for j in range(1, lim)],
                                  [Vc[0, g, j] for j in range(1, lim)], G[t, h])
                e = _cmp(out[t, h], [float(v) for v in o], 1e-13, "-Inf score drops key")
                if e:
                    return e
    return "" if seen_neg else "no row with q_d < 0 (pick another seed)"


def check_nonfinite_k_nan(ora):
    """A NaN in key 1 makes every row that sees key 1 NaN (its score is NaN);
    row 0 of a prompt from position 0 does not see it and is unchanged."""
    x = make_prefill(1, 2, 1, 4, seed=46)
    Q, K, V, G = (f64(t) for t in (x.q, x.k, x.v, x.g))
    a, _ = ora.prefill(Q, K, V, G, 0)
    K[0, 0, 1, 100] = np.nan
    b, lb = ora.prefill(Q, K, V, G, 0)
    if not np.array_equal(a[:, :, 0], b[:, :, 0]):
        return "NaN key changed a row that does not see it"
    return "" if np.isnan(b[:, :, 1:]).all() and np.isnan(lb[:, :, 1:]).all() else "NaN key"


def check_nonfinite_gate(ora):
    """Gate -Inf gives exactly 0, +Inf passes the attention through, NaN is NaN."""
    x = make_prefill(1, 2, 1, 3, seed=43)
    Q, K, V, G = (f64(t) for t in (x.q, x.k, x.v, x.g))
    plain, _ = ora.prefill(Q, K, V, None, 0)
    G[0, 0, 1, 3] = -np.inf
    G[0, 0, 1, 4] = np.inf
    G[0, 1, 2, 5] = np.nan
    out, _ = ora.prefill(Q, K, V, G, 0)
    if out[0, 0, 1, 3] != 0.0 or out[0, 0, 1, 4] != plain[0, 0, 1, 4]:
        return "infinite gate"
    return "" if np.isnan(out[0, 1, 2, 5]) else "NaN gate"


def check_nonfinite_unseen(ora):
    """NaN/Inf in K and V positions no row sees (prompt keys past the last row,
    cache rows past kv_len) and in K of keys masked for a row change nothing in
    the rows that do not see them."""
    x = make_prefill(1, 4, 2, 6, Lkv=12, kv_offset=2, seed=44)
    Q, K, V, G = (f64(t) for t in (x.q, x.k, x.v, x.g))
    a, _ = ora.prefill(Q, K, V, G, 2)
    K[:, :, 8:] = np.nan                  # positions 8..11: past the last row (7)
    V[:, :, 8:] = -np.inf
    K[:, 0, 6, 0] = np.inf                # key 6: rows 4, 5 see it
    b, _ = ora.prefill(Q, K, V, G, 2)
    if not np.array_equal(a[:, :, :4], b[:, :, :4]) or not np.array_equal(a[:, 2:], b[:, 2:]):
        return "unseen non-finite keys changed a row"
    y = make_decode(2, 4, 2, rows=[2, 1], kv_lens=[5, 3], Lcap=9, seed=45, pad_value=np.inf)
    Qd, Kd, Vd, Gd = (f64(t) for t in (y.q, y.k_cache, y.v_cache, y.g))
    c, _ = ora.decode(Qd, Kd, Vd, Gd, [5, 3], y.cu_rows.tolist())
    Kd[0, :, 5:] = np.nan
    Vd[1, :, 3:] = -np.inf
    e, _ = ora.decode(Qd, Kd, Vd, Gd, [5, 3], y.cu_rows.tolist())
    return "" if np.array_equal(c, e) and np.isfinite(c).all() else "cache padding changed a row"


def _expect_rows(a, la, b, lb, spec, what):
    """Row-by-row comparison of a planted run (b, lb) with the clean run (a, la).
    spec(idx) is None (the row and its lse are bitwise unchanged), "nan" (out and
    lse NaN), or {column: "nan" | "+inf" | "-inf"} (those columns so, every other
    column and the lse bitwise unchanged)."""
    kinds = {"nan": np.isnan, "+inf": lambda v: v == np.inf, "-inf": lambda v: v == -np.inf}
    for idx in np.ndindex(*la.shape):
        want = spec(idx)
        if want is None:
            if not (np.array_equal(a[idx], b[idx]) and la[idx] == lb[idx]):
                return f"{what}: row {idx} changed by a key it does not see"
        elif want == "nan":
            if not (np.isnan(b[idx]).all() and np.isnan(lb[idx])):
                return f"{what}: row {idx} is not NaN"
        else:
            for c, kind in want.items():
                if not kinds[kind](b[idx][c]):
                    return f"{what}: row {idx} column {c} is {b[idx][c]}, want {kind}"
            rest = np.ones(a.shape[-1], bool)
            rest[list(want)] = False
            if not (np.array_equal(a[idx][rest], b[idx][rest]) and la[idx] == lb[idx]):
                return f"{what}: row {idx} changed outside the planted columns"
    return ""


def check_nonfinite_masked_kv(ora):
    """NaN, +Inf and -Inf in the V rows (and NaN in a K row) of keys that earlier
    rows of the same call do not see and later rows do, in a prompt chunk at an
    offset and in a chain-verify block.  Keys a row does not see are excluded from
    its sums, so that row equals the clean run bit for bit (a probability-0
    product would make it NaN); a row that sees a planted V value is NaN / +Inf /
    -Inf in exactly that column (probability > 0, gate > 0) and bitwise unchanged
    elsewhere; a row that sees the NaN key is NaN.  Every row evaluated alone
    (rows=) gives the block evaluation's bits."""
    x = make_prefill(1, 4, 2, 6, Lkv=9, kv_offset=3, seed=47)
    Q, K, V, G = (f64(t) for t in (x.q, x.k, x.v, x.g))
    a, la = ora.prefill(Q, K, V, G, 3)            # row i sees keys 0 .. 3 + i
    V[0, 0, 5, 7] = np.nan                        # KV head 0: key 5 seen by rows 2..5
    V[0, 0, 6, 8] = np.inf                        # key 6: rows 3..5
    V[0, 0, 8, 9] = -np.inf                       # key 8: row 5 only
    V[0, 1, 4, 10] = np.inf                       # KV head 1: key 4 seen by rows 1..5
    K[0, 1, 7, 3] = np.nan                        # key 7: rows 4, 5 score NaN
    b, lb = ora.prefill(Q, K, V, G, 3)

    def pre_spec(idx):
        _, h, i = idx
        if h < 2:
            cols = {c: k for c, k, first in ((7, "nan", 2), (8, "+inf", 3), (9, "-inf", 5))
                    if i >= first}
            return cols or None
        if i >= 4:
            return "nan"
        return {10: "+inf"} if i >= 1 else None

    e = _expect_rows(a, la, b, lb, pre_spec, "prefill chunk")
    if e:
        return e
    rows = [(0, h, i) for h in range(4) for i in range(6)]
    c, lc = ora.prefill(Q, K, V, G, 3, rows=rows)
    for n, idx in enumerate(rows):
        if not (np.array_equal(c[n], b[idx], equal_nan=True) and
                np.array_equal(lc[n], lb[idx], equal_nan=True)):
            return f"prefill row {idx} alone differs from the block"

    y = make_decode(1, 4, 2, rows=[4], kv_lens=[9], Lcap=10, seed=48, pad_value=0.0)
    Qd, Kd, Vd, Gd = (f64(t) for t in (y.q, y.k_cache, y.v_cache, y.g))
    a, la = ora.decode(Qd, Kd, Vd, Gd, [9], [0, 4])   # row t sees keys 0 .. 5 + t
    Vd[0, 0, 6, 20] = -np.inf                     # KV head 0: key 6 seen by rows 1..3
    Kd[0, 0, 7, 30] = np.nan                      # key 7: rows 2, 3 score NaN
    Vd[0, 1, 7, 22] = np.inf                      # KV head 1: key 7 seen by rows 2, 3
    Vd[0, 1, 8, 21] = np.nan                      # key 8: row 3 only
    b, lb = ora.decode(Qd, Kd, Vd, Gd, [9], [0, 4])

    def dec_spec(idx):
        t, h = idx
        if h < 2:
            return None if t == 0 else {20: "-inf"} if t == 1 else "nan"
        cols = {c: k for c, k, first in ((22, "+inf", 2), (21, "nan", 3)) if t >= first}
        return cols or None

    e = _expect_rows(a, la, b, lb, dec_spec, "chain verify")
    if e:
        return e
    rows = [(t, h) for t in range(4) for h in range(4)]
    c, lc = ora.decode(Qd, Kd, Vd, Gd, [9], [0, 4], rows=rows)
    for n, idx in enumerate(rows):
        if not (np.array_equal(c[n], b[idx], equal_nan=True) and
                np.array_equal(lc[n], lb[idx], equal_nan=True)):
            return f"verify row {idx} alone differs from the block"
    return ""


def check_nonfinite_merge(ora):
    """A NaN part makes its row NaN (out and lse); a -inf part with NaN O is not
    read; +Inf lse gives NaN (exp(Inf - Inf))."""
    parts = np.ones((3, 3, 256))
    lses = np.array([[0.1, 0.2, 0.3], [np.nan, -np.inf, np.inf], [0.5, 0.5, 0.5]])
    parts[1, 1] = np.nan
    out, lse = ora.lse_merge(parts, lses)
    if not (np.isnan(out[0]).all() and np.isnan(lse[0])):
        return "NaN part did not poison its row"
    if not (np.all(out[1] == 1.0) and np.isfinite(lse[1])):
        return "-inf part was read"
    return "" if np.isnan(out[2]).all() and np.isnan(lse[2]) else "+Inf lse"


# ---------------------------------------------------------------------------
# general masks (dense SDPA consumer)
# ---------------------------------------------------------------------------

def _mask_case(seed, B=1, Hq=4, Hkv=2, Lq=3, Lkv=6):
    x = make_prefill(B, Hq, Hkv, Lq, Lkv=Lkv, kv_offset=Lkv - Lq, seed=seed)
    return (f64(t) for t in (x.q, x.k, x.v, x.g))


def check_masked_brute_bool(ora):
    """Bool mask (full-head) with the causal rule, against 40-digit brute force
    over exactly the keys each row keeps; rows keeping nothing are zeros."""
    Q, K, V, G = _mask_case(60)
    rng = np.random.default_rng(60)
    mask = rng.random((1, 4, 3, 6)) < 0.6
    mask[0, 1, 2] = False                           # a row that keeps no key
    out, lse = ora.sdpa_masked(Q, K, V, G, mask, causal=True, kv_offset=2,
                               head_chunking=False)
    for h in range(4):
        g = h * 2 // 4
        for i in range(3):
            keys = [j for j in range(6) if j <= 2 + i and mask[0, h, i, j]]
            o, l = brute._row(Q[0, h, i], [K[0, g, j] for j in keys],
                              [V[0, g, j] for j in keys], G[0, h, i])
            e = _cmp(out[0, h, i], [float(v) for v in o], 1e-13, f"bool mask row {h, i}")
            if e:
                return e
            if l is None:
                if lse[0, h, i] != -np.inf or np.any(out[0, h, i] != 0):
                    return "row with no kept key"
            elif abs(lse[0, h, i] - float(l)) > 1e-13:
                return "bool mask lse"
    return ""


def check_masked_brute_additive(ora):
    """Additive 2-D mask (dyadic values, one -inf) against brute force with the
    biases added exactly to the scaled scores."""
    Q, K, V, G = _mask_case(61)
    rng = np.random.default_rng(61)
    bias = np.round(rng.normal(0, 2, (3, 6)) * 8) / 8
    bias[1, 4] = -np.inf
    out, lse = ora.sdpa_masked(Q, K, V, G, bias)
    for h in range(4):
        g = h * 2 // 4
        for i in range(3):
            keys = [j for j in range(6) if bias[i, j] != -np.inf]
            o, l = brute._row(Q[0, h, i], [K[0, g, j] for j in keys],
                              [V[0, g, j] for j in keys], G[0, h, i],
                              biases=[bias[i, j] for j in keys])
            e = _cmp(out[0, h, i], [float(v) for v in o], 1e-13, f"additive row {h, i}")
            if e or abs(lse[0, h, i] - float(l)) > 1e-13:
                return e or "additive lse"
    return ""


def check_masked_library_sdpa(ora):
    """torch scaled_dot_product_attention in float64 (bool and additive attn_mask,
    GQA by repeat_interleave), ungated, full-head masks without chunking."""
    import torch.nn.functional as F
    Q, K, V, _ = _mask_case(62, B=2, Hq=6, Hkv=2, Lq=5, Lkv=9)
    rng = np.random.default_rng(62)
    bmask = rng.random((2, 6, 5, 9)) < 0.7
    bmask[..., 0] = True                            # no fully masked row (torch gives NaN)
    amask = rng.normal(0, 3, (2, 6, 5, 9))
    kt = torch.from_numpy(K).repeat_interleave(3, dim=1)
    vt = torch.from_numpy(V).repeat_interleave(3, dim=1)
    for m in (bmask, amask):
        ref = F.scaled_dot_product_attention(torch.from_numpy(Q), kt, vt,
                                             attn_mask=torch.from_numpy(m), scale=1.0 / 16)
        out, _ = ora.sdpa_masked(Q, K, V, None, m, head_chunking=False)
        e = _cmp(out, ref.numpy(), 1e-12, f"library sdpa {m.dtype}")
        if e:
            return e
    return ""


def check_masked_reductions(ora):
    """A 2-D mask equals its explicit 4-D expansion; an all-True mask with the
    causal rule is the prefill oracle; an additive -inf is a False; adding a
    constant c to a row's biases keeps its output and moves its lse by c; a row
    whose biases are all -inf sees no key (zeros, lse -inf)."""
    Q, K, V, G = _mask_case(63, Lq=4, Lkv=7)
    rng = np.random.default_rng(63)
    m2 = rng.random((4, 7)) < 0.6
    m2[:, 0] = True
    a, la = ora.sdpa_masked(Q, K, V, G, m2)
    b, lb = ora.sdpa_masked(Q, K, V, G, np.broadcast_to(m2, (1, 4, 4, 7)).copy())
    if not (np.array_equal(a, b) and np.array_equal(la, lb)):
        return "2-D mask differs from its expansion"
    c, lc = ora.sdpa_masked(Q, K, V, G, np.ones((4, 7), bool), causal=True, kv_offset=3)
    p, lp = ora.prefill(Q, K, V, G, kv_offset=3)
    e = _cmp(c, p, 1e-13, "causal all-True") or _cmp(lc, lp, 1e-13, "causal all-True lse")
    if e:
        return e
    add = np.where(m2, 0.0, -np.inf)
    d, ld = ora.sdpa_masked(Q, K, V, G, add)
    e = _cmp(d, a, 1e-13, "-inf vs False") or _cmp(ld, la, 1e-13, "-inf vs False lse")
    if e:
        return e
    add2 = add.copy()
    add2[2] = -np.inf                                 # row 2 excludes every key
    z, lz = ora.sdpa_masked(Q, K, V, G, add2)
    if not (np.all(z[:, :, 2] == 0) and np.all(lz[:, :, 2] == -np.inf)):
        return "a row whose biases are all -inf is not empty"
    shift = rng.normal(0, 5, (4, 1))
    f, lf = ora.sdpa_masked(Q, K, V, G, add + shift)
    return (_cmp(f, a, 1e-12, "row shift") or
            _cmp(lf, la + shift[:, 0][None, None, :], 1e-12, "row shift lse"))


def check_masked_chunk_local(ora):
    """4 rows x GQA 16 with chunking runs chunks [8, 8]: a chunk-local mask of 8
    heads gives query head h mask head (h mod 16) mod 8, the same as the tiled
    full-head mask run without chunking."""
    Q, K, V, G = _mask_case(64, Hq=32, Hkv=2, Lq=4, Lkv=6)
    rng = np.random.default_rng(64)
    local = rng.random((1, 8, 4, 6)) < 0.6
    local[..., 0] = True
    full = np.concatenate([local] * 4, axis=1)        # head h -> local[h % 8]
    a, la = ora.sdpa_masked(Q, K, V, G, local, head_chunking=True)
    b, lb = ora.sdpa_masked(Q, K, V, G, full, head_chunking=False)
    if not (np.array_equal(a, b) and np.array_equal(la, lb)):
        return "chunk-local mask"
    return ""


def _load_mask_rules():
    rows = []
    with open(os.path.join(GOLDEN, "mask_head_rules.txt")) as f:
        for line in f:
            line = line.split("#")[0].split()
            if line:
                r, gqa, hkv, hm = (int(v) for v in line[:4])
                rows.append((r, gqa, hkv, hm, line[4] == "on", line[5]))
    return rows


def check_mask_rules_golden(ora):
    """Accept / reject of mask head counts against the rules derived by hand from
    the page (tests/golden/mask_head_rules.txt), plus refusals of batch, row and
    key dimensions that do not broadcast and of masks with more than 4 dims."""
    rules = _load_mask_rules()
    if len(rules) < 20:
        return "golden file too short"
    for r, gqa, hkv, hm, chunking, expect in rules:
        Q = np.zeros((1, gqa * hkv, r, 256))
        K = np.zeros((1, hkv, 2, 256))
        mask = np.ones((1, hm, r, 2), bool)
        try:
            ora.sdpa_masked(Q, K, K, None, mask, head_chunking=chunking)
            got = "ok"
        except ValueError:
            got = "reject"
        if got != expect:
            return f"rows {r} GQA {gqa} Hkv {hkv} mask heads {hm} chunking {chunking}: {got}"
    Q = np.zeros((2, 4, 3, 256))
    K = np.zeros((2, 2, 5, 256))
    for shape in ((3, 1, 3, 5), (1, 1, 2, 5), (1, 1, 3, 4), (1, 1, 1, 3, 5), (2, 4, 3, 5, 1)):
        try:
            ora.sdpa_masked(Q, K, K, None, np.ones(shape, bool), head_chunking=False)
            return f"mask {shape} accepted"
        except ValueError:
            pass
    return ""


CHECKS = [
    check_brute_prefill, check_brute_prefill_ungated, check_brute_decode, check_library_sdpa,
    check_one_key, check_gate_zero_half, check_gate_large_passthrough, check_equal_keys_mean,
    check_dominant_key, check_masked_keys_ignored, check_chunked_prefill,
    check_verify_equals_prefill, check_head_chunks, check_merge_partition,
    check_merge_empty_row, check_plan_golden, check_brute_tree, check_tree_chain_is_decode,
    check_tree_storage_permutation, check_kv_append_brute, check_kv_keep_brute,
    check_append_then_chain_verify, check_nonfinite_q_row, check_nonfinite_v_column,
    check_nonfinite_k_sign, check_nonfinite_k_nan, check_nonfinite_gate, check_nonfinite_unseen,
    check_nonfinite_masked_kv, check_nonfinite_merge,
    check_masked_brute_bool, check_masked_brute_additive, check_masked_library_sdpa,
    check_masked_reductions, check_masked_chunk_local, check_mask_rules_golden,
]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    err = check(O)
    assert not err, err


def test_plan_rule_properties():
    """The plan always covers the group exactly, in order, with chunks <= 32/rows
    whenever it splits; counts that are not positive are refused."""
    for rows in range(1, 40):
        for gqa in range(1, 30):
            plan = O.head_chunk_plan(rows, gqa)
            assert sum(plan) == gqa
            if len(plan) > 1:
                assert rows * gqa > 32 and rows <= 32
                assert max(plan) == min(gqa, 32 // rows)
                assert all(c == plan[0] for c in plan[:-1])
    for bad in [(0, 4), (4, 0), (-1, 2)]:
        with pytest.raises(ValueError):
            O.head_chunk_plan(*bad)
    assert O.head_chunk_plan(4, 12, enabled=False) == [12]
