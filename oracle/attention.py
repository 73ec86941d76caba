"""Float64 CPU oracle for causal grouped-query attention with sigmoid output gating.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
baseline may import this module.  It shares no code with the CUDA library: it
receives float64 numpy arrays (exact copies of the bf16 inputs) and computes
the plain definition, row by row, without blocking over keys, fusion or an
online softmax.

What it computes (for every batch b, query head h, query row i):

    g      = h // (Hq // Hkv)                      KV head of query head h
    V_i    = { j : j < lim_i }                     keys row i may see
    s_j    = (Q[b,h,i,:] . K[b,g,j,:]) / 16        j in V_i      (1/16 = 1/sqrt(256))
    m      = max_j s_j,  p_j = exp(s_j - m),  l = sum_j p_j
    o      = sum_j p_j V[b,g,j,:] / l
    out    = o * 1 / (1 + exp(-G[b,h,i,:]))        sigmoid output gate
    lse    = m + ln l

Sources (page, section):
  * TensorFold PR #1009, "Receipt", attention contract paragraph: the kernels are
    checked against float64 gated attention at the 24/4 and 16/2 head shapes;
    masked future keys must not contaminate a row (the -Inf x 0 prediction in the
    same PR's second comment).
  * TensorFold PR #1009, "Design: one engine": gated full attention layers.
  * DS4Server issue113 README, opening rule: query heads inside each KV group,
    head chunks of min(GQA, 32/rows) with remainders, concatenated in head order.
  * The formula, scale 1/16 and the causal/offset mask as the task states them.

Readings where the pages are silent (each listed in the design notes):
  * the gate is elementwise, G has the shape of the output;
  * query head h uses KV head h // GQA (consecutive grouping);
  * prefill row i sits at absolute position kv_offset + i and sees keys
    j <= kv_offset + i;
  * decode/verify: kv_lens[b] counts the verify rows, row i of r_b rows sees
    keys j < kv_lens[b] - r_b + i + 1;
  * tree verify: row i sees the keys before the new rows plus the new keys its
    mask selects (bit k = new row k); a chain is the mask of bits 0..i;
  * a row that sees no key outputs zeros and lse = -inf (float64 would give 0/0);
  * keys a row does not see are excluded from its sums, never weighted by 0: each
    row is evaluated on its own over exactly the keys it sees, so a NaN or Inf in
    the K or V row of a key the row does not see cannot reach it (0 x Inf is NaN,
    the hazard the TensorFold PR's second comment predicts for masked keys), and a
    row's result does not depend on which other rows share the call.
"""
from __future__ import annotations

import math

import numpy as np

HEAD_DIM = 256
SCALE = 1.0 / 16.0          # 1/sqrt(head_dim)
ROW_BLOCK = 256             # rows handed to attend_rows at a time (each evaluated alone)


def sigmoid(x):
    """Elementwise logistic function in float64."""
    return 1.0 / (1.0 + np.exp(-x))


def kv_head_of(h: int, Hq: int, Hkv: int) -> int:
    """KV head serving query head h: consecutive groups of GQA = Hq/Hkv heads."""
    return h // (Hq // Hkv)


def prefill_visible(i: int, kv_offset: int) -> int:
    """Number of keys prompt row i may see: keys 0..kv_offset+i."""
    return kv_offset + i + 1


def verify_visible(i: int, rows: int, kv_len: int) -> int:
    """Number of keys verify row i (0-based of `rows`) may see: the cache holds
    kv_len keys including the rows themselves, so the row sits at absolute
    position kv_len - rows + i."""
    return kv_len - rows + i + 1


def attend_rows(q_rows, K, V, g_rows, lims):
    """Gated attention of query rows against one KV head.

    q_rows [n,D], g_rows [n,D] or None, K,V [L,D], lims [n]: row i sees keys
    0 .. lims[i]-1 and no other.  Every row is evaluated alone over the slice of
    keys it sees (scores, max shift, sum and the weighted sum of V rows), so keys
    past its limit take no part in any product for it.  Calling this with one row
    or with that row inside a block gives the same bits.
    Returns (out [n,D], lse [n]) in float64.
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    lims = [int(x) for x in lims]
    n, D = q_rows.shape
    out = np.zeros((n, D))
    lse = np.full(n, -np.inf)
    kmax = max(lims, default=0)
    if kmax <= 0:
        return out, lse
    Kb = np.asarray(K[:kmax], dtype=np.float64)
    Vb = np.asarray(V[:kmax], dtype=np.float64)
    for i in range(n):
        lim = lims[i]
        if lim <= 0:
            continue                                  # sees no key: zeros, lse -inf
        s = (Kb[:lim] @ q_rows[i]) * SCALE            # scores of the visible keys
        m = np.max(s)
        p = np.exp(s - m)
        l = np.sum(p)
        o = (p @ Vb[:lim]) / l
        if g_rows is not None:
            o = o * sigmoid(np.asarray(g_rows[i], dtype=np.float64))
        out[i] = o
        lse[i] = m + math.log(l)                      # l >= 1, or NaN
    return out, lse


def prefill(Q, K, V, G, kv_offset=0, rows=None):
    """Prompt-row attention.  Q,G [B,Hq,Lq,D]; K,V [B,Hkv,Lkv,D] (float64-able).

    ``rows``: optional iterable of (b, h, i) to evaluate only those rows (for
    sampled checks at full size).  Returns (out, lse): full arrays
    [B,Hq,Lq,D]/[B,Hq,Lq] when rows is None, else arrays [n,D]/[n] in the order
    given.
    """
    B, Hq, Lq, D = Q.shape
    Hkv, Lkv = K.shape[1], K.shape[2]
    assert D == HEAD_DIM and Hq % Hkv == 0 and kv_offset + Lq <= Lkv
    if rows is not None:
        rows = list(rows)
        out = np.zeros((len(rows), D))
        lse = np.zeros(len(rows))
        for n, (b, h, i) in enumerate(rows):
            g = kv_head_of(h, Hq, Hkv)
            o, s = attend_rows(np.asarray(Q[b, h, i:i + 1], dtype=np.float64), K[b, g], V[b, g],
                               None if G is None else G[b, h, i:i + 1],
                               [prefill_visible(i, kv_offset)])
            out[n], lse[n] = o[0], s[0]
        return out, lse
    out = np.zeros((B, Hq, Lq, D))
    lse = np.zeros((B, Hq, Lq))
    for b in range(B):
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            for r0 in range(0, Lq, ROW_BLOCK):
                r1 = min(Lq, r0 + ROW_BLOCK)
                lims = [prefill_visible(i, kv_offset) for i in range(r0, r1)]
                o, s = attend_rows(Q[b, h, r0:r1], K[b, g], V[b, g],
                                   None if G is None else G[b, h, r0:r1], lims)
                out[b, h, r0:r1] = o
                lse[b, h, r0:r1] = s
    return out, lse


def decode(Q, Kc, Vc, G, kv_lens, cu_rows=None, rows=None):
    """Decode (one row per sequence) and chain verify (rows causal within the
    sequence's new rows) against a contiguous cache.

    Q,G [T,Hq,D] token-major; Kc,Vc [B,Hkv,Lcap,D]; kv_lens [B] (includes the
    rows); cu_rows [B+1] or None (one row per sequence).  ``rows``: optional
    iterable of (t, h) to evaluate only those outputs.  Returns (out, lse) of
    shapes [T,Hq,D]/[T,Hq] or [n,D]/[n].
    """
    T, Hq, D = Q.shape
    B, Hkv = Kc.shape[0], Kc.shape[1]
    kv_lens = [int(x) for x in kv_lens]
    cu = list(range(B + 1)) if cu_rows is None else [int(x) for x in cu_rows]
    assert D == HEAD_DIM and Hq % Hkv == 0 and cu[-1] == T
    seq_of = np.zeros(T, dtype=np.int64)
    for b in range(B):
        seq_of[cu[b]:cu[b + 1]] = b

    def lim_of(t):
        b = int(seq_of[t])
        return verify_visible(t - cu[b], cu[b + 1] - cu[b], kv_lens[b])

    if rows is not None:
        rows = list(rows)
        out = np.zeros((len(rows), D))
        lse = np.zeros(len(rows))
        for n, (t, h) in enumerate(rows):
            b = int(seq_of[t])
            g = kv_head_of(h, Hq, Hkv)
            o, s = attend_rows(np.asarray(Q[t, h:h + 1], dtype=np.float64), Kc[b, g], Vc[b, g],
                               None if G is None else G[t, h:h + 1], [lim_of(t)])
            out[n], lse[n] = o[0], s[0]
        return out, lse
    out = np.zeros((T, Hq, D))
    lse = np.zeros((T, Hq))
    for b in range(B):
        ts = list(range(cu[b], cu[b + 1]))
        if not ts:
            continue
        lims = [lim_of(t) for t in ts]
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            o, s = attend_rows(Q[ts[0]:ts[-1] + 1, h], Kc[b, g], Vc[b, g],
                               None if G is None else G[ts[0]:ts[-1] + 1, h], lims)
            out[ts[0]:ts[-1] + 1, h] = o
            lse[ts[0]:ts[-1] + 1, h] = s
    return out, lse


def tree_visible_keys(i, rows, kv_len, mask):
    """Keys new row i (0-based of `rows`) sees under a tree mask: every key before
    the new rows (positions < kv_len - rows) and the new key at position
    kv_len - rows + k for each set bit k of `mask` (an integer; bit k = new row k)."""
    base = kv_len - rows
    return list(range(base)) + [base + k for k in range(rows) if (int(mask) >> k) & 1]


def decode_tree(Q, Kc, Vc, G, kv_lens, cu_rows, tree_masks, rows=None):
    """Draft verify over a token tree.  Like decode(), but new row i of a sequence
    sees the new keys that its mask selects (its ancestors and itself) instead of
    all earlier new keys.  tree_masks [T]: integer masks over the sequence's new
    rows.  A chain (mask of row i = bits 0..i) gives decode()'s result.  Keys a row
    does not see are excluded from its sums (gathered out, never multiplied)."""
    T, Hq, D = Q.shape
    B, Hkv = Kc.shape[0], Kc.shape[1]
    cu = [int(x) for x in cu_rows]
    assert D == HEAD_DIM and Hq % Hkv == 0 and cu[-1] == T
    want = None if rows is None else list(rows)
    out = np.zeros((T, Hq, D)) if want is None else np.zeros((len(want), D))
    lse = np.zeros((T, Hq)) if want is None else np.zeros(len(want))
    index = {}
    if want is not None:
        for n, th in enumerate(want):
            index.setdefault(th[0], []).append((n, th[1]))
    for b in range(B):
        r = cu[b + 1] - cu[b]
        L = int(kv_lens[b])
        for i in range(r):
            t = cu[b] + i
            if want is not None and t not in index:
                continue
            keys = np.asarray(tree_visible_keys(i, r, L, tree_masks[t]), dtype=np.int64)
            heads = range(Hq) if want is None else [h for _, h in index[t]]
            for h in heads:
                g = kv_head_of(h, Hq, Hkv)
                Kg = np.asarray(Kc[b, g], dtype=np.float64)[keys]
                Vg = np.asarray(Vc[b, g], dtype=np.float64)[keys]
                o, l = attend_rows(np.asarray(Q[t, h:h + 1], dtype=np.float64), Kg, Vg,
                                   None if G is None else G[t, h:h + 1], [len(keys)])
                if want is None:
                    out[t, h], lse[t, h] = o[0], l[0]
                else:
                    for n, hh in index[t]:
                        if hh == h:
                            out[n], lse[n] = o[0], l[0]
    return out, lse


def kv_append(Kc, Vc, Knew, Vnew, kv_lens, cu_rows):
    """Writes the new rows of each sequence into its cache after the keys it holds:
    cache[b, g, kv_lens[b] + i] = new[cu_rows[b] + i, g] for i < rows of b.
    Knew, Vnew: [T, Hkv, D] token-major; caches [B, Hkv, Lcap, D].  Returns new
    arrays (the inputs are not modified).  This is the append the TensorFold
    attention contract compares bit for bit (its control: an append one row late)."""
    Kc, Vc = np.array(Kc, copy=True), np.array(Vc, copy=True)
    cu = [int(x) for x in cu_rows]
    for b in range(len(cu) - 1):
        L = int(kv_lens[b])
        r = cu[b + 1] - cu[b]
        Kc[b, :, L:L + r] = np.swapaxes(np.asarray(Knew)[cu[b]:cu[b + 1]], 0, 1)
        Vc[b, :, L:L + r] = np.swapaxes(np.asarray(Vnew)[cu[b]:cu[b + 1]], 0, 1)
    return Kc, Vc


def kv_keep(Kc, Vc, kv_lens, cu_rows, keep):
    """After verifying r_b draft rows held at positions kv_lens[b] - r_b ..
    kv_lens[b] - 1, keeps the accepted ones: draft row keep[b][k] moves to position
    kv_lens[b] - r_b + k, in order.  Returns (new caches, new kv_lens)."""
    Kc, Vc = np.array(Kc, copy=True), np.array(Vc, copy=True)
    cu = [int(x) for x in cu_rows]
    new_lens = []
    for b in range(len(cu) - 1):
        r = cu[b + 1] - cu[b]
        base = int(kv_lens[b]) - r
        src = [base + int(i) for i in keep[b]]
        Kc[b, :, base:base + len(src)] = Kc[b][:, src]
        Vc[b, :, base:base + len(src)] = Vc[b][:, src]
        new_lens.append(base + len(src))
    return Kc, Vc, new_lens


def chain_masks(rows_per_seq):
    """Masks of chain verify: new row i sees new rows 0..i."""
    return [(1 << (i + 1)) - 1 for r in rows_per_seq for i in range(r)]


def lse_merge(O_parts, lse_parts, G=None):
    """Combine S partial results of the same rows over disjoint key sets.

    O_parts [S,N,D]: each part normalised (sum_j p_j V_j / l_s over its keys);
    lse_parts [S,N]: m_s + ln l_s of the part, -inf for a part with no key.
    out_n = sum_s exp(lse_s) O_s / sum_s exp(lse_s), times sigmoid(G) when given;
    lse_n = ln sum_s exp(lse_s).  Parts of weight 0 (lse -inf) are not read.  A
    row whose parts are all empty outputs zeros and lse -inf.  A NaN or +Inf lse
    enters the sums as float64 arithmetic takes it (weight NaN: the row is NaN), so
    a part that saw a NaN score poisons its row as it would in the unsplit row.

    This is the tail-chunk merge the TensorFold attention contract checks (its
    control "a merge dropping later tail chunks" must fail).
    """
    O_parts = np.asarray(O_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    S, N, D = O_parts.shape
    out = np.zeros((N, D))
    lse = np.full(N, -np.inf)
    for n in range(N):
        live = [s for s in range(S) if lse_parts[s, n] != -np.inf]
        if not live:
            continue
        M = float(np.max(lse_parts[live, n]))          # NaN if any part is NaN
        w = np.array([math.exp(lse_parts[s, n] - M) for s in live])
        acc = np.zeros(D)
        for ws, s in zip(w, live):
            acc += ws * O_parts[s, n]
        out[n] = acc / w.sum()
        lse[n] = M + math.log(w.sum())
    if G is not None:
        out = out * sigmoid(np.asarray(G, dtype=np.float64).reshape(N, D))
    return out, lse


def head_chunk_plan(rows: int, gqa: int, enabled: bool = True, limit: int = 32):
    """Head-chunk sizes for one KV group (DS4Server issue113 README, opening
    rule): when enabled, rows <= 32 and rows*GQA > 32, the group's query heads are
    split into chunks of min(GQA, 32 // rows) heads with the remainder kept as a
    last, smaller chunk; otherwise the group is one chunk.  Invalid counts are
    refused."""
    if rows < 1 or gqa < 1:
        raise ValueError("rows and heads per group must be positive")
    if not enabled or rows > limit or rows * gqa <= limit:
        return [gqa]
    c = min(gqa, limit // rows)
    plan = [c] * (gqa // c)
    if gqa % c:
        plan.append(gqa % c)
    return plan


def _broadcast_mask(mask, shape):
    """The caller's mask as one SDPA call broadcasts it against that call's scores
    [B, heads, rows, keys] (trailing dimensions aligned, size-1 dimensions
    repeated).  A mask that cannot broadcast is refused with ValueError."""
    m = np.asarray(mask)
    if m.ndim > 4:
        raise ValueError(f"mask has {m.ndim} dimensions; at most 4")
    try:
        return np.broadcast_to(m, shape)
    except ValueError:
        raise ValueError(f"mask of shape {m.shape} cannot broadcast to {shape}") from None


def masked_rows(q_rows, K, V, g_rows, keep, bias=None):
    """Gated attention of query rows against one KV head under an explicit mask.

    q_rows [n,D]; K, V [L,D]; g_rows [n,D] or None; keep [n,L] bool (the keys each
    row attends to); bias [n,L] float64 or None, added to the scaled scores
    (natural-log units).  Keys a row does not keep are excluded from its sums.  A
    row that keeps no key outputs zeros and lse -inf.  Returns (out [n,D], lse [n]).
    """
    q_rows = np.asarray(q_rows, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    n, D = q_rows.shape
    out = np.zeros((n, D))
    lse = np.full(n, -np.inf)
    for i in range(n):
        idx = np.nonzero(keep[i])[0]
        if idx.size == 0:
            continue
        s = (K[idx] @ q_rows[i]) * SCALE
        if bias is not None:
            s = s + bias[i, idx]
        m = s.max()
        p = np.exp(s - m)
        l = p.sum()
        o = (p @ V[idx]) / l
        if g_rows is not None:
            o = o * sigmoid(np.asarray(g_rows[i], dtype=np.float64))
        out[i] = o
        lse[i] = m + np.log(l)
    return out, lse


def sdpa_masked(Q, K, V, G, mask=None, causal=False, kv_offset=None, head_chunking=True):
    """Gated attention with a general mask, as the DS4Server issue113 README's
    dense SDPA consumer takes it ("Exact scope found during review"; its fixtures:
    no, bool, additive, two-dimensional, full-head and chunk-local masks).

    Q, G [B,Hq,Lq,D]; K, V [B,Hkv,Lkv,D].  ``mask``: None, a bool array (True =
    attend) or a float array (added to the scaled scores; -inf excludes the key
    like False), of any shape that broadcasts as below.  ``causal``: also exclude
    keys j > kv_offset + i (kv_offset defaults to Lkv - Lq).

    The head-chunk rule decides how the mask meets the heads: with chunking on,
    Lq <= 32 and Lq*GQA > 32, every KV group's heads run in chunks of
    min(GQA, 32 // Lq) (remainder last), each chunk one call that receives the
    mask unchanged, so the mask must broadcast to [B, chunk, Lq, Lkv] for every
    chunk, and head k of a chunk reads mask head k (chunk-local).  Otherwise one
    call takes all Hq heads and the mask must broadcast to [B, Hq, Lq, Lkv].  A
    mask that cannot broadcast is refused (ValueError) before anything runs.
    Returns (out [B,Hq,Lq,D], lse [B,Hq,Lq]).
    """
    B, Hq, Lq, D = Q.shape
    Hkv, Lkv = K.shape[1], K.shape[2]
    assert D == HEAD_DIM and Hq % Hkv == 0
    gqa = Hq // Hkv
    if kv_offset is None:
        kv_offset = Lkv - Lq
    out = np.zeros((B, Hq, Lq, D))
    lse = np.full((B, Hq, Lq), -np.inf)
    if Lq == 0:
        return out, lse
    plan = head_chunk_plan(Lq, gqa, head_chunking)
    # per query head: the [B, Lq, Lkv] slice of the mask its call sees
    head_mask = [None] * Hq
    if mask is not None:
        if len(plan) == 1:
            M = _broadcast_mask(mask, (B, Hq, Lq, Lkv))
            for h in range(Hq):
                head_mask[h] = M[:, h]
        else:
            for g in range(Hkv):
                h0 = g * gqa
                for c in plan:
                    M = _broadcast_mask(mask, (B, c, Lq, Lkv))
                    for k in range(c):
                        head_mask[h0 + k] = M[:, k]
                    h0 += c
    is_bool = mask is not None and np.asarray(mask).dtype == np.bool_
    base = np.ones((Lq, Lkv), dtype=bool)
    if causal:
        base = np.arange(Lkv)[None, :] <= kv_offset + np.arange(Lq)[:, None]
    for b in range(B):
        for h in range(Hq):
            g = kv_head_of(h, Hq, Hkv)
            keep, bias = base, None
            if head_mask[h] is not None:
                m = head_mask[h][b]
                if is_bool:
                    keep = base & m
                else:
                    a = np.asarray(m, dtype=np.float64)
                    keep = base & (a != -np.inf)
                    bias = np.where(keep, a, 0.0)
            o, l = masked_rows(Q[b, h], K[b, g], V[b, g], None if G is None else G[b, h],
                               keep, bias)
            out[b, h], lse[b, h] = o, l
    return out, lse


def decode_head_chunked(Q, Kc, Vc, G, kv_lens, cu_rows=None, enabled=True):
    """Decode/verify evaluated group by group and head chunk by head chunk, then
    concatenated in head order (DS4Server issue113 README, opening rule).  The
    method reaches the unchunked result; this exists so that the invariant can be
    checked."""
    T, Hq, D = Q.shape
    B, Hkv = Kc.shape[0], Kc.shape[1]
    gqa = Hq // Hkv
    cu = list(range(B + 1)) if cu_rows is None else [int(x) for x in cu_rows]
    out = np.zeros((T, Hq, D))
    lse = np.zeros((T, Hq))
    for b in range(B):
        r = cu[b + 1] - cu[b]
        if r == 0:
            continue
        sub_cu = [0, r]
        for g in range(Hkv):
            h0 = g * gqa
            for c in head_chunk_plan(r, gqa, enabled):
                hs = slice(h0, h0 + c)
                o, s = decode(Q[cu[b]:cu[b + 1], hs], Kc[b:b + 1, g:g + 1], Vc[b:b + 1, g:g + 1],
                              None if G is None else G[cu[b]:cu[b + 1], hs],
                              [kv_lens[b]], sub_cu)
                out[cu[b]:cu[b + 1], hs] = o
                lse[cu[b]:cu[b + 1], hs] = s
                h0 += c
    return out, lse
