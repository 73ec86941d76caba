"""Brute-force gated attention in 40-digit arithmetic, written independently of the
oracle, for tiny inputs only.

Differences from the oracle on purpose: dot products are exact rationals
(bf16 values are dyadic), the softmax is taken without a max shift (40 digits
do not overflow at these scores), the visible set is enumerated by comparing
absolute positions key by key, and the KV head is found by scaling the head
index (h * Hkv // Hq) instead of dividing by the group size.
"""
from __future__ import annotations

from fractions import Fraction

import mpmath

mpmath.mp.dps = 40


def _exact(x):
    return Fraction(float(x))


def _row(q, keys, vals, gate, biases=None):
    """q: list[D] floats; keys/vals: list of rows that the query sees; gate: list[D]
    or None; biases: None or one float per key, added exactly to its scaled score.
    Returns (out list[D] of mpf, lse mpf or None)."""
    D = len(q)
    if not keys:
        return [mpmath.mpf(0)] * D, None
    qf = [_exact(x) for x in q]
    w = []
    for n, k in enumerate(keys):
        dot = sum((qf[d] * _exact(k[d]) for d in range(D)), Fraction(0)) / 16
        if biases is not None:
            dot += _exact(biases[n])
        w.append(mpmath.exp(mpmath.mpf(dot.numerator) / dot.denominator))
    Z = mpmath.fsum(w)
    out = []
    for d in range(D):
        acc = mpmath.fsum(w[j] * mpmath.mpf(float(vals[j][d])) for j in range(len(keys)))
        o = acc / Z
        if gate is not None:
            o = o / (1 + mpmath.exp(-mpmath.mpf(float(gate[d]))))
        out.append(o)
    return out, mpmath.log(Z)


def prefill(Q, K, V, G, kv_offset):
    """Q,G [B,Hq,Lq,D]; K,V [B,Hkv,Lkv,D] as nested sequences (numpy ok)."""
    B, Hq, Lq = len(Q), len(Q[0]), len(Q[0][0])
    Hkv, Lkv = len(K[0]), len(K[0][0])
    out = {}
    for b in range(B):
        for h in range(Hq):
            kvh = (h * Hkv) // Hq
            for i in range(Lq):
                pos = kv_offset + i                      # absolute position of the query
                seen = [j for j in range(Lkv) if j <= pos]
                o, lse = _row(Q[b][h][i], [K[b][kvh][j] for j in seen],
                              [V[b][kvh][j] for j in seen],
                              None if G is None else G[b][h][i])
                out[(b, h, i)] = (o, lse)
    return out


def decode(Q, Kc, Vc, G, kv_lens, rows):
    """Q,G [T,Hq,D]; Kc,Vc [B,Hkv,Lcap,D]; rows: list of rows per sequence."""
    Hq = len(Q[0])
    Hkv = len(Kc[0])
    out = {}
    t = 0
    for b, r in enumerate(rows):
        L = int(kv_lens[b])
        first_new = L - r                                # position of the first new row
        for i in range(r):
            pos = first_new + i
            for h in range(Hq):
                kvh = (h * Hkv) // Hq
                seen = [j for j in range(L) if j <= pos]
                o, lse = _row(Q[t][h], [Kc[b][kvh][j] for j in seen],
                              [Vc[b][kvh][j] for j in seen],
                              None if G is None else G[t][h])
                out[(t, h)] = (o, lse)
            t += 1
    return out


def decode_tree(Q, Kc, Vc, G, kv_lens, rows, masks):
    """Tree verify, brute force: row i of a sequence with r new rows at positions
    L-r .. L-1 sees position p when p is before the new rows, or when p is new and
    the mask bit of its new-row index is set."""
    Hq = len(Q[0])
    Hkv = len(Kc[0])
    out = {}
    t = 0
    for b, r in enumerate(rows):
        L = int(kv_lens[b])
        for i in range(r):
            m = int(masks[t])
            seen = []
            for p in range(L):
                new_index = p - (L - r)
                if new_index < 0 or (m >> new_index) % 2 == 1:
                    seen.append(p)
            for h in range(Hq):
                kvh = (h * Hkv) // Hq
                o, lse = _row(Q[t][h], [Kc[b][kvh][p] for p in seen],
                              [Vc[b][kvh][p] for p in seen], None if G is None else G[t][h])
                out[(t, h)] = (o, lse)
            t += 1
    return out
