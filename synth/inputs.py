"""Seeded synthetic inputs for gated GQA attention at head_dim 256.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path (tests, bench, smoke) and the float64
oracle read the tensors it returns, so both sides see the same bf16 values.

Draw order (fixed so that a seed names one input exactly):
  1. structural values (kv lengths, rows per sequence, outlier key positions),
  2. Q, 3. K, 4. V, 5. G,
each drawn as float32 ``randn`` on a CPU ``torch.Generator`` and rounded to
bf16 (round to nearest even), or to fp16 when ``dtype=torch.float16`` (the same
draws, so a seed names the same real values up to the rounding).  G is
``randn * 2`` (std 2).

The five named workloads are the head geometries the pages quote for the
Qwen3.6 family: 24 query heads over 4 KV heads (the 27B) and 16 over 2 (the
35B-A3B), head_dim 256 (TensorFold PR #1009, "Receipt", attention contract
paragraph; d-inference PR #640, "Summary").
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

HEAD_DIM = 256


def _bf16(x: torch.Tensor, dtype=torch.bfloat16) -> torch.Tensor:
    assert dtype in (torch.bfloat16, torch.float16)
    return x.to(dtype)


@dataclass
class PrefillInputs:
    """Prompt rows: Q,G,out [B,Hq,Lq,256]; K,V [B,Hkv,Lkv,256]."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    kv_offset: int
    seed: int
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        B, Hq, Lq, _ = self.q.shape
        return dict(B=B, Hq=Hq, Hkv=self.k.shape[1], Lq=Lq, Lkv=self.k.shape[2],
                    kv_offset=self.kv_offset)


@dataclass
class DecodeInputs:
    """Decode / chain-verify rows against a contiguous cache.

    q, g: [T,Hq,256] packed token-major (T = sum of rows per sequence).
    k_cache, v_cache: [B,Hkv,Lcap,256]; keys >= kv_lens[b] are padding.
    kv_lens: int32 [B], counting the verify rows themselves.
    cu_rows: int32 [B+1] exclusive prefix sum of rows per sequence.
    """
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    g: torch.Tensor
    kv_lens: torch.Tensor
    cu_rows: torch.Tensor
    seed: int
    meta: dict = field(default_factory=dict)

    @property
    def rows(self):
        return (self.cu_rows[1:] - self.cu_rows[:-1]).tolist()

    @property
    def shape(self):
        T, Hq, _ = self.q.shape
        B, Hkv, Lcap, _ = self.k_cache.shape
        return dict(B=B, T=T, Hq=Hq, Hkv=Hkv, Lcap=Lcap, max_rows=max(self.rows),
                    max_kv_len=int(self.kv_lens.max()))


def make_prefill(B, Hq, Hkv, Lq, Lkv=None, kv_offset=0, seed=0, outlier_frac=0.0,
                 outlier_scale=8.0, g_std=2.0, dtype=torch.bfloat16) -> PrefillInputs:
    """Prompt-row inputs.  ``outlier_frac`` of the key rows of every (b, KV head)
    are multiplied by ``outlier_scale`` (x8 is exact in bf16); positions are drawn
    without replacement before any tensor, one permutation per (b, KV head)."""
    if Lkv is None:
        Lkv = kv_offset + Lq
    gen = torch.Generator().manual_seed(seed)
    n_out = int(round(outlier_frac * Lkv))
    outliers = []
    if n_out:
        for _ in range(B * Hkv):
            outliers.append(torch.randperm(Lkv, generator=gen)[:n_out])
    q = _bf16(torch.randn(B, Hq, Lq, HEAD_DIM, generator=gen), dtype)
    k = _bf16(torch.randn(B, Hkv, Lkv, HEAD_DIM, generator=gen), dtype)
    v = _bf16(torch.randn(B, Hkv, Lkv, HEAD_DIM, generator=gen), dtype)
    g = _bf16(torch.randn(B, Hq, Lq, HEAD_DIM, generator=gen) * g_std, dtype)
    if n_out:
        kf = k.view(B * Hkv, Lkv, HEAD_DIM)
        for i, pos in enumerate(outliers):
            kf[i, pos] = _bf16(kf[i, pos].float() * outlier_scale, dtype)
    return PrefillInputs(q, k, v, g, kv_offset, seed,
                         meta=dict(outliers=[p.tolist() for p in outliers]))


def make_decode(B, Hq, Hkv, rows, kv_lens, Lcap=None, seed=0, pad_value=float("nan"),
                g_std=2.0, gen=None, dtype=torch.bfloat16) -> DecodeInputs:
    """Decode/verify inputs with explicit rows per sequence and kv lengths.

    Keys [0, kv_lens[b]) of every (b, KV head) are drawn; the padding beyond is
    filled with ``pad_value`` (NaN by default, so that any read of it shows), or
    left as zeros when ``pad_value`` is None.
    """
    rows = [int(r) for r in rows]
    kv_lens = [int(x) for x in kv_lens]
    assert len(rows) == B and len(kv_lens) == B
    if Lcap is None:
        Lcap = max(kv_lens) if kv_lens else 1
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    T = sum(rows)
    cu = [0]
    for r in rows:
        cu.append(cu[-1] + r)
    q = _bf16(torch.randn(T, Hq, HEAD_DIM, generator=gen), dtype)
    fill = 0.0 if pad_value is None else pad_value
    kc = torch.full((B, Hkv, Lcap, HEAD_DIM), fill, dtype=dtype)
    vc = torch.full((B, Hkv, Lcap, HEAD_DIM), fill, dtype=dtype)
    for b in range(B):
        kc[b, :, :kv_lens[b]] = _bf16(torch.randn(Hkv, kv_lens[b], HEAD_DIM, generator=gen), dtype)
    for b in range(B):
        vc[b, :, :kv_lens[b]] = _bf16(torch.randn(Hkv, kv_lens[b], HEAD_DIM, generator=gen), dtype)
    g = _bf16(torch.randn(T, Hq, HEAD_DIM, generator=gen) * g_std, dtype)
    return DecodeInputs(q, kc, vc, g, torch.tensor(kv_lens, dtype=torch.int32),
                        torch.tensor(cu, dtype=torch.int32), seed)


def random_tree_masks(rows, seed):
    """Seeded token trees for draft verify: new row i of each sequence takes a
    uniformly drawn earlier row as parent, or none; its mask holds its own bit and
    its ancestors' bits (bit k = new row k).  Returns a list of ints, one per row."""
    gen = torch.Generator().manual_seed(seed)
    out = []
    for r in rows:
        anc = []
        for i in range(int(r)):
            par = int(torch.randint(-1, i, (1,), generator=gen)) if i else -1
            anc.append((1 << i) | (anc[par] if par >= 0 else 0))
        out.extend(anc)
    return out


# ---------------------------------------------------------------------------
# The five named workloads.
# ---------------------------------------------------------------------------

def tiny_prefill(dtype=torch.bfloat16):
    """B=1, 24/4 heads, Lq=Lkv=128 causal, seed 0."""
    return make_prefill(1, 24, 4, 128, seed=0, dtype=dtype)


def decode_27b(pad_value=float("nan"), dtype=torch.bfloat16):
    """B=16 sequences, 24/4 heads, one row each, kv lengths uniform in
    [1024, 32768] in a [16,4,32768,256] cache, seed 1."""
    gen = torch.Generator().manual_seed(1)
    kv = torch.randint(1024, 32769, (16,), generator=gen).tolist()
    return make_decode(16, 24, 4, [1] * 16, kv, Lcap=32768, seed=1, gen=gen,
                       pad_value=pad_value, dtype=dtype)


def prefill_27b(dtype=torch.bfloat16):
    """B=1, 24/4 heads, Lq=Lkv=8192 causal, 1% of key rows x8, seed 2."""
    return make_prefill(1, 24, 4, 8192, seed=2, outlier_frac=0.01, dtype=dtype)


def chunked_prefill_35b(dtype=torch.bfloat16):
    """B=1, 16/2 heads, a 2048-row chunk at kv_offset 30720 (Lkv 32768), seed 3."""
    return make_prefill(1, 16, 2, 2048, Lkv=32768, kv_offset=30720, seed=3, dtype=dtype)


VERIFY_ROWS = (1, 3, 4, 8, 16, 32)


def verify_35b(pad_value=float("nan"), dtype=torch.bfloat16):
    """B=8, 16/2 heads, rows per sequence from {1,3,4,8,16,32} (taken in turn,
    sequence b gets VERIFY_ROWS[b % 6]), kv lengths uniform in [4097, 65536]
    in a [8,2,65536,256] cache, seed 4."""
    gen = torch.Generator().manual_seed(4)
    kv = torch.randint(4097, 65537, (8,), generator=gen).tolist()
    rows = [VERIFY_ROWS[b % len(VERIFY_ROWS)] for b in range(8)]
    return make_decode(8, 16, 2, rows, kv, Lcap=65536, seed=4, gen=gen,
                       pad_value=pad_value, dtype=dtype)


WORKLOADS = {
    "tiny_prefill": tiny_prefill,
    "decode_27b": decode_27b,
    "prefill_27b": prefill_27b,
    "chunked_prefill_35b": chunked_prefill_35b,
    "verify_35b": verify_35b,
}
