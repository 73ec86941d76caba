"""gqa_attn_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (a serving loop that must not touch an allocator between steps, a
plug-in whose host application only hands it fixed buffers).  It keeps its partial
results in a fixed 16 MiB area owned by the library instead of a caller workspace.

The test calls it through the C ABI and checks its output against the existing
gqa_attn_decode (caller workspace) within the parity tolerance the other tests use,
on two calls in a row with different inputs, so a stale partial result left in the
shared area by the first call would show in the second.  This file is named to be
collected last."""
import ctypes

import pytest
import torch

import gqa_head_gated_gb300 as G
from gqa_head_gated_gb300 import _lib
from synth import inputs as S
from tests.parity import MAX_ABS, MEDIAN_REL, errors

pytestmark = pytest.mark.gpu
DEV = "cuda"
LIMIT = 16 << 20


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, x, q, kc, vc, g, kv, cu, out, lse):
    T, Hq, _ = x.q.shape
    B, Hkv, Lcap, _ = x.k_cache.shape
    return lib.gqa_attn_decode_noalloc(
        _p(q), _p(kc), _p(vc), _p(g), _p(kv), _p(cu), _p(out), _p(lse), B, T, Hq, Hkv, Lcap,
        max(x.rows), int(x.kv_lens.max()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_decode_matches_workspace_decode_twice():
    lib = _lib.load()
    cases = [
        S.make_decode(3, 16, 2, [1, 3, 8], [3000, 500, 7000], seed=31),
        S.make_decode(4, 24, 4, [2, 1, 4, 1], [9000, 64, 1200, 20000], seed=32),
    ]
    for x in cases:
        q, kc, vc, g = (t.to(DEV) for t in (x.q, x.k_cache, x.v_cache, x.g))
        kv, cu = x.kv_lens.to(DEV), x.cu_rows.to(DEV)
        T, Hq, _ = x.q.shape
        B, Hkv = x.k_cache.shape[:2]
        assert G.decode_workspace_size(B, T, Hq, Hkv, max(x.rows), int(x.kv_lens.max())) <= LIMIT
        ref, ref_lse = G.decode(q, kc, vc, g, kv, cu, max_rows=max(x.rows),
                                max_kv_len=int(x.kv_lens.max()), return_lse=True)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device=DEV)
        assert _noalloc(lib, x, q, kc, vc, g, kv, cu, out, lse) == 0
        torch.cuda.synchronize()
        assert G.last_device_status() == 0
        e = errors(out, ref.float())
        assert e["nonfinite"] == 0 and e["max_abs"] <= MAX_ABS and e["median_rel"] <= MEDIAN_REL, e
        assert (lse - ref_lse).abs().max().item() <= 2e-3


def test_noalloc_refuses_sizes_past_its_area():
    """Partial results that would not fit the 16 MiB area are refused with
    GQA_ERR_WORKSPACE before any launch."""
    lib = _lib.load()
    x = S.make_decode(2, 16, 2, [32, 32], [40000, 40000], Lcap=40000, seed=33, pad_value=None)
    T, Hq, _ = x.q.shape
    B, Hkv = x.k_cache.shape[:2]
    assert G.decode_workspace_size(B, T, Hq, Hkv, 32, 40000) > LIMIT
    q = x.q.to(DEV)
    kc = x.k_cache.to(DEV)
    kv, cu = x.kv_lens.to(DEV), x.cu_rows.to(DEV)
    out = torch.empty_like(q)
    assert _noalloc(lib, x, q, kc, kc, None, kv, cu, out, None) == 5
