"""gqa_attn_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (a serving loop that must not touch an allocator between steps, a
plug-in whose host application only hands it fixed buffers).  It is gqa_attn_decode
with a fixed 16 MiB area owned by the library as its workspace.

The test calls it through the C ABI on each of the one-call decode's paths (tcgen05
split kernel; mma.sync kernel with balanced shares, near the size where the area is
just enough; mma.sync kernel with fixed splits for a batch past the balanced table)
and checks every output against the float64 oracle at the parity bar, and bit for
bit (out and lse) against gqa_attn_decode with a caller workspace.  Each shape is
called twice in a row with different inputs, so a stale partial result left in the
shared area by the first call would show in the second.  This file is named to be
collected last."""
import ctypes

import pytest
import torch

import gqa_head_gated_gb300 as G
import oracle
from gqa_head_gated_gb300 import _lib
from synth import inputs as S
from tests.parity import assert_parity, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
LIMIT = 16 << 20
GQA_ERR_WORKSPACE = 5


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, x, q, kc, vc, g, kv, cu, out, lse):
    T, Hq, _ = x.q.shape
    B, Hkv, Lcap, _ = x.k_cache.shape
    return lib.gqa_attn_decode_noalloc(
        _p(q), _p(kc), _p(vc), _p(g), _p(kv), _p(cu), _p(out), _p(lse), B, T, Hq, Hkv, Lcap,
        max(x.rows), int(x.kv_lens.max()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _lens(n, lo, hi, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi, (n,), generator=gen).tolist()


# (B, Hq, Hkv, rows per sequence, kv lengths): one shape per path of the one-call decode
SHAPES = {
    # 8 new rows x GQA 8 = 64 packed rows: the tcgen05 split kernel
    "tc_split": (3, 16, 2, [1, 3, 8], [3000, 500, 7000]),
    # one row x GQA 16 over 15 sequences: balanced shares whose 16 part slots take
    # 15.8 MB of the area
    "balanced_near_limit": (15, 64, 4, [1] * 15, _lens(15, 200, 1500, 9)),
    # 300 sequences (past the balanced table's 256): fixed splits on the mma.sync kernel
    "fixed_split": (300, 16, 2, [1] * 300, _lens(300, 40, 400, 7)),
}


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_noalloc_decode_matches_oracle_and_decode(shape):
    lib = _lib.load()
    B, Hq, Hkv, rows, lens = SHAPES[shape]
    for seed in (31, 32):   # the same shape twice, different inputs
        x = S.make_decode(B, Hq, Hkv, rows, lens, seed=seed)
        q, kc, vc, g = (t.to(DEV) for t in (x.q, x.k_cache, x.v_cache, x.g))
        kv, cu = x.kv_lens.to(DEV), x.cu_rows.to(DEV)
        T = x.q.shape[0]
        need = G.decode_workspace_size(B, T, Hq, Hkv, max(rows), int(x.kv_lens.max()))
        assert need <= LIMIT
        out = torch.full_like(q, float("nan"))
        lse = torch.full((T, Hq), float("nan"), dtype=torch.float32, device=DEV)
        assert _noalloc(lib, x, q, kc, vc, g, kv, cu, out, lse) == 0
        torch.cuda.synchronize()
        assert G.last_device_status() == 0
        r_out, r_lse = oracle.decode(to_f64(x.q), to_f64(x.k_cache), to_f64(x.v_cache),
                                     to_f64(x.g), x.kv_lens.tolist(), x.cu_rows.tolist())
        assert_parity(out, r_out, f"noalloc {shape} seed {seed}")
        assert_parity(lse, r_lse, f"noalloc lse {shape} seed {seed}", max_abs=2e-3,
                      median_rel=1.0)
        ref, ref_lse = G.decode(q, kc, vc, g, kv, cu, max_rows=max(rows),
                                max_kv_len=int(x.kv_lens.max()), return_lse=True)
        assert torch.equal(out, ref), f"{shape} seed {seed}: out differs from gqa_attn_decode"
        assert torch.equal(lse, ref_lse), f"{shape} seed {seed}: lse differs from gqa_attn_decode"


def test_noalloc_refuses_sizes_past_its_area():
    """A call whose gqa_attn_decode_workspace_size exceeds the 16 MiB area is refused
    with GQA_ERR_WORKSPACE before any launch."""
    lib = _lib.load()
    x = S.make_decode(2, 16, 2, [32, 32], [40000, 40000], Lcap=40000, seed=33, pad_value=None)
    T, Hq, _ = x.q.shape
    B, Hkv = x.k_cache.shape[:2]
    assert G.decode_workspace_size(B, T, Hq, Hkv, 32, 40000) > LIMIT
    q = x.q.to(DEV)
    kc = x.k_cache.to(DEV)
    kv, cu = x.kv_lens.to(DEV), x.cu_rows.to(DEV)
    out = torch.empty_like(q)
    assert _noalloc(lib, x, q, kc, kc, None, kv, cu, out, None) == GQA_ERR_WORKSPACE
