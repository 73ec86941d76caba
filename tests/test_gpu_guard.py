"""Guard bands: every output and workspace buffer sits inside a larger allocation
whose margins hold a canary pattern; after each call the margins must be unchanged
(no write lands outside the buffer the call was given).  Stands in for a memory
checker, which this pool does not offer."""
import pytest
import torch

import gqa_head_gated_gb300 as G
from synth import inputs as S

pytestmark = pytest.mark.gpu
DEV = "cuda"
MARGIN = 4096          # bytes on each side
CANARY = 0xA5


class Guarded:
    """A tensor of `shape` / `dtype` carved out of a byte buffer with canary margins
    (16-byte aligned)."""

    def __init__(self, shape, dtype, fill=None):
        n = 1
        for d in shape:
            n *= d
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((nbytes + 2 * MARGIN,), CANARY, dtype=torch.uint8, device=DEV)
        body = self.raw[MARGIN:MARGIN + nbytes]
        self.t = body.view(dtype).view(*shape) if nbytes else body.view(dtype)
        if fill is not None:
            self.t.copy_(fill)

    def check(self, what):
        torch.cuda.synchronize()
        lo = self.raw[:MARGIN]
        hi = self.raw[self.raw.numel() - MARGIN:]
        assert torch.all(lo == CANARY) and torch.all(hi == CANARY), f"{what}: guard band written"


def test_prefill_and_masked_guard_bands():
    x = S.make_prefill(1, 24, 4, 300, Lkv=450, kv_offset=150, seed=90)
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    out = Guarded(q.shape, q.dtype)
    lse = Guarded(q.shape[:3], torch.float32)
    o, l = G.prefill(q, k, v, g, kv_offset=150, out=out.t, return_lse=True)
    lse.t.copy_(l)
    out.check("prefill out")
    m = torch.rand(300, 450, device=DEV) < 0.7
    out2 = Guarded(q.shape, q.dtype)
    G.masked(q, k, v, g, m, causal=True, kv_offset=150, out=out2.t)
    out2.check("masked out")
    assert G.last_device_status() == 0


@pytest.mark.parametrize("Hq,Hkv,rows,kv", [(24, 4, [1, 1, 1], [5000, 129, 31000]),
                                         (16, 2, [8, 32, 3], [3000, 9000, 700])])
def test_decode_verify_guard_bands(Hq, Hkv, rows, kv):
    x = S.make_decode(len(rows), Hq, Hkv, rows, kv, seed=91)
    q, kc, vc, g, kvd, cu = (t.to(DEV) for t in (x.q, x.k_cache, x.v_cache, x.g, x.kv_lens,
                                                 x.cu_rows))
    B, T = len(rows), q.shape[0]
    need = G.decode_workspace_size(B, T, Hq, Hkv, max(rows), max(kv))
    ws = Guarded((need,), torch.uint8)
    out = Guarded(q.shape, q.dtype)
    G.decode(q, kc, vc, g, kvd, cu, max_rows=max(rows), max_kv_len=max(kv), workspace=ws.t,
             out=out.t)
    ws.check("decode workspace")
    out.check("decode out")
    masks = S.random_tree_masks(rows, 5)
    tm = torch.tensor(masks, dtype=torch.int64, device=DEV)
    out3 = Guarded(q.shape, q.dtype)
    G.verify_tree(q, kc, vc, g, kvd, cu, tm, max_rows=max(rows), max_kv_len=max(kv),
                  workspace=ws.t, out=out3.t)
    ws.check("tree workspace")
    out3.check("tree out")
    S_, C_ = G.decode_plan(B, T, Hq, Hkv, max(rows), max(kv))
    op = Guarded((S_, T * Hq, 256), torch.float32)
    lp = Guarded((S_, T * Hq), torch.float32)
    G.decode_split(q, kc, vc, kvd, cu, max_rows=max(rows), max_kv_len=max(kv), num_splits=S_,
                   split_keys=C_, o_parts=op.t, lse_parts=lp.t)
    op.check("split O parts")
    lp.check("split lse parts")
    out4 = Guarded((T * Hq, 256), q.dtype)
    G.lse_merge(op.t, lp.t, g, out=out4.t)
    out4.check("merge out")
    assert G.last_device_status() == 0


def test_kv_cache_guard_bands():
    x = S.make_decode(2, 8, 2, [3, 2], [10, 7], Lcap=16, seed=92, pad_value=0.0)
    kc = Guarded(x.k_cache.shape, x.k_cache.dtype, x.k_cache.to(DEV))
    vc = Guarded(x.v_cache.shape, x.v_cache.dtype, x.v_cache.to(DEV))
    gen = torch.Generator().manual_seed(93)
    kn = torch.randn(5, 2, 256, generator=gen).to(torch.bfloat16).to(DEV)
    G.kv_append(kn, kn, x.kv_lens.to(DEV), kc.t, vc.t, x.cu_rows.to(DEV))
    kc.check("append K cache")
    vc.check("append V cache")
    lens_out = Guarded((2,), torch.int32)
    G.kv_keep(kc.t, vc.t, torch.tensor([13, 9], dtype=torch.int32, device=DEV),
              x.cu_rows.to(DEV), torch.tensor([0, 2, 1], dtype=torch.int32, device=DEV),
              torch.tensor([0, 2, 3], dtype=torch.int32, device=DEV), lens_out.t)
    kc.check("keep K cache")
    lens_out.check("keep lengths")
    assert lens_out.t.tolist() == [12, 8]
    assert G.last_device_status() == 0
