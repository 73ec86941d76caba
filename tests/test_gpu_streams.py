"""The library keeps no per-call host state: calls on two CUDA streams, issued back to
back and running concurrently on the device, give the same bits as the same calls
run one after the other."""
import pytest
import torch

import gqa_head_gated_gb300 as G
from synth import inputs as S

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_prefill_and_decode_on_two_streams():
    xp = S.make_prefill(1, 24, 4, 700, seed=120)
    xd = S.make_decode(6, 16, 2, [1, 3, 8, 32, 1, 2], [3000, 900, 5000, 12000, 64, 700],
                       seed=121)
    q, k, v, g = (t.to(DEV) for t in (xp.q, xp.k, xp.v, xp.g))
    dq, kc, vc, dg, kv, cu = (t.to(DEV) for t in (xd.q, xd.k_cache, xd.v_cache, xd.g,
                                                   xd.kv_lens, xd.cu_rows))
    mr, mk = max(xd.rows), int(xd.kv_lens.max())
    ref_p = G.prefill(q, k, v, g, kv_offset=0)
    ref_d = G.decode(dq, kc, vc, dg, kv, cu, max_rows=mr, max_kv_len=mk)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(s1):
            op = G.prefill(q, k, v, g, kv_offset=0)
        with torch.cuda.stream(s2):
            od = G.decode(dq, kc, vc, dg, kv, cu, max_rows=mr, max_kv_len=mk)
        outs.append((op, od))
    torch.cuda.synchronize()
    for op, od in outs:
        assert torch.equal(op, ref_p)
        assert torch.equal(od, ref_d)
    assert G.last_device_status() == 0
