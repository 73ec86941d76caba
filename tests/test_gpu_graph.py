"""The C ABI calls are stream-ordered and allocate nothing, so they can be captured
in a CUDA graph (after one eager call on the device, which looks up the device
status word): a replay gives the eager outputs bit for bit, and replays with new
inputs copied into the captured buffers follow the new inputs."""
import pytest
import torch

import gqa_head_gated_gb300 as G
from synth import inputs as S

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_decode_and_verify_graph_replay():
    for rows, Hq, Hkv in (([1] * 6, 24, 4), ([8, 32, 3], 16, 2)):
        x = S.make_decode(len(rows), Hq, Hkv, rows, [4000, 9000, 700, 3000, 50, 12000][:len(rows)],
                          seed=95)
        q, kc, vc, g, kv, cu = (t.to(DEV) for t in (x.q, x.k_cache, x.v_cache, x.g, x.kv_lens,
                                                     x.cu_rows))
        B, T = len(rows), q.shape[0]
        mk = int(x.kv_lens.max())
        ws = torch.empty(G.decode_workspace_size(B, T, Hq, Hkv, max(rows), mk), dtype=torch.uint8,
                         device=DEV)
        out = torch.empty_like(q)
        eager = G.decode(q, kc, vc, g, kv, cu, max_rows=max(rows), max_kv_len=mk, workspace=ws)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            G.decode(q, kc, vc, g, kv, cu, max_rows=max(rows), max_kv_len=mk, workspace=ws,
                     out=out)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
        # new query rows through the captured buffers
        q2 = torch.randn(q.shape, generator=torch.Generator().manual_seed(96)).to(q.dtype).to(DEV)
        q.copy_(q2)
        graph.replay()
        ref = G.decode(q2, kc, vc, g, kv, cu, max_rows=max(rows), max_kv_len=mk)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
        assert G.last_device_status() == 0


def test_prefill_graph_replay():
    x = S.make_prefill(1, 16, 2, 300, Lkv=500, kv_offset=200, seed=97)
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    eager = G.prefill(q, k, v, g, kv_offset=200)
    out = torch.empty_like(q)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        G.prefill(q, k, v, g, kv_offset=200, out=out)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert G.last_device_status() == 0
