"""The library's launch log (gqa_launch_log) reports the kernels a call launched with
the grid, block and dynamic shared memory they ran with."""
import pytest
import torch

import gqa_head_gated_gb300 as G
from synth import inputs as S

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_prefill_launch_is_logged():
    x = S.make_prefill(1, 24, 4, 300, seed=5)
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    G.prefill(q, k, v, g, kv_offset=0)
    torch.cuda.synchronize()
    rec = G.launch_log(1)[0]
    R = 128 // 6
    assert rec["kernel"] == "attn_tc_kernel<prefill,bf16>"
    assert rec["grid"] == -(-300 // R) * 4 and rec["block"] == 320
    assert rec["dynamic_smem"] > 200 * 1024


def test_long_prefill_runs_on_cta_pairs():
    """A prompt whose last row sees 2048 keys or more runs on the CTA-pair kernel:
    clusters of two CTAs over pairs of row tiles."""
    x = S.make_prefill(1, 24, 4, 2048, seed=7)
    q, k, v, g = (t.to(DEV) for t in (x.q, x.k, x.v, x.g))
    G.prefill(q, k, v, g, kv_offset=0)
    torch.cuda.synchronize()
    rec = G.launch_log(1)[0]
    R = 128 // 6
    n_rtiles = -(-2048 // R)
    assert rec["kernel"] == "attn_pair_kernel<prefill,bf16>"
    assert rec["grid"] == 2 * ((n_rtiles + 1) // 2) * 4 and rec["block"] == 320


def test_decode_launches_are_logged_in_order():
    x = S.make_decode(4, 24, 4, [1] * 4, [900, 50, 3000, 128], seed=6)
    q, kc, vc, g = (t.to(DEV) for t in (x.q, x.k_cache, x.v_cache, x.g))
    kv = x.kv_lens.to(DEV)
    before = G.launch_log(1)
    G.decode(q, kc, vc, g, kv, None, max_rows=1, max_kv_len=3000)
    torch.cuda.synchronize()
    merge, split = G.launch_log(2)
    if before:
        assert split["seq"] == before[0]["seq"] + 1
    assert merge["seq"] == split["seq"] + 1
    assert split["kernel"].startswith("decode_split_kernel<") and split["kernel"].endswith("balanced")
    assert split["block"] == 128
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert split["grid"] % sms == 0
    assert merge["kernel"] == "lse_merge_kernel<bf16> dependent"
