"""The output gate sigmoid(G) over every 16-bit gate value.

The gate is one fp32 computation (an ex2 and a reciprocal instruction) followed by
the output's one rounding to bf16 / fp16, in every kernel that applies it.  These
tests feed all 65,536 bit patterns of the gate type through three such epilogues
with O / l = 1 exactly, so that each output is sigmoid(G) rounded once, and compare
it with the float64 logistic function (the oracle's sigmoid):

  * attn_lse_merge with one part (O = 1, lse = 0): the merge kernel's gate;
  * gqa_attn_prefill (and its fp16 twin) with Q = K = 0 and V = 1 (every
    probability equal, every O row exactly l), on a short prompt (single CTAs) and a
    2048-row one (CTA pairs): the prefill epilogues, which compute the gate on packed
    pairs.

Bar: within half an ulp of the output type at the float64 value, plus 2^-20 relative
for the fp32 pipeline (a few fp32 ulp); +inf gives exactly 1, -inf exactly 0, NaN
stays NaN; where the float64 value lies below fp32's smallest normal the pipeline
flushes, and 0 is accepted there."""
import numpy as np
import pytest
import torch

import gqa_head_gated_gb300 as G
import oracle
from tests.parity import to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda"
DTYPES = [torch.bfloat16, torch.float16]
IDS = ["bf16", "fp16"]


def every_value(dtype):
    """All 65,536 bit patterns of a 16-bit type, in bit order."""
    return torch.arange(65536, dtype=torch.int32).to(torch.int16).view(dtype)


def check_gate(got, g, dtype, what):
    got = to_f64(got).reshape(-1)
    gv = g.reshape(-1).to(torch.float64).numpy()
    with np.errstate(over="ignore"):
        ref = oracle.sigmoid(gv)
    nan = np.isnan(gv)
    assert np.isnan(got[nan]).all(), f"{what}: a NaN gate did not give NaN"
    fin = ~nan
    assert not np.isnan(got[fin]).any(), f"{what}: NaN output for a non-NaN gate"
    assert (got[gv == np.inf] == 1.0).all(), f"{what}: sigmoid(+inf) != 1"
    assert (got[gv == -np.inf] == 0.0).all(), f"{what}: sigmoid(-inf) != 0"
    mant = 7 if dtype == torch.bfloat16 else 10
    sub_half = 2.0 ** -134 if dtype == torch.bfloat16 else 2.0 ** -25   # half the smallest subnormal
    r, x = ref[fin], got[fin]
    tiny = 2.0 ** -126
    e = np.floor(np.log2(np.maximum(r, tiny)))
    bound = np.maximum(2.0 ** (e - mant - 1), sub_half) + r * 2.0 ** -20
    ok = np.abs(x - r) <= bound
    ok |= (r < tiny) & (x == 0.0)
    bad = np.nonzero(~ok)[0]
    assert bad.size == 0, (f"{what}: {bad.size} gate values off, e.g. g={gv[fin][bad[:4]]} "
                           f"got {x[bad[:4]]} want {r[bad[:4]]}")


@pytest.mark.parametrize("dtype", DTYPES, ids=IDS)
def test_gate_every_value_merge(dtype):
    g = every_value(dtype).reshape(256, 256).contiguous()
    o = torch.ones((1, 256, 256), dtype=torch.float32, device=DEV)
    lse = torch.zeros((1, 256), dtype=torch.float32, device=DEV)
    out = G.lse_merge(o, lse, g=g.to(DEV))
    torch.cuda.synchronize()
    assert G.last_device_status() == 0
    check_gate(out, g, dtype, "merge")


@pytest.mark.parametrize("pair", [False, True], ids=["single_cta", "cta_pair"])
@pytest.mark.parametrize("dtype", DTYPES, ids=IDS)
def test_gate_every_value_prefill(dtype, pair):
    # Q = K = 0 gives every visible key probability 1, and V = 1 makes every O row
    # equal its l.  Single CTAs: 4 heads x 64 causal rows x 256 dims = 65,536 gate
    # elements.  CTA pairs: one head of 2048 rows (the prefill call sends prompts of
    # 2048 keys or more to the pair kernel), the 65,536 values repeated 8 times.
    B, H, L = (1, 1, 2048) if pair else (1, 4, 64)
    reps = B * H * L * 256 // 65536
    g = every_value(dtype).repeat(reps).reshape(B, H, L, 256).contiguous()
    q = torch.zeros((B, H, L, 256), dtype=dtype, device=DEV)
    k = torch.zeros((B, H, L, 256), dtype=dtype, device=DEV)
    v = torch.ones((B, H, L, 256), dtype=dtype, device=DEV)
    out = G.prefill(q, k, v, g.to(DEV), kv_offset=0)
    torch.cuda.synchronize()
    assert G.last_device_status() == 0
    kernel = G.launch_log(1)[0]["kernel"]
    assert kernel.startswith("attn_pair_kernel" if pair else "attn_tc_kernel<prefill"), kernel
    check_gate(out, g, dtype, kernel)
