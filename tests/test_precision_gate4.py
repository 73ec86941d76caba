"""Gate 4 of the TensorFold attention contract (PR #1009, "Receipt"): inputs on
which bf16 accumulation of score sums or softmax sums misses the tolerance by at
least 100x while fp32 accumulation passes.  The separation is shown on the CPU by
simulating both accumulations (round to bf16 after every addition, as a kernel
keeping those sums in bf16 would); the GPU kernels must then pass.

* Row sums: 4096 keys with equal scores, V rows of +2 for the first half and -2 for
  the second; float64 gives 0.  A bf16 running sum of p stalls at 256 and the bf16
  running O at +512, then walks down to -512: out = -2, 100x the 2e-2 bound.
* Score sums: q = 8 in every dimension, keys of +-8.125 with small per-key offsets,
  the first half of the dimensions positive and the second negative, so the exact
  dot products are small sums of large terms; a bf16 running dot product is off by
  nats, thousands of times the 2e-3 lse bound.
"""
import numpy as np
import pytest
import torch

from synth import inputs as S
from tests.parity import MAX_ABS, errors, to_f64

D = 256


def _bf(x):
    return x.to(torch.bfloat16).to(torch.float64)


def rowsum_inputs(L=4096):
    """Decode layout: one sequence, 8 query heads over 1 KV head, one row."""
    gen = torch.Generator().manual_seed(41)
    q = torch.randn(1, 8, D, generator=gen).to(torch.bfloat16)
    k = torch.randn(1, 1, 1, D, generator=gen).expand(1, 1, L, D).to(torch.bfloat16).contiguous()
    v = torch.full((1, 1, L, D), 2.0)
    v[:, :, L // 2:] = -2.0
    return q, k, v.to(torch.bfloat16)


def scoresum_inputs(L=64):
    gen = torch.Generator().manual_seed(42)
    q = torch.full((1, 4, D), 8.0)
    base = torch.full((L, D), 8.125)
    base[:, D // 2:] *= -1
    k = base + torch.randint(-2, 3, (L, D), generator=gen).to(torch.float32) * 0.0625
    v = torch.randn(L, D, generator=gen)
    return (q.to(torch.bfloat16), k.reshape(1, 1, L, D).to(torch.bfloat16),
            v.reshape(1, 1, L, D).to(torch.bfloat16))


def simulate(q, k, v, bf16_scores, bf16_sums):
    """One query row against the keys, accumulating in bf16 or float64 as asked."""
    q = q.double()
    k = k.double()
    v = v.double()
    if bf16_scores:
        acc = torch.zeros(k.shape[0], dtype=torch.float64)
        for d in range(D):
            acc = _bf(acc + k[:, d] * q[d])
        s = acc / 16
    else:
        s = (k @ q) / 16
    p = torch.exp(s - s.max())
    if bf16_sums:
        o = torch.zeros(D, dtype=torch.float64)
        l = torch.zeros((), dtype=torch.float64)
        for j in range(k.shape[0]):
            o = _bf(o + _bf(p[j]) * v[j])
            l = _bf(l + _bf(p[j]))
    else:
        o, l = p @ v, p.sum()
    return o / l, s.max() + torch.log(p.sum())


def test_rowsum_separation_on_cpu():
    q, k, v = rowsum_inputs()
    exact, _ = simulate(q[0, 0], k[0, 0], v[0, 0], False, False)
    bad, _ = simulate(q[0, 0], k[0, 0], v[0, 0], False, True)
    assert torch.all(exact.abs() < 1e-12)
    assert (bad - exact).abs().max().item() >= 100 * MAX_ABS


def test_scoresum_separation_on_cpu():
    q, k, v = scoresum_inputs()
    _, lse_exact = simulate(q[0, 0], k[0, 0], v[0, 0], False, False)
    _, lse_bad = simulate(q[0, 0], k[0, 0], v[0, 0], True, False)
    assert abs(lse_bad - lse_exact).item() >= 100 * 2e-3
    # the fp32 sum of the same products is exact here (integers times 1/256)
    acc32 = torch.zeros(k.shape[2], dtype=torch.float32)
    for d in range(D):
        acc32 = acc32 + (k[0, 0, :, d].float() * q[0, 0, d].float())
    assert torch.equal(acc32.double(), k[0, 0].double() @ q[0, 0].double())


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["rowsum", "scoresum"])
@pytest.mark.parametrize("path", ["decode", "prefill"])
def test_gpu_passes_gate4(case, path):
    import gqa_head_gated_gb300 as G
    import oracle
    from tests.parity import assert_parity
    q, k, v = rowsum_inputs() if case == "rowsum" else scoresum_inputs()
    Hq, L = q.shape[1], k.shape[2]
    if path == "decode":
        out, lse = G.decode(q.cuda(), k.cuda(), v.cuda(), None,
                            torch.tensor([L], dtype=torch.int32, device="cuda"), None,
                            max_rows=1, max_kv_len=L, return_lse=True)
        r_out, r_lse = oracle.decode(to_f64(q), to_f64(k), to_f64(v), None, [L])
    else:   # the row as the last prompt row of a prefill over the same keys
        qp = q.reshape(1, Hq, 1, D).contiguous()
        out, lse = G.prefill(qp.cuda(), k.cuda(), v.cuda(), None, kv_offset=L - 1,
                             return_lse=True)
        r_out, r_lse = oracle.prefill(to_f64(qp), to_f64(k), to_f64(v), None, kv_offset=L - 1)
    assert G.last_device_status() == 0
    if case == "rowsum":
        # float64 gives exactly 0 here; the median relative error is undefined at 0,
        # so the bound is the absolute one (a split merge leaves ~1e-7 of rounding)
        e = errors(out, r_out)
        assert e["nonfinite"] == 0 and e["max_abs"] <= MAX_ABS, e
    else:
        assert_parity(out, r_out, f"gate 4 {case} {path}")
    np.testing.assert_allclose(to_f64(lse), r_lse, rtol=0, atol=2e-3)
