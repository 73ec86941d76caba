"""The seeded generators reproduce the recorded structural draws of the named
workloads (so that byte and FLOP counts quoted for them stay valid)."""
import torch

from synth import inputs as S


def test_decode_27b_kv_lens():
    gen = torch.Generator().manual_seed(1)
    kv = torch.randint(1024, 32769, (16,), generator=gen).tolist()
    assert kv == [12224, 32233, 30428, 5997, 16112, 23507, 12035, 2695, 15808, 28411, 1987,
                  24298, 8540, 23877, 30797, 28679]
    assert sum(kv) == 297628


def test_verify_35b_structure():
    gen = torch.Generator().manual_seed(4)
    kv = torch.randint(4097, 65537, (8,), generator=gen).tolist()
    assert kv == [21627, 4271, 22968, 21190, 38786, 18793, 20056, 45513]
    rows = [S.VERIFY_ROWS[b % 6] for b in range(8)]
    assert rows == [1, 3, 4, 8, 16, 32, 1, 3]


def test_small_decode_layout():
    x = S.make_decode(3, 4, 2, rows=[2, 0, 1], kv_lens=[3, 1, 4], Lcap=5, seed=7)
    assert x.q.shape == (3, 4, 256) and x.g.shape == (3, 4, 256)
    assert x.cu_rows.tolist() == [0, 2, 2, 3]
    assert torch.isnan(x.k_cache[0, :, 3:].float()).all()
    assert torch.isfinite(x.k_cache[0, :, :3].float()).all()
    assert x.q.dtype == torch.bfloat16


def test_prefill_outliers_exact_x8():
    x = S.make_prefill(1, 4, 2, 200, seed=2, outlier_frac=0.01)
    gen = torch.Generator().manual_seed(2)
    perms = [torch.randperm(200, generator=gen)[:2].tolist() for _ in range(2)]
    torch.randn(1, 4, 200, 256, generator=gen)                       # Q
    k0 = torch.randn(1, 2, 200, 256, generator=gen).to(torch.bfloat16)  # K before scaling
    assert x.meta["outliers"] == perms
    kx = x.k.view(2, 200, 256).float()
    k0 = k0.view(2, 200, 256).float()
    for g in range(2):
        for j in range(200):
            want = k0[g, j] * 8 if j in perms[g] else k0[g, j]
            assert torch.equal(kx[g, j], want)


def test_fp16_inputs_are_the_same_draws():
    """fp16 inputs are the same float32 draws as the bf16 ones, rounded to fp16:
    the two agree to bf16's rounding (2^-8 relative), and the fp16 values are
    finer (fp16 keeps 10 mantissa bits)."""
    a = S.make_decode(2, 4, 2, rows=[2, 1], kv_lens=[5, 3], Lcap=7, seed=9)
    b = S.make_decode(2, 4, 2, rows=[2, 1], kv_lens=[5, 3], Lcap=7, seed=9, dtype=torch.float16)
    assert b.q.dtype == torch.float16 and b.k_cache.dtype == torch.float16
    for x, y in ((a.q, b.q), (a.g, b.g), (a.k_cache[0, :, :5], b.k_cache[0, :, :5])):
        xf, yf = x.float(), y.float()
        assert torch.all((xf - yf).abs() <= xf.abs() * 2.0 ** -8 + 1e-30)
        assert torch.equal(yf.half().float(), yf)
    assert torch.isnan(b.k_cache[0, :, 5:]).all()
    p = S.make_prefill(1, 2, 1, 9, seed=3, outlier_frac=0.2, dtype=torch.float16)
    assert p.q.dtype == torch.float16 and p.k.dtype == torch.float16
