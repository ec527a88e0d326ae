"""The split-BF16 operand format, checked on the host in exact arithmetic.

Each operand is held as hi = bf16(v) and lo = bf16(v - hi), both rounded to
nearest even (torch's float32 -> bfloat16 conversion).  v - hi is exact in fp32
and |v - hi - lo| <= 2^-16 |v|; a product a*b computed as a_hi*b_hi + a_hi*b_lo
+ a_lo*b_hi (exact bf16 products, as on the tensor cores) is within about
3 * 2^-16 of a*b relative to |a*b|.  These are the bounds the library's header
states for CONVT3D_PREC_3XBF16.
"""
import numpy as np
import torch


def split(v):
    hi = v.to(torch.bfloat16).to(torch.float32)
    rem = v - hi                       # exact in fp32: hi is v rounded to 8 significant bits
    lo = rem.to(torch.bfloat16).to(torch.float32)
    return hi, lo, rem


def test_remainder_is_exact_and_split_bound_holds():
    g = torch.Generator().manual_seed(7)
    v = torch.randn(200_000, generator=g, dtype=torch.float32) * torch.exp(
        torch.randn(200_000, generator=g, dtype=torch.float32) * 4)
    hi, lo, rem = split(v)
    v64, hi64, lo64 = v.double(), hi.double(), lo.double()
    assert torch.equal(rem.double(), v64 - hi64)      # the subtraction lost nothing
    err = (v64 - hi64 - lo64).abs()
    assert torch.all(err <= 2.0 ** -16 * v64.abs())
    # the bound is nearly attained: two 8-bit halves of a 16-bit significand
    assert (err / v64.abs().clamp_min(1e-300)).max() > 2.0 ** -18


def test_three_products_match_the_fp64_product():
    g = torch.Generator().manual_seed(11)
    a = torch.randn(100_000, generator=g, dtype=torch.float32)
    b = torch.randn(100_000, generator=g, dtype=torch.float32)
    ah, al, _ = split(a)
    bh, bl, _ = split(b)
    p3 = ah.double() * bh.double() + ah.double() * bl.double() + al.double() * bh.double()
    exact = a.double() * b.double()
    rel = ((p3 - exact).abs() / exact.abs().clamp_min(1e-300)).numpy()
    assert rel.max() <= 3 * 2.0 ** -16
    # a sum of K such products with random signs stays far inside the 1e-4 bar
    K = 1728
    s3 = p3[:K * 50].reshape(50, K).sum(1)
    se = exact[:K * 50].reshape(50, K).sum(1)
    scale = exact[:K * 50].reshape(50, K).abs().sum(1)
    assert np.all(((s3 - se).abs() / scale).numpy() < 1e-5)


def test_single_bf16_is_not_enough():
    # one bf16 product per term (CONVT3D_PREC_BF16) misses the fp32 bar by orders of magnitude
    g = torch.Generator().manual_seed(13)
    a = torch.randn(10_000, generator=g, dtype=torch.float32)
    b = torch.randn(10_000, generator=g, dtype=torch.float32)
    p1 = a.to(torch.bfloat16).double() * b.to(torch.bfloat16).double()
    rel = ((p1 - a.double() * b.double()).abs() / (a.double() * b.double()).abs()).max().item()
    assert rel > 1e-3
