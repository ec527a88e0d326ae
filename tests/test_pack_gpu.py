"""The packed split-BF16 weight planes, read back from the workspace.

The header states that the split-BF16 precision represents each operand as
hi = bf16(v) and lo = bf16(v - hi), both rounded to nearest even, so that
|v - hi - lo| <= 2^-16 |v|.  tests/test_split_bf16_bound.py proves the bound
for that split in exact arithmetic on the host; this test pins the device's
own split: it packs a weight with CONVT3D_PREC_3XBF16, copies the hi and lo
planes out of the workspace, and requires them to equal the host split bit
for bit (PyTorch's float32 -> bfloat16 conversion is also round to nearest
even) and to meet the bound.

Workspace layout (the library's, for a stride-1 problem): a 256-byte status
word, then the hi plane [tap][cout_pad][cin_pad] of bf16 (cin_pad a multiple
of 64, cout_pad of 16), then the lo plane at the next 256-byte boundary.  With
stride 1 there is one parity class whose taps are the kernel's in order, so
packed[j][co][ci] = w[ci][co][j].
"""
import numpy as np
import pytest
import torch

import workloads as E
from transposed_convolution_convt3d_gb300 import PREC_3XBF16, Plan


def _round_up(v, a):
    return (v + a - 1) // a * a


@pytest.mark.gpu
def test_split_bf16_planes_match_host_split_bitwise():
    spec = E.Spec("pack_split_bf16", N=1, Cin=40, Cout=24, D=2, H=2, W=2, k=3, seed_index=70)
    g = torch.Generator().manual_seed(70)
    # magnitudes over many binades, so rounding happens at every exponent
    w = torch.randn((spec.Cin, spec.Cout, 3, 3, 3), generator=g) * \
        torch.exp2(torch.randint(-30, 30, (spec.Cin, spec.Cout, 3, 3, 3), generator=g).float())
    dev = torch.device("cuda")
    plan = Plan.from_spec(spec, precision=PREC_3XBF16)
    ws = plan.new_workspace(dev)
    ws.zero_()
    plan.pack_weights(w.to(dev), ws)
    torch.cuda.synchronize()

    taps, cin_pad, cout_pad = 27, _round_up(spec.Cin, 64), _round_up(spec.Cout, 16)
    n = taps * cout_pad * cin_pad
    off_hi = 256
    off_lo = _round_up(off_hi + 2 * n, 256)
    raw = ws.cpu()
    hi = raw[off_hi:off_hi + 2 * n].view(torch.bfloat16).reshape(taps, cout_pad, cin_pad)
    lo = raw[off_lo:off_lo + 2 * n].view(torch.bfloat16).reshape(taps, cout_pad, cin_pad)

    v = w.reshape(spec.Cin, spec.Cout, taps).permute(2, 1, 0).contiguous()  # [tap][co][ci]
    ref_hi = v.to(torch.bfloat16)
    ref_lo = (v - ref_hi.float()).to(torch.bfloat16)
    got_hi = hi[:, :spec.Cout, :spec.Cin].contiguous()
    got_lo = lo[:, :spec.Cout, :spec.Cin].contiguous()
    assert torch.equal(got_hi.view(torch.int16), ref_hi.view(torch.int16))
    assert torch.equal(got_lo.view(torch.int16), ref_lo.view(torch.int16))
    # the padding rows and columns are zero
    assert not hi[:, spec.Cout:, :].float().any() and not hi[:, :, spec.Cin:].float().any()
    assert not lo[:, spec.Cout:, :].float().any() and not lo[:, :, spec.Cin:].float().any()

    vv = v.double().numpy()
    resid = np.abs(vv - got_hi.double().numpy() - got_lo.double().numpy())
    assert np.all(resid <= 2.0 ** -16 * np.abs(vv))
