"""GPU parity of the direct-input tensor-core kernel (direct.cu) against the CPU oracle.

Plans with stride 2 along w, at most 32 input channels, at most 64 output
channels, NCDHW fp32 tensors, an identity or softmax+sigmoid epilogue and bf16
operands (split BF16, BF16 or FP16), and q-grid rows of 8, 16, 32, 64 or 128
positions, read x straight from the caller's tensor: one TMA slab per input
d-slice, operands built on chip.  The cases cover 16 to 1 q-rows per tile,
ragged channel counts, w-parity classes of different width, three merged w
offsets, an h halo, stride 1 along d, tiles whose d-slices all fall outside the
input (no products: bias only), no bias, and the full-size softmax workload;
each asserts that the plan runs this kernel.
"""
import numpy as np
import pytest

import workloads as E
from test_parity_gpu import TOL, TOL_LOW_VS_FP32, assert_close, rounded_inputs, run_gpu, run_oracle
from transposed_convolution_convt3d_gb300 import PREC_3XBF16, PREC_BF16, PREC_FP16, Plan

DIRECT = [
    E.Spec("direct_softmax_w8", N=2, Cin=32, Cout=64, D=4, H=6, W=8, k=3, stride=2, pad=1, out_pad=1, bias=True,
           epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=80),
    # Cin 17 (ragged channels), Cout 40, odd output width: class widths 16 and 15
    E.Spec("direct_softmax_ragged", N=1, Cin=17, Cout=40, D=3, H=5, W=16, k=3, stride=2, pad=1, out_pad=0,
           bias=True, epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=81),
    # k = 4: three merged w offsets, an h halo of one row
    E.Spec("direct_identity_k4", N=2, Cin=8, Cout=24, D=3, H=4, W=16, k=4, stride=2, pad=1, bias=True,
           seed_index=82),
    E.Spec("direct_softmax_k2_nobias", N=1, Cin=3, Cout=16, D=2, H=3, W=8, k=2, stride=2,
           epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=83),
    E.Spec("direct_softmax_c33", N=1, Cin=32, Cout=33, D=3, H=7, W=16, k=3, stride=2, pad=1, out_pad=1,
           bias=True, epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=84),
    # one q-row per tile: Qw = 128
    E.Spec("direct_wide_w128", N=1, Cin=16, Cout=32, D=2, H=3, W=128, k=3, stride=2, pad=1, out_pad=1,
           bias=True, epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=85),
    # two q-rows per tile: Qw = 64
    E.Spec("direct_w64", N=1, Cin=32, Cout=64, D=2, H=3, W=64, k=3, stride=2, pad=1, out_pad=1,
           bias=True, epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=89),
    # stride 1 along d (one pair per h parity, three d-slices)
    E.Spec("direct_stride_d1", N=1, Cin=20, Cout=24, D=3, H=4, W=8, k=3, stride=(1, 2, 2), pad=(1, 1, 1),
           out_pad=(0, 1, 1), bias=True, epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=86),
    # dilation 3 along d with k = 2: the first and last output d-planes of each parity
    # receive no input (their tiles have no live d-slice and hold the bias alone)
    E.Spec("direct_dead_tiles", N=2, Cin=8, Cout=16, D=2, H=3, W=8, k=(2, 3, 3), stride=2, pad=(0, 1, 1),
           out_pad=(0, 1, 1), dilation=(3, 1, 1), bias=True, seed_index=87),
    E.Spec("direct_dead_tiles_softmax", N=1, Cin=8, Cout=16, D=2, H=3, W=8, k=(2, 3, 3), stride=2,
           pad=(0, 1, 1), out_pad=(0, 1, 1), dilation=(3, 1, 1), bias=True, epilogue=E.EPI_SOFTMAX_SIGMOID,
           seed_index=88),
]


def main_kernel(spec, precision):
    return Plan.from_spec(spec, precision=precision).info["main_kernel"]


@pytest.mark.gpu
@pytest.mark.parametrize("spec", DIRECT, ids=lambda s: s.name)
def test_direct_split_bf16(spec):
    assert main_kernel(spec, PREC_3XBF16) == 2
    inputs = E.make_inputs(spec)
    assert_close(run_gpu(spec, inputs, PREC_3XBF16), run_oracle(spec, inputs), spec.name)


@pytest.mark.gpu
@pytest.mark.parametrize("spec", DIRECT, ids=lambda s: s.name)
def test_direct_bf16(spec):
    """One product of bf16-rounded operands: equal to the oracle on identically
    rounded x and w within the fp32 tolerance."""
    assert main_kernel(spec, PREC_BF16) == 2
    inputs = E.make_inputs(spec)
    got = run_gpu(spec, inputs, PREC_BF16)
    assert_close(got, run_oracle(spec, rounded_inputs(inputs, PREC_BF16)), spec.name, TOL)


@pytest.mark.gpu
@pytest.mark.parametrize("spec", DIRECT[:4] + DIRECT[6:8], ids=lambda s: s.name)
def test_direct_fp16(spec):
    """One product of fp16-rounded operands (kind::f16 with fp16 A and B): equal to the
    oracle on identically rounded x and w within the fp32 tolerance."""
    assert main_kernel(spec, PREC_FP16) == 2
    inputs = E.make_inputs(spec)
    got = run_gpu(spec, inputs, PREC_FP16)
    assert_close(got, run_oracle(spec, rounded_inputs(inputs, PREC_FP16)), spec.name, TOL)


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["bf16", "fp16"])
@pytest.mark.parametrize("spec", DIRECT[:4] + DIRECT[6:8], ids=lambda s: s.name)
def test_direct_16bit_tensors(spec, kind):
    """x, w and y as 16-bit arrays in the operands' format (BF16 / FP16 precision): the slab
    holds the operands and y is rounded once more on the way out, so the oracle on
    identically rounded x and w is matched within the 1e-2 tier."""
    s = spec.replace(name=spec.name + "_io" + kind, io_bf16=kind == "bf16", io_fp16=kind == "fp16")
    prec = PREC_BF16 if kind == "bf16" else PREC_FP16
    assert main_kernel(s, prec) == 2
    inputs = E.make_inputs(s)
    got = run_gpu(s, inputs, prec)
    assert_close(got, run_oracle(s, rounded_inputs(inputs, prec)), s.name, TOL_LOW_VS_FP32)


@pytest.mark.gpu
def test_direct_full_size_softmax():
    spec = E.SOFTMAX
    assert main_kernel(spec, PREC_3XBF16) == 2
    inputs = E.make_inputs(spec)
    got = run_gpu(spec, inputs, PREC_3XBF16)
    for n in (0, spec.N // 2, spec.N - 1):
        sub = E.sample_slice(inputs, n, n + 1)
        assert_close(got[n:n + 1], run_oracle(spec.replace(N=1), sub), f"{spec.name}[n={n}]")


@pytest.mark.gpu
def test_direct_repeat_is_bitwise_deterministic():
    spec = DIRECT[1]
    inputs = E.make_inputs(spec)
    a = run_gpu(spec, inputs, PREC_3XBF16)
    b = run_gpu(spec, inputs, PREC_3XBF16)
    assert np.array_equal(a, b)
