"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle.

Same seeded inputs on both sides; every output element must satisfy
|gpu - oracle| <= 1e-4 * (1 + |oracle|), the tolerance the method is held to.
Small cases span several tiles with ragged tails, odd extents, channel counts
that are not multiples of the K chunk and the degenerate sizes; the five
workloads run at full size and are compared on whole samples the oracle can
compute (GroupNorm, softmax and identity are per sample; BatchNorm's batch
statistics need the whole batch, which the oracle computes in full).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from transposed_convolution_convt3d_gb300 import (PREC_3XBF16, PREC_3XTF32, PREC_BF16, PREC_FFMA, PREC_FP16,
                                                  PREC_TF32, Plan)

TOL = 1e-4
# The fp32-accurate paths, all held to the same 1e-4 bar: split TF32 (the method's),
# split BF16 (hi/lo bf16 planes, three products; operands represented to
# 2^-16 relative) and the FFMA ablation.
PRECISIONS = [pytest.param(PREC_3XTF32, id="3xtf32"), pytest.param(PREC_3XBF16, id="3xbf16"),
              pytest.param(PREC_FFMA, id="ffma")]


def run_gpu(spec, inputs, precision, running=None, momentum=0.1):
    """Forward on the GPU.  running: (mean, var) CPU tensors; they are copied to
    the device, attached to the plan, and their values after the forward are
    returned beside y."""
    dev = torch.device("cuda")
    plan = Plan.from_spec(spec, precision=precision)
    ws = plan.new_workspace(dev)
    y = plan.new_output(dev)
    y.fill_(float("nan"))
    d = {k: (v.to(dev) if v is not None else None) for k, v in inputs.items()}
    if spec.channels_last:  # same values, NDHWC memory order
        d["x"] = d["x"].permute(0, 2, 3, 4, 1).contiguous()
    if spec.io_bf16:  # x and w handed over as bf16 tensors
        d["x"], d["w"] = d["x"].to(torch.bfloat16), d["w"].to(torch.bfloat16)
    if spec.io_fp16:  # x and w handed over as fp16 tensors
        d["x"], d["w"] = d["x"].to(torch.float16), d["w"].to(torch.float16)
    if running is not None:
        rm, rv = (t.to(dev).clone() for t in running)
        plan.set_running_stats(rm, rv, momentum)
    plan.pack_weights(d["w"], ws)
    plan.forward(d["x"], y, ws, d["bias"], d["gamma"], d["beta"])
    plan.check(ws)
    if spec.channels_last and y.dim() == 5 and tuple(y.shape) != plan.out_shape:
        y = y.permute(0, 4, 1, 2, 3)  # back to NCDHW for the comparison
    y = y.float().contiguous()
    if running is not None:
        return y.cpu().numpy(), rm.cpu().numpy(), rv.cpu().numpy()
    return y.cpu().numpy()


def run_oracle(spec, inputs, running=None, momentum=0.1):
    """The oracle's output; with running=(mean, var) CPU tensors, also the
    running statistics after the forward (the oracle updates copies)."""
    f = lambda t: None if t is None else t.numpy()  # noqa: E731
    rm = rv = None
    if running is not None:
        rm, rv = (t.numpy().copy() for t in running)
    out = oracle.forward(f(inputs["x"]), f(inputs["w"]), f(inputs["bias"]), stride=spec.stride, pad=spec.pad,
                         out_pad=spec.out_pad, dilation=spec.dilation, conv_groups=spec.conv_groups,
                         epilogue=spec.epilogue, groups=spec.groups, eps=spec.eps,
                         scale=spec.scale, gamma=f(inputs["gamma"]), beta=f(inputs["beta"]), running_mean=rm,
                         running_var=rv, momentum=momentum)
    if running is not None:
        return out, rm, rv
    return out


def assert_close(got, ref, what="", tol=TOL):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64)) / (1.0 + np.abs(ref.astype(np.float64)))
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= tol, f"{what}: max scaled err {err.max():.3e} at {worst}: got {got[worst]} ref {ref[worst]}"


E = workloads
SMALL = [
    E.TINY,
    # ReLU + GroupNorm, ragged everything: Cin 40 (not a multiple of 32), Cout 48, 12 channels per group
    E.Spec("gn_ragged", N=2, Cin=40, Cout=48, D=5, H=7, W=9, k=3, epilogue=E.EPI_RELU_GROUPNORM, groups=4,
           seed_index=11),
    E.Spec("gn_pad1_bias", N=1, Cin=16, Cout=32, D=6, H=5, W=7, k=4, pad=1, bias=True,
           epilogue=E.EPI_RELU_GROUPNORM, groups=8, seed_index=12),
    # 32 channels per group: two 16-channel chunks per group
    E.Spec("gn_cpg32", N=2, Cin=32, Cout=64, D=4, H=5, W=6, k=3, epilogue=E.EPI_RELU_GROUPNORM, groups=2,
           seed_index=25),
    # stride-2 GroupNorm (w-parity pairs feed the same groups)
    E.Spec("gn_s2", N=2, Cin=16, Cout=32, D=3, H=4, W=4, k=4, stride=2, pad=1, bias=True,
           epilogue=E.EPI_RELU_GROUPNORM, groups=2, seed_index=26),
    # scale + BatchNorm (batch statistics) + pool, k=5
    E.Spec("bn_small", N=3, Cin=20, Cout=32, D=4, H=6, W=5, k=5, bias=True,
           epilogue=E.EPI_SCALE_BATCHNORM_AVGPOOL, scale=2.0, seed_index=13),
    E.Spec("bn_k3_s2", N=2, Cin=8, Cout=16, D=3, H=4, W=5, k=3, stride=2, pad=1, out_pad=1, bias=True,
           epilogue=E.EPI_SCALE_BATCHNORM_AVGPOOL, scale=0.5, seed_index=14),
    # stride-2 softmax + sigmoid over 64 channels
    E.Spec("softmax_s2", N=2, Cin=12, Cout=64, D=5, H=6, W=7, k=3, stride=2, pad=1, out_pad=1, bias=True,
           epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=15),
    # odd output extents: w-parity classes of different length
    E.Spec("softmax_s2_odd", N=1, Cin=32, Cout=32, D=4, H=5, W=6, k=3, stride=2, pad=1, out_pad=0, bias=True,
           epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=16),
    # softmax channel counts on both sides of the register-kept limit (64), ragged chunks
    E.Spec("softmax_s2_c96", N=1, Cin=16, Cout=96, D=3, H=4, W=5, k=3, stride=2, pad=1, out_pad=1, bias=True,
           epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=27),
    E.Spec("softmax_s1_c100", N=2, Cin=20, Cout=100, D=4, H=5, W=3, k=3, bias=True,
           epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=28),
    E.Spec("softmax_s1_c40", N=1, Cin=8, Cout=40, D=3, H=3, W=5, k=2, bias=True,
           epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=29),
    # bare stride-2 k=4
    E.Spec("identity_s2_k4", N=2, Cin=36, Cout=40, D=3, H=5, W=6, k=4, stride=2, pad=1, bias=True,
           seed_index=17),
    E.Spec("identity_s2_k5_op1", N=1, Cin=24, Cout=16, D=3, H=4, W=3, k=5, stride=2, pad=2, out_pad=1,
           bias=True, seed_index=18),
    E.Spec("identity_s1_k2", N=3, Cin=7, Cout=20, D=4, H=3, W=9, k=2, seed_index=19),
    # degenerate sizes
    E.Spec("one_channel", N=1, Cin=1, Cout=1, D=1, H=1, W=1, k=3, bias=True, seed_index=20),
    E.Spec("k1", N=2, Cin=5, Cout=16, D=3, H=4, W=5, k=1, bias=True, seed_index=21),
    E.Spec("cout256", N=1, Cin=32, Cout=256, D=3, H=4, W=5, k=3, bias=True, seed_index=22),
    E.Spec("cout256_softmax", N=1, Cin=32, Cout=256, D=3, H=3, W=4, k=3, bias=True,
           epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=23),
    E.Spec("wide_w", N=1, Cin=32, Cout=32, D=2, H=3, W=200, k=3, seed_index=24),
    # the largest kernel (k = 7: tap offsets up to 6 per load), stride 1 and 2
    E.Spec("k7_s1", N=1, Cin=16, Cout=32, D=3, H=4, W=5, k=7, pad=3, bias=True, seed_index=60),
    E.Spec("k7_s2_softmax", N=1, Cin=8, Cout=48, D=2, H=3, W=4, k=7, stride=2, pad=3, out_pad=1, bias=True,
           epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=61),
    # several K chunks with a ragged last one: Cin 72 (3 chunks), K = 1,944 (the GN workload's 1,728)
    E.Spec("cin72", N=1, Cin=72, Cout=64, D=2, H=3, W=4, k=3, bias=True, epilogue=E.EPI_RELU_GROUPNORM,
           groups=8, seed_index=62),
]


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
def test_small_cases(spec, precision):
    inputs = E.make_inputs(spec)
    assert_close(run_gpu(spec, inputs, precision), run_oracle(spec, inputs), spec.name)


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
def test_repeat_is_bitwise_deterministic(precision):
    spec = SMALL[1]
    inputs = E.make_inputs(spec)
    a = run_gpu(spec, inputs, precision)
    b = run_gpu(spec, inputs, precision)
    assert np.array_equal(a, b)


FULL = [E.GN, E.BN, E.SOFTMAX, E.IDENTITY]


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("spec", FULL, ids=lambda s: s.name)
def test_full_size_workloads(spec, precision):
    inputs = E.make_inputs(spec)
    got = run_gpu(spec, inputs, precision)
    if spec.epilogue == E.EPI_SCALE_BATCHNORM_AVGPOOL:
        ref = run_oracle(spec, inputs)  # batch statistics: the whole batch
        assert_close(got, ref, spec.name)
        return
    # per-sample epilogues: compare whole samples 0 and N-1
    for n in (0, spec.N - 1):
        sub = E.sample_slice(inputs, n, n + 1)
        ref = run_oracle(spec.replace(N=1), sub)
        assert_close(got[n:n + 1], ref, f"{spec.name}[n={n}]")


@pytest.mark.gpu
@pytest.mark.parametrize("spec", [SMALL[1], SMALL[7], SMALL[5]], ids=lambda s: s.name)
def test_host_pipeline_matches_device_path(spec):
    from transposed_convolution_convt3d_gb300 import HostPipeline
    spec = spec.replace(N=4) if spec.epilogue != E.EPI_SCALE_BATCHNORM_AVGPOOL else spec
    inputs = E.make_inputs(spec)
    ref = run_oracle(spec, inputs)
    host = {k: (v.pin_memory() if v is not None else None) for k, v in inputs.items()}
    pipe = HostPipeline(spec.N, spec.Cin, spec.Cout, spec.D, spec.H, spec.W, spec.k, spec.stride, spec.pad,
                        spec.out_pad, spec.bias, spec.epilogue, spec.groups, spec.eps, spec.scale, chunks=2)
    y_host = torch.full(pipe.full_shape, float("nan")).pin_memory()
    for _ in range(2):
        pipe(host["x"], host["w"], y_host, host["bias"], host["gamma"], host["beta"])
        torch.cuda.synchronize()
        assert_close(y_host.numpy(), ref, spec.name)


EVAL_CASES = [
    E.BN.replace(name="bn_eval_full", epilogue=E.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL),
    E.Spec("bn_eval_s2_p1_op1", N=2, Cin=24, Cout=40, D=5, H=6, W=7, k=3, stride=2, pad=1, out_pad=1, bias=True,
           epilogue=E.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL, scale=0.75, seed_index=30),
    E.Spec("bn_eval_k4_p2", N=3, Cin=33, Cout=20, D=4, H=5, W=9, k=4, pad=2, bias=False,
           epilogue=E.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL, scale=-1.5, seed_index=31),
    E.Spec("bn_eval_k7_s2_small", N=1, Cin=5, Cout=7, D=2, H=3, W=2, k=7, stride=2, pad=3, out_pad=1, bias=True,
           epilogue=E.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL, scale=2.0, seed_index=32),
]


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("spec", EVAL_CASES, ids=lambda s: s.name)
def test_batchnorm_eval_mode(spec, precision):
    """Evaluation-mode BatchNorm+pool (no convolution is run) against the
    oracle's full convolution followed by the normalisation; the statistics are
    fixed, so every sample is independent and the full-size case is checked on
    samples 0 and N-1."""
    inputs = E.make_inputs(spec)
    running = E.make_running_stats(spec)
    got, rm, rv = run_gpu(spec, inputs, precision, running)
    # evaluation mode leaves the running statistics untouched
    assert np.array_equal(rm, running[0].numpy()) and np.array_equal(rv, running[1].numpy())
    samples = range(spec.N) if spec.N <= 3 else (0, spec.N - 1)
    for n in samples:
        ref, _, _ = run_oracle(spec.replace(N=1), E.sample_slice(inputs, n, n + 1), running)
        assert_close(got[n:n + 1], ref, f"{spec.name}[n={n}]")


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("spec", [SMALL[5], SMALL[6], E.BN], ids=lambda s: s.name)
def test_batchnorm_running_stats_update(spec, precision):
    """Training-mode BatchNorm updates the running statistics in place with
    momentum 0.3 and the unbiased batch variance; output and both statistics
    match the oracle."""
    inputs = E.make_inputs(spec)
    running = E.make_running_stats(spec)
    got, rm, rv = run_gpu(spec, inputs, precision, running, momentum=0.3)
    ref, rm_ref, rv_ref = run_oracle(spec, inputs, running, momentum=0.3)
    assert_close(got, ref, spec.name)
    assert_close(rm, rm_ref, spec.name + " running_mean")
    assert_close(rv, rv_ref, spec.name + " running_var")


# General shapes: per-dimension kernel/stride/padding, dilation, grouped convolution.
GENERAL = [
    E.Spec("gen_kdims_strides", N=2, Cin=20, Cout=24, D=4, H=5, W=6, k=(3, 2, 4), stride=(1, 2, 2),
           pad=(1, 0, 2), out_pad=(0, 1, 1), bias=True, seed_index=40),
    E.Spec("gen_dilation", N=2, Cin=16, Cout=32, D=4, H=5, W=5, k=3, pad=(1, 2, 0), dilation=(2, 1, 3),
           bias=True, epilogue=E.EPI_RELU_GROUPNORM, groups=4, seed_index=41),
    E.Spec("gen_groups", N=2, Cin=32, Cout=48, D=3, H=4, W=5, k=3, stride=2, pad=1, out_pad=1, bias=True,
           conv_groups=4, seed_index=42),
    E.Spec("gen_mixed_softmax", N=1, Cin=24, Cout=40, D=3, H=5, W=4, k=(2, 3, 3), stride=(2, 1, 2),
           pad=(0, 1, 1), out_pad=(1, 0, 0), dilation=(1, 2, 3), bias=True, epilogue=E.EPI_SOFTMAX_SIGMOID,
           seed_index=43),
    E.Spec("gen_groups_bn", N=3, Cin=12, Cout=18, D=3, H=4, W=4, k=(3, 3, 2), stride=(1, 2, 1), pad=(1, 0, 0),
           out_pad=(0, 1, 0), bias=True, conv_groups=3, epilogue=E.EPI_SCALE_BATCHNORM_AVGPOOL, scale=1.5,
           seed_index=44),
    E.Spec("gen_dil_s2_d_only", N=1, Cin=32, Cout=16, D=4, H=3, W=5, k=(3, 3, 3), stride=(2, 1, 1),
           pad=(2, 1, 0), out_pad=(1, 0, 0), dilation=(3, 1, 1), seed_index=45),
]


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("spec", GENERAL, ids=lambda s: s.name)
def test_general_shapes(spec, precision):
    inputs = E.make_inputs(spec)
    assert_close(run_gpu(spec, inputs, precision), run_oracle(spec, inputs), spec.name)


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
def test_unaddressable_shape_falls_back_to_ffma(precision):
    """Dilation 5 with k = 7 along d: beyond the TMA im2col corner range, so the
    tensor-core precisions run the FFMA kernel (same 1e-4 bar)."""
    spec = E.Spec("fallback_dil5_k7", N=1, Cin=8, Cout=16, D=2, H=3, W=3, k=(7, 3, 3), dilation=(5, 1, 1),
                  pad=(2, 1, 0), bias=True, epilogue=E.EPI_RELU_GROUPNORM, groups=4, seed_index=47)
    inputs = E.make_inputs(spec)
    assert_close(run_gpu(spec, inputs, precision), run_oracle(spec, inputs), spec.name)


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
def test_general_shapes_eval_batchnorm(precision):
    spec = E.Spec("gen_eval_bn", N=2, Cin=12, Cout=20, D=4, H=5, W=6, k=(3, 2, 4), stride=(2, 1, 2),
                  pad=(1, 0, 2), out_pad=(1, 0, 0), dilation=(1, 2, 1), bias=True, conv_groups=2,
                  epilogue=E.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL, scale=0.5, seed_index=46)
    inputs = E.make_inputs(spec)
    running = E.make_running_stats(spec)
    got, _, _ = run_gpu(spec, inputs, precision, running)
    ref, _, _ = run_oracle(spec, inputs, running)
    assert_close(got, ref, spec.name)


# Single-product TF32 and BF16.  The library rounds x and w to TF32 (nearest,
# ties away from zero: PTX cvt.rna) or bf16 (nearest even) before the tensor
# cores multiply them; products of such values are exact in fp32, so the
# result must match the oracle run on identically rounded x and w (bias and the
# affine parameters stay fp32) within the fp32 tolerance.  The distance to the
# unrounded fp32 result is the inputs' rounding, a property of the precision:
# the single-TF32 path is also held to the 1e-2 tier that page l2_p49 quotes
# for reduced precision; bf16 inputs can exceed it where K is small and the
# output cancels.
TOL_LOW_VS_FP32 = 1e-2
LOW = [pytest.param(PREC_TF32, id="tf32"), pytest.param(PREC_BF16, id="bf16"), pytest.param(PREC_FP16, id="fp16")]


def round_tf32(a):
    """Nearest TF32 value, ties away from zero (10 explicit mantissa bits)."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    return ((u + np.uint32(0x1000)) & np.uint32(0xFFFFE000)).view(np.float32)


def round_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def round_fp16(a):
    """Nearest IEEE half (ties to even), back in fp32."""
    return np.ascontiguousarray(a, np.float32).astype(np.float16).astype(np.float32)


def rounded_inputs(inputs, precision):
    rnd = {PREC_TF32: round_tf32, PREC_BF16: round_bf16, PREC_FP16: round_fp16}[precision]
    out = dict(inputs)
    for k in ("x", "w"):
        out[k] = torch.from_numpy(rnd(inputs[k].numpy()))
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("precision", LOW)
@pytest.mark.parametrize("spec", SMALL + GENERAL, ids=lambda s: s.name)
def test_low_precision_small_and_general(spec, precision):
    inputs = E.make_inputs(spec)
    got = run_gpu(spec, inputs, precision)
    assert_close(got, run_oracle(spec, rounded_inputs(inputs, precision)), spec.name)
    if precision == PREC_TF32:
        assert_close(got, run_oracle(spec, inputs), spec.name + " vs fp32", TOL_LOW_VS_FP32)


@pytest.mark.gpu
@pytest.mark.parametrize("precision", LOW)
def test_low_precision_eval_batchnorm(precision):
    spec = EVAL_CASES[1]
    inputs = E.make_inputs(spec)
    rin = rounded_inputs(inputs, precision)
    running = E.make_running_stats(spec)
    got, _, _ = run_gpu(spec, inputs, precision, running)
    for n in range(spec.N):
        ref, _, _ = run_oracle(spec.replace(N=1), E.sample_slice(rin, n, n + 1), running)
        assert_close(got[n:n + 1], ref, spec.name)


@pytest.mark.gpu
@pytest.mark.parametrize("precision", LOW)
@pytest.mark.parametrize("spec", FULL, ids=lambda s: s.name)
def test_low_precision_full_size_workloads(spec, precision):
    inputs = E.make_inputs(spec)
    rin = rounded_inputs(inputs, precision)
    got = run_gpu(spec, inputs, precision)
    if spec.epilogue == E.EPI_SCALE_BATCHNORM_AVGPOOL:
        assert_close(got, run_oracle(spec, rin), spec.name)
        return
    n = spec.N - 1
    ref = run_oracle(spec.replace(N=1), E.sample_slice(rin, n, n + 1))
    assert_close(got[n:n + 1], ref, f"{spec.name}[n={n}]")


# Channels-last x and y (NDHWC), every epilogue, both precisions and the
# evaluation-mode BatchNorm; ragged channel counts take the scalar store path.
CHANNELS_LAST = [
    SMALL[1].replace(name="cl_gn_ragged", channels_last=True),
    SMALL[2].replace(name="cl_gn_pad1_bias", channels_last=True),
    SMALL[5].replace(name="cl_bn_small", channels_last=True),
    SMALL[7].replace(name="cl_softmax_s2", channels_last=True),
    SMALL[8].replace(name="cl_softmax_s2_odd", channels_last=True),
    E.Spec("cl_identity_s2_k4_c36", N=2, Cin=36, Cout=36, D=3, H=5, W=6, k=4, stride=2, pad=1, bias=True,
           channels_last=True, seed_index=50),
    GENERAL[0].replace(name="cl_gen_kdims_strides", channels_last=True),
    GENERAL[3].replace(name="cl_gen_mixed_softmax", channels_last=True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("spec", CHANNELS_LAST, ids=lambda s: s.name)
def test_channels_last(spec, precision):
    inputs = E.make_inputs(spec)
    assert_close(run_gpu(spec, inputs, precision), run_oracle(spec, inputs), spec.name)


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
def test_channels_last_eval_batchnorm(precision):
    spec = EVAL_CASES[1].replace(name="cl_bn_eval", channels_last=True)
    inputs = E.make_inputs(spec)
    running = E.make_running_stats(spec)
    got, _, _ = run_gpu(spec, inputs, precision, running)
    ref, _, _ = run_oracle(spec, inputs, running)
    assert_close(got, ref, spec.name)


# bf16 tensors at the boundary (x, w, y; bias and affine parameters fp32) with
# the bf16 tensor-core precision.  Reference: the oracle on the same
# bf16-rounded x and w; the output is rounded to bf16 once more (relative
# 2^-9), so the comparison uses the 1e-2 tier page l2_p49 quotes for bf16.
IO_BF16 = [
    SMALL[1].replace(name="io16_gn_ragged", io_bf16=True),
    SMALL[5].replace(name="io16_bn_small", io_bf16=True),
    SMALL[7].replace(name="io16_softmax_s2", io_bf16=True),
    SMALL[9].replace(name="io16_softmax_s2_c96", io_bf16=True),
    SMALL[12].replace(name="io16_identity_s2_k4", io_bf16=True),
    SMALL[1].replace(name="io16_cl_gn_ragged", io_bf16=True, channels_last=True),
    SMALL[7].replace(name="io16_cl_softmax_s2", io_bf16=True, channels_last=True),
    GENERAL[2].replace(name="io16_gen_groups", io_bf16=True),
]


@pytest.mark.gpu
@pytest.mark.parametrize("spec", IO_BF16, ids=lambda s: s.name)
def test_bf16_tensors(spec):
    inputs = E.make_inputs(spec)
    got = run_gpu(spec, inputs, PREC_BF16)
    assert_close(got, run_oracle(spec, rounded_inputs(inputs, PREC_BF16)), spec.name, TOL_LOW_VS_FP32)


# fp16 tensors at the boundary (x, w, y; bias and affine parameters fp32) with
# the fp16 tensor-core precision (kind::f16 with fp16 operands), the other
# format page l2_p49's reduced-precision tier names.  Reference: the oracle on
# the same fp16-rounded x and w; the output is rounded to fp16 once more
# (relative 2^-11), inside the 1e-2 tier.
IO_FP16 = [s.replace(name=s.name.replace("io16", "iofp16"), io_bf16=False, io_fp16=True) for s in IO_BF16]


@pytest.mark.gpu
@pytest.mark.parametrize("spec", IO_FP16, ids=lambda s: s.name)
def test_fp16_tensors(spec):
    inputs = E.make_inputs(spec)
    got = run_gpu(spec, inputs, PREC_FP16)
    assert_close(got, run_oracle(spec, rounded_inputs(inputs, PREC_FP16)), spec.name, TOL_LOW_VS_FP32)


@pytest.mark.gpu
def test_fp16_tensors_eval_batchnorm():
    spec = EVAL_CASES[1].replace(name="iofp16_bn_eval", io_fp16=True)
    inputs = E.make_inputs(spec)
    running = E.make_running_stats(spec)
    got, _, _ = run_gpu(spec, inputs, PREC_FP16, running)
    ref, _, _ = run_oracle(spec, rounded_inputs(inputs, PREC_FP16), running)
    assert_close(got, ref, spec.name, TOL_LOW_VS_FP32)


@pytest.mark.gpu
def test_bf16_tensors_eval_batchnorm():
    spec = EVAL_CASES[1].replace(name="io16_bn_eval", io_bf16=True)
    inputs = E.make_inputs(spec)
    running = E.make_running_stats(spec)
    got, _, _ = run_gpu(spec, inputs, PREC_BF16, running)
    ref, _, _ = run_oracle(spec, rounded_inputs(inputs, PREC_BF16), running)
    assert_close(got, ref, spec.name, TOL_LOW_VS_FP32)


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("cin", [264, 520, 1024])
def test_long_reduction(cin, precision):
    """K = Cin * 27 = 7,128, 14,040 and 27,648 products per output element with an
    elementwise epilogue, held to the 1e-4 bar.  The tensor cores round the fp32
    accumulator once per MMA and that error grows with the length of the chain, so
    the tensor-core kernels accumulate such a tile's K walk in segments of at most
    64 K steps and add the segments' partial sums in fp32."""
    spec = E.Spec(f"cin{cin}", N=1, Cin=cin, Cout=64, D=2, H=3, W=4, k=3, bias=True,
                  epilogue=E.EPI_RELU_GROUPNORM, groups=8, seed_index=63)
    inputs = E.make_inputs(spec)
    assert_close(run_gpu(spec, inputs, precision), run_oracle(spec, inputs), spec.name)


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
def test_long_reduction_pairs(precision):
    """The same for w-parity pairs (stride 2 along w, Cout 96: two accumulators per
    tile, single-buffered beside the running sum) with 12 channels per GroupNorm
    group (the statistics' second pass over tensor memory): K = 512 * 8 per class."""
    spec = E.Spec("cin512_s2_pairs", N=1, Cin=512, Cout=96, D=2, H=3, W=4, k=4, stride=2, pad=1, bias=True,
                  epilogue=E.EPI_RELU_GROUPNORM, groups=8, seed_index=64)
    inputs = E.make_inputs(spec)
    assert_close(run_gpu(spec, inputs, precision), run_oracle(spec, inputs), spec.name)


# Wide channel counts (up to the 512 output channels of one tensor-memory
# accumulator): above 256 the tensor-core tile walks its K steps once per N slice
# of at most 256 columns and keeps a single accumulator; above 128 at stride 2
# along w the two w-parity classes take separate tiles.  The softmax's row
# reduction runs over every channel of the row in one tile.
WIDE = [
    E.Spec("wide_identity_s1_c384", N=1, Cin=24, Cout=384, D=3, H=4, W=5, k=3, bias=True, seed_index=90),
    E.Spec("wide_identity_s2_c512", N=1, Cin=16, Cout=512, D=2, H=3, W=4, k=3, stride=2, pad=1, out_pad=1,
           bias=True, seed_index=91),
    E.Spec("wide_gn_s1_c512", N=2, Cin=16, Cout=512, D=2, H=3, W=4, k=3, bias=True, epilogue=E.EPI_RELU_GROUPNORM,
           groups=8, seed_index=92),
    E.Spec("wide_gn_s2_c384_cpg12", N=1, Cin=20, Cout=384, D=2, H=3, W=3, k=3, stride=2, pad=1, out_pad=1,
           bias=True, epilogue=E.EPI_RELU_GROUPNORM, groups=32, seed_index=93),
    E.Spec("wide_bn_s1_c384", N=2, Cin=12, Cout=384, D=2, H=3, W=4, k=3, bias=True,
           epilogue=E.EPI_SCALE_BATCHNORM_AVGPOOL, scale=2.0, seed_index=94),
    E.Spec("wide_bn_s2_c512", N=2, Cin=8, Cout=512, D=2, H=3, W=3, k=4, stride=2, pad=1, bias=True,
           epilogue=E.EPI_SCALE_BATCHNORM_AVGPOOL, scale=0.5, seed_index=95),
    E.Spec("wide_softmax_s1_c512", N=1, Cin=16, Cout=512, D=2, H=3, W=5, k=3, bias=True,
           epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=96),
    E.Spec("wide_softmax_s2_c384", N=1, Cin=24, Cout=384, D=2, H=3, W=4, k=3, stride=2, pad=1, out_pad=1,
           bias=True, epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=97),
    E.Spec("wide_softmax_s2_c256", N=1, Cin=32, Cout=256, D=2, H=3, W=4, k=3, stride=2, pad=1, out_pad=1,
           bias=True, epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=98),
    # 300 channels: two slices of 160 (Cout_pad rounded to 320), ragged last chunk
    E.Spec("wide_softmax_s1_c300", N=1, Cin=8, Cout=300, D=2, H=2, W=3, k=2, bias=True,
           epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=99),
]


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("spec", WIDE, ids=lambda s: s.name)
def test_wide_channels(spec, precision):
    inputs = E.make_inputs(spec)
    assert_close(run_gpu(spec, inputs, precision), run_oracle(spec, inputs), spec.name)


# Statistics under a large common offset: bias + 100 puts the group / channel
# means some 250 standard deviations from zero, where a one-pass
# E[v^2] - mean^2 over fp32 sums would lose most of the variance's digits.  The
# epilogues sum deviations from each warp's own mean and the finalize kernels
# combine (count, sum, M2) rows, so the 1e-4 bar holds.
OFFSET_CASES = [
    E.Spec("gn_offset", N=2, Cin=16, Cout=32, D=4, H=5, W=6, k=3, bias=True, epilogue=E.EPI_RELU_GROUPNORM,
           groups=2, seed_index=80),
    # 12 channels per group: the group statistics take the second pass over tensor memory
    E.Spec("gn_offset_cpg12", N=2, Cin=16, Cout=48, D=3, H=4, W=5, k=3, bias=True, epilogue=E.EPI_RELU_GROUPNORM,
           groups=4, seed_index=81),
    E.Spec("gn_offset_s2", N=2, Cin=16, Cout=32, D=3, H=4, W=4, k=4, stride=2, pad=1, bias=True,
           epilogue=E.EPI_RELU_GROUPNORM, groups=2, seed_index=82),
    E.Spec("bn_offset", N=3, Cin=20, Cout=32, D=4, H=6, W=5, k=5, bias=True,
           epilogue=E.EPI_SCALE_BATCHNORM_AVGPOOL, scale=2.0, seed_index=83),
    E.Spec("bn_offset_s2", N=2, Cin=8, Cout=16, D=3, H=4, W=5, k=3, stride=2, pad=1, out_pad=1, bias=True,
           epilogue=E.EPI_SCALE_BATCHNORM_AVGPOOL, scale=0.5, seed_index=84),
]


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("spec", OFFSET_CASES, ids=lambda s: s.name)
def test_statistics_large_offset(spec, precision):
    inputs = E.make_inputs(spec)
    inputs["bias"] = inputs["bias"] + 100.0
    assert_close(run_gpu(spec, inputs, precision), run_oracle(spec, inputs), spec.name)


@pytest.mark.gpu
@pytest.mark.parametrize("layout", ["cl", "io16", "cl_io16", "iofp16"])
def test_host_pipeline_layouts(layout):
    """HostPipeline from pinned host tensors with channels-last and/or 16-bit x/w/y."""
    from transposed_convolution_convt3d_gb300 import HostPipeline
    cl, io16, fp16 = "cl" in layout, "io16" in layout, "fp16" in layout
    spec = SMALL[7].replace(N=4, channels_last=cl, io_bf16=io16, io_fp16=fp16)
    prec = PREC_BF16 if io16 else (PREC_FP16 if fp16 else PREC_3XTF32)
    dt = torch.bfloat16 if io16 else torch.float16
    inputs = E.make_inputs(spec)
    ref = run_oracle(spec, rounded_inputs(inputs, prec) if (io16 or fp16) else inputs)
    host = {k: (v.pin_memory() if v is not None else None) for k, v in inputs.items()}
    if cl:
        host["x"] = host["x"].permute(0, 2, 3, 4, 1).contiguous().pin_memory()
    if io16 or fp16:
        host["x"], host["w"] = host["x"].to(dt).pin_memory(), host["w"].to(dt).pin_memory()
    io16 = io16 or fp16
    pipe = HostPipeline(spec.N, spec.Cin, spec.Cout, spec.D, spec.H, spec.W, spec.k, spec.stride, spec.pad,
                        spec.out_pad, spec.bias, spec.epilogue, spec.groups, spec.eps, spec.scale, prec, chunks=2,
                        channels_last=cl, io_bf16=io16 and not fp16, io_fp16=fp16)
    y_host = torch.full(pipe.full_shape, float("nan"), dtype=pipe.plan.io_dtype).pin_memory()
    pipe(host["x"], host["w"], y_host, host["bias"], host["gamma"], host["beta"])
    torch.cuda.synchronize()
    got = y_host.float()
    if cl:
        got = got.permute(0, 4, 1, 2, 3)
    assert_close(got.contiguous().numpy(), ref, spec.name, TOL_LOW_VS_FP32 if io16 else TOL)
