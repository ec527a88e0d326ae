"""GPU checks of the forward split into sample ranges (convt3d_forward_samples +
convt3d_forward_finish) and of HostPipeline's chunked BatchNorm.

The split forward runs the same kernels on the same tiles as one convt3d_forward
(a tile belongs to one sample; its statistics land in the same per-tile slot
whichever launch wrote it; the whole-batch passes run once at the end), so its
y and running statistics must equal the one-call forward's bit for bit; they are
also held to the oracle at the 1e-4 tier.  Plans whose main kernel reads x
directly accept only the whole batch, and evaluation-mode BatchNorm only the
one-call forward.
"""
import numpy as np
import pytest
import torch

import workloads as E
from test_parity_gpu import PRECISIONS, assert_close, run_oracle
from transposed_convolution_convt3d_gb300 import (PREC_3XBF16, PREC_BF16, PREC_FP16, Convt3dError, HostPipeline,
                                                  Plan)

CASES = [
    E.Spec("rng_bn_k5", N=3, Cin=20, Cout=32, D=4, H=6, W=5, k=5, bias=True,
           epilogue=E.EPI_SCALE_BATCHNORM_AVGPOOL, scale=0.5, seed_index=100),
    E.Spec("rng_bn_s2", N=4, Cin=8, Cout=16, D=3, H=4, W=5, k=3, stride=2, pad=1, out_pad=1, bias=True,
           epilogue=E.EPI_SCALE_BATCHNORM_AVGPOOL, scale=2.0, seed_index=101),
    E.Spec("rng_gn", N=4, Cin=40, Cout=48, D=3, H=5, W=6, k=3, epilogue=E.EPI_RELU_GROUPNORM, groups=4,
           seed_index=102),
    E.Spec("rng_softmax_s2", N=3, Cin=12, Cout=64, D=3, H=4, W=7, k=3, stride=2, pad=1, out_pad=1, bias=True,
           epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=103),
    E.Spec("rng_identity_groups", N=3, Cin=32, Cout=48, D=3, H=4, W=5, k=3, stride=2, pad=1, out_pad=1,
           bias=True, conv_groups=2, seed_index=104),
    E.Spec("rng_bn_channels_last", N=3, Cin=16, Cout=24, D=3, H=4, W=4, k=3, bias=True, channels_last=True,
           epilogue=E.EPI_SCALE_BATCHNORM_AVGPOOL, scale=1.5, seed_index=105),
]


def device_inputs(spec, inputs, dev):
    d = {k: (v.to(dev) if v is not None else None) for k, v in inputs.items()}
    if spec.channels_last:
        d["x"] = d["x"].permute(0, 2, 3, 4, 1).contiguous()
    for flag, dt in ((spec.io_bf16, torch.bfloat16), (spec.io_fp16, torch.float16)):
        if flag:  # x and w handed over as 16-bit tensors
            d["x"], d["w"] = d["x"].to(dt), d["w"].to(dt)
    return d


def run_both(spec, precision, ranges):
    """(y of one forward, y of the ranges + finish, running stats of each) on the GPU."""
    dev = torch.device("cuda")
    inputs = E.make_inputs(spec)
    d = device_inputs(spec, inputs, dev)
    plan = Plan.from_spec(spec, precision=precision)
    ws = plan.new_workspace(dev)
    bn = spec.epilogue == E.EPI_SCALE_BATCHNORM_AVGPOOL
    outs = []
    for split in (False, True):
        y = plan.new_output(dev).fill_(float("nan"))
        if bn:
            rm, rv = (t.to(dev).clone() for t in E.make_running_stats(spec))
            plan.set_running_stats(rm, rv)
        plan.pack_weights(d["w"], ws)
        if split:
            for n0, n1 in ranges:
                plan.forward_samples(d["x"], y, ws, n0, n1, d["bias"])
            plan.forward_finish(y, ws, d["bias"], d["gamma"], d["beta"])
        else:
            plan.forward(d["x"], y, ws, d["bias"], d["gamma"], d["beta"])
        plan.check(ws)
        if spec.channels_last and y.dim() == 5 and tuple(y.shape) != plan.out_shape:
            y = y.permute(0, 4, 1, 2, 3)
        stats = (rm.cpu().numpy(), rv.cpu().numpy()) if bn else None
        outs.append((y.float().contiguous().cpu().numpy(), stats))
    return inputs, outs


def split_of(n):
    """Ranges of unequal length covering 0..n-1, in a shuffled order."""
    if n == 1:
        return [(0, 1)]
    cuts = [(0, 1), (1, n)] if n < 4 else [(1, 3), (0, 1), (3, n)]
    return cuts


@pytest.mark.gpu
@pytest.mark.parametrize("precision", PRECISIONS)
@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_sample_ranges_equal_one_forward(spec, precision):
    inputs, ((y1, st1), (y2, st2)) = run_both(spec, precision, split_of(spec.N))
    assert np.array_equal(y1, y2, equal_nan=False), spec.name
    if st1 is not None:
        assert np.array_equal(st1[0], st2[0]) and np.array_equal(st1[1], st2[1])
        ref, rm, rv = run_oracle(spec, inputs, E.make_running_stats(spec))
        assert_close(y2, ref, spec.name)
        assert_close(st2[0], rm, spec.name + " running_mean")
        assert_close(st2[1], rv, spec.name + " running_var")
    else:
        assert_close(y2, run_oracle(spec, inputs), spec.name)


@pytest.mark.gpu
def test_full_size_batchnorm_in_four_ranges():
    """The BatchNorm workload at full size, its batch in four ranges: bitwise the one-call forward."""
    spec = E.BN
    q = spec.N // 4
    ranges = [(2 * q, 3 * q), (0, q), (3 * q, spec.N), (q, 2 * q)]
    _, ((y1, st1), (y2, st2)) = run_both(spec, PREC_3XBF16, ranges)
    assert np.array_equal(y1, y2)
    assert np.array_equal(st1[0], st2[0]) and np.array_equal(st1[1], st2[1])


@pytest.mark.gpu
def test_direct_input_plan_takes_only_the_whole_batch():
    import test_direct_gpu as T
    spec = T.DIRECT[0]
    assert Plan.from_spec(spec, precision=PREC_3XBF16).info["main_kernel"] == 2
    inputs, ((y1, _), (y2, _)) = run_both(spec, PREC_3XBF16, [(0, spec.N)])
    assert np.array_equal(y1, y2)
    dev = torch.device("cuda")
    plan = Plan.from_spec(spec, precision=PREC_3XBF16)
    ws = plan.new_workspace(dev)
    d = device_inputs(spec, inputs, dev)
    plan.pack_weights(d["w"], ws)
    y = plan.new_output(dev)
    with pytest.raises(Convt3dError) as ei:
        plan.forward_samples(d["x"], y, ws, 0, 1, d["bias"])
    assert ei.value.status == 2


@pytest.mark.gpu
@pytest.mark.parametrize("chunks", [2, 3, 6])
@pytest.mark.parametrize("epilogue", [E.EPI_SCALE_BATCHNORM_AVGPOOL, E.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL],
                         ids=["bn_train", "bn_eval"])
def test_host_pipeline_batchnorm_chunks(epilogue, chunks):
    """HostPipeline overlaps BatchNorm's input copy with the computation: training mode
    through one whole-batch plan in sample ranges, evaluation mode (per-sample) through
    chunk-sized plans.  y and the running statistics against the oracle, twice in a row."""
    spec = E.Spec("pipe_bn", N=6, Cin=16, Cout=24, D=3, H=5, W=4, k=3, stride=2, pad=1, out_pad=1, bias=True,
                  epilogue=epilogue, scale=0.75, seed_index=106)
    inputs = E.make_inputs(spec)
    host = {k: (v.pin_memory() if v is not None else None) for k, v in inputs.items()}
    dev = torch.device("cuda")
    pipe = HostPipeline(spec.N, spec.Cin, spec.Cout, spec.D, spec.H, spec.W, spec.k, spec.stride, spec.pad,
                        spec.out_pad, spec.bias, spec.epilogue, spec.groups, spec.eps, spec.scale, chunks=chunks)
    assert pipe.chunks == chunks
    rm0, rv0 = E.make_running_stats(spec)
    rm, rv = rm0.to(dev).clone(), rv0.to(dev).clone()
    pipe.set_running_stats(rm, rv)
    y_host = torch.full(pipe.full_shape, float("nan")).pin_memory()
    ref_rm, ref_rv = rm0.numpy().copy(), rv0.numpy().copy()
    for _ in range(2):
        pipe(host["x"], host["w"], y_host, host["bias"], host["gamma"], host["beta"])
        torch.cuda.synchronize()
        ref, ref_rm, ref_rv = run_oracle(spec, inputs, (torch.from_numpy(ref_rm), torch.from_numpy(ref_rv)))
        assert_close(y_host.numpy(), ref, spec.name)
        assert_close(rm.cpu().numpy(), ref_rm, spec.name + " running_mean")
        assert_close(rv.cpu().numpy(), ref_rv, spec.name + " running_var")


@pytest.mark.gpu
def test_host_pipeline_batchnorm_uneven_ranges():
    """Training-mode BatchNorm through HostPipeline with a batch the chunk count does not
    divide (5 samples in ranges of 2 and 3): y and the running statistics against the oracle."""
    spec = E.Spec("pipe_bn_uneven", N=5, Cin=12, Cout=16, D=3, H=4, W=5, k=3, bias=True,
                  epilogue=E.EPI_SCALE_BATCHNORM_AVGPOOL, scale=1.25, seed_index=107)
    inputs = E.make_inputs(spec)
    host = {k: (v.pin_memory() if v is not None else None) for k, v in inputs.items()}
    dev = torch.device("cuda")
    pipe = HostPipeline(spec.N, spec.Cin, spec.Cout, spec.D, spec.H, spec.W, spec.k, spec.stride, spec.pad,
                        spec.out_pad, spec.bias, spec.epilogue, spec.groups, spec.eps, spec.scale, chunks=2)
    assert pipe.chunks == 2
    rm0, rv0 = E.make_running_stats(spec)
    rm, rv = rm0.to(dev).clone(), rv0.to(dev).clone()
    pipe.set_running_stats(rm, rv)
    y_host = torch.full(pipe.full_shape, float("nan")).pin_memory()
    pipe(host["x"], host["w"], y_host, host["bias"], host["gamma"], host["beta"])
    torch.cuda.synchronize()
    ref, ref_rm, ref_rv = run_oracle(spec, inputs, (rm0, rv0))
    assert_close(y_host.numpy(), ref, spec.name)
    assert_close(rm.cpu().numpy(), ref_rm, spec.name + " running_mean")
    assert_close(rv.cpu().numpy(), ref_rv, spec.name + " running_var")


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["bf16", "fp16"])
@pytest.mark.parametrize("spec", [CASES[0], CASES[2], CASES[4]], ids=lambda s: s.name)
def test_sample_ranges_16bit_tensors(spec, kind):
    """Ranges over 16-bit x and y (staging offsets in 2-byte elements): bitwise the one-call
    forward, BatchNorm's running statistics included."""
    s = spec.replace(name=spec.name + "_io" + kind, io_bf16=kind == "bf16", io_fp16=kind == "fp16")
    prec = PREC_BF16 if kind == "bf16" else PREC_FP16
    assert Plan.from_spec(s, precision=prec).info["main_kernel"] == 0
    _, ((y1, st1), (y2, st2)) = run_both(s, prec, split_of(s.N))
    assert np.all(np.isfinite(y1))
    assert np.array_equal(y1, y2)
    if st1 is not None:
        assert np.array_equal(st1[0], st2[0]) and np.array_equal(st1[1], st2[1])
