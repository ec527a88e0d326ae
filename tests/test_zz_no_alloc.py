"""The forward that allocates nothing (convt3d_forward_static_workspace).

For callers that may not allocate device memory -- a plugin whose host owns
every device allocation, or a latency-critical caller that cannot afford
cudaMalloc's implicit synchronisation -- the library carries a built-in 32 MiB
device workspace.  These tests call that entry point through the C ABI twice in
a row and compare each result with the regular caller-workspace path; the
tolerance is the one every parity test uses.  This file is collected last so a
failure here leaves the rest of the suite already run.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as E
from transposed_convolution_convt3d_gb300 import PREC_3XBF16, PREC_3XTF32, PREC_FFMA, Plan, _lib

TOL = 1e-4

CASES = [
    E.TINY,
    E.Spec("static_ws_softmax_s2", N=2, Cin=12, Cout=64, D=5, H=6, W=7, k=3, stride=2, pad=1, out_pad=1,
           bias=True, epilogue=E.EPI_SOFTMAX_SIGMOID, seed_index=40),
    E.Spec("static_ws_bn", N=3, Cin=20, Cout=32, D=4, H=6, W=5, k=5, bias=True,
           epilogue=E.EPI_SCALE_BATCHNORM_AVGPOOL, scale=2.0, seed_index=41),
]


def _regular(plan, d):
    ws = plan.new_workspace(d["x"].device)
    y = plan.new_output(d["x"].device)
    plan.pack_weights(d["w"], ws)
    plan.forward(d["x"], y, ws, d["bias"], d["gamma"], d["beta"])
    plan.check(ws)
    return y.cpu().numpy()


def _static_ws_call(plan, d, y):
    lib = _lib.load()
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.convt3d_forward_static_workspace(plan.handle, p(d["w"]), p(d["x"]), p(d["bias"]), p(d["gamma"]),
                                              p(d["beta"]), p(y), stream)
    assert st == 0, lib.convt3d_last_error().decode()
    # the call's device-side status lives in the built-in workspace: a NULL
    # workspace makes convt3d_check read (and clear) that one
    st = lib.convt3d_check(plan.handle, None, stream)
    assert st == 0, lib.convt3d_last_error().decode()
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("precision", [PREC_3XTF32, PREC_3XBF16, PREC_FFMA], ids=["3xtf32", "3xbf16", "ffma"])
@pytest.mark.parametrize("spec", CASES, ids=lambda s: s.name)
def test_static_workspace_matches_regular_path_twice(spec, precision):
    dev = torch.device("cuda")
    inputs = E.make_inputs(spec)
    d = {k: (v.to(dev) if v is not None else None) for k, v in inputs.items()}
    plan = Plan.from_spec(spec, precision=precision)
    ref = _regular(plan, d)
    for _ in range(2):
        y = torch.full(plan.out_shape, float("nan"), device=dev)
        got = _static_ws_call(plan, d, y)
        assert np.all(np.isfinite(got))
        err = np.abs(got.astype(np.float64) - ref) / (1.0 + np.abs(ref.astype(np.float64)))
        assert err.max() <= TOL, err.max()


@pytest.mark.gpu
def test_static_workspace_rejects_oversized_problem():
    lib = _lib.load()
    plan = Plan.from_spec(E.GN)  # needs ~270 MB of workspace, more than the built-in 32 MiB
    assert plan.workspace_bytes > 32 << 20
    dummy = ctypes.c_void_p(256)
    st = lib.convt3d_forward_static_workspace(plan.handle, dummy, dummy, None, dummy, dummy, dummy, None)
    assert st == 3  # CONVT3D_ERR_WORKSPACE, nothing launched
    assert b"built-in workspace" in lib.convt3d_last_error()
