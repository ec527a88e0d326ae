"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, and validates descriptions on the host (no GPU needed)."""
import ctypes
import os
import re

import pytest

import oracle
import workloads
from transposed_convolution_convt3d_gb300 import _lib
from transposed_convolution_convt3d_gb300 import build as libbuild
from transposed_convolution_convt3d_gb300.api import Plan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return _lib.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "convt3d.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(convt3d_[a-z_]+)\s*\(", text)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in _lib.STATUS:
        assert lib.convt3d_status_string(code)
    assert lib.convt3d_version() >= 100


def make_desc(**kw):
    base = dict(N=2, Cin=8, Cout=16, Din=8, Hin=8, Win=8, k=3, stride=1, pad=0, out_pad=0, has_bias=0,
                epilogue=0, groups=1, eps=1e-5, scale=1.0, precision=0, per_dim=0, kdims=(0, 0, 0),
                strides=(0, 0, 0), pads=(0, 0, 0), out_pads=(0, 0, 0), dilation=(0, 0, 0), conv_groups=0,
                channels_last=0, io_bf16=0, io_fp16=0)
    base.update(kw)
    return _lib.Desc(*[base[f] for f, _ in _lib.Desc._fields_])


def create(lib, **kw):
    d = make_desc(**kw)
    h = ctypes.c_void_p()
    st = lib.convt3d_plan_create(ctypes.byref(d), ctypes.byref(h))
    return st, h


@pytest.mark.parametrize("kw,status", [
    (dict(N=0), 1), (dict(Cin=0), 1), (dict(k=0), 1), (dict(stride=0), 1), (dict(pad=-1), 1),
    (dict(out_pad=1, stride=1), 1), (dict(epilogue=9), 1), (dict(precision=-1), 1),
    (dict(epilogue=1, groups=3), 1), (dict(epilogue=1, groups=4, eps=0.0), 1),
    (dict(Din=1, Hin=1, Win=1, k=1, pad=1), 1),
    (dict(stride=3, k=3), 2), (dict(k=8), 2), (dict(Cout=513), 2), (dict(k=3, pad=3, Din=9, Hin=9, Win=9), 2),
    (dict(stride=2, k=1), 2),
    (dict(epilogue=4, eps=-1.0), 1), (dict(epilogue=4, scale=float("inf")), 1),
    (dict(epilogue=4, Hin=256, Win=256), 2),
    # general shapes
    (dict(dilation=(-1, 1, 1)), 1), (dict(conv_groups=-2), 1), (dict(conv_groups=3), 1),
    (dict(per_dim=1, kdims=(3, 0, 3), strides=(1, 1, 1)), 1),
    (dict(per_dim=1, kdims=(3, 3, 3), strides=(1, 2, 1), out_pads=(0, 2, 0)), 1),
    (dict(per_dim=1, kdims=(3, 3, 3), strides=(1, 1, 3)), 2), (dict(per_dim=1, kdims=(3, 8, 3), strides=(1, 1, 1)), 2),
    (dict(stride=2, dilation=(2, 2, 2)), 2), (dict(dilation=(16, 1, 1)), 2),
    (dict(io_bf16=1), 2), (dict(io_bf16=1, precision=2), 2), (dict(io_bf16=1, precision=1), 2),
    (dict(io_bf16=1, precision=4), 2),
    (dict(precision=6), 1), (dict(io_fp16=1), 2), (dict(io_fp16=1, precision=3), 2),
    (dict(io_bf16=1, io_fp16=1, precision=3), 1),
])
def test_plan_validation(lib, kw, status):
    st, h = create(lib, **kw)
    assert st == status, lib.convt3d_last_error()
    assert not h.value
    assert lib.convt3d_last_error()


def test_eval_batchnorm_box_planes_follow_distinct_d_intervals(lib):
    """Evaluation-mode BN keeps one H x W plane of box sums per distinct d-interval
    of the taps (shared memory, at most 200 KB per block): unpadded, all three
    taps of k = 3 cover the whole input along d and share one plane (accepted at
    200 x 200); with padding 1 the first tap's interval starts one plane later and
    the last tap's ends one plane earlier, three planes are needed and the same
    extent is rejected as unsupported."""
    st, h = create(lib, epilogue=4, k=3, pad=0, Din=4, Hin=200, Win=200)
    assert st == 0, lib.convt3d_last_error()
    lib.convt3d_plan_destroy(h)
    st, h = create(lib, epilogue=4, k=3, pad=1, Din=4, Hin=200, Win=200)
    assert st == 2 and not h.value


def test_check_null_workspace_reads_the_builtin_one(lib):
    """convt3d_check with a NULL workspace reads the status word of the built-in
    workspace of convt3d_forward_static_workspace on the current device; without a
    GPU the device lookup fails and the call reports a CUDA error (it does not
    treat NULL as an invalid argument any more, and it does not crash)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("checks the no-device path")
    st, h = create(lib)
    assert st == 0
    assert lib.convt3d_check(h, None, None) == 4
    assert lib.convt3d_last_error()
    assert lib.convt3d_check(None, None, None) == 1
    lib.convt3d_plan_destroy(h)


def test_tensor_core_unaddressable_shape_runs_on_ffma(lib):
    """A dilation of 5 with k = 7 puts the TMA im2col corners at -30 (beyond [-16, 15]):
    the plan keeps the requested tensor-core precision but runs the FFMA kernel; with
    16-bit tensors (which the FFMA kernel does not take) the shape is unsupported."""
    from transposed_convolution_convt3d_gb300 import Plan
    pl = Plan(1, 8, 16, 2, 3, 3, (7, 3, 3), dilation=(5, 1, 1), precision=0)
    assert pl.info["main_kernel"] == 1
    assert Plan(1, 8, 16, 2, 3, 3, 3).info["main_kernel"] == 0
    st, h = create(lib, per_dim=1, kdims=(7, 3, 3), strides=(1, 1, 1), dilation=(5, 1, 1), precision=3, io_bf16=1)
    assert st == 2 and not h.value


def test_direct_input_kernel_selection():
    """The softmax workload's shape (stride 2, Cin 32, Cout 64, 32-wide q-rows) runs the
    kernel that reads NCDHW x itself when the operands are bf16 (split or single), and
    then needs no staged copy of x in the workspace; split TF32 keeps the staged kernel,
    and so do shapes outside the direct kernel's range (Cin > 32, q-rows of 12)."""
    import workloads as E
    from transposed_convolution_convt3d_gb300 import PREC_3XBF16, PREC_3XTF32, PREC_BF16, PREC_FP16, Plan
    spec = E.SOFTMAX
    direct = Plan.from_spec(spec, precision=PREC_3XBF16)
    staged = Plan.from_spec(spec, precision=PREC_3XTF32)
    assert direct.info["main_kernel"] == 2 and Plan.from_spec(spec, precision=PREC_BF16).info["main_kernel"] == 2
    assert Plan.from_spec(spec, precision=PREC_FP16).info["main_kernel"] == 2
    assert staged.info["main_kernel"] == 0
    # the staged kernel's workspace holds two bf16 planes of x (channels padded to 64); the direct one's does not
    staged_cl = Plan.from_spec(spec.replace(channels_last=True), precision=PREC_3XBF16)
    assert staged_cl.info["main_kernel"] == 0
    x_planes = 2 * 2 * spec.N * 64 * spec.D * spec.H * spec.W
    assert staged_cl.workspace_bytes - direct.workspace_bytes >= x_planes
    assert direct.info["launches_per_forward"] == 1
    assert Plan.from_spec(spec.replace(Cin=40), precision=PREC_3XBF16).info["main_kernel"] == 0
    assert Plan.from_spec(spec.replace(W=12), precision=PREC_3XBF16).info["main_kernel"] == 0


@pytest.mark.parametrize("precision", [0, 1, 4])
@pytest.mark.parametrize("kw", [dict(stride=2, k=3, pad=1, Cout=144), dict(Cout=384), dict(Cout=512, epilogue=3),
                                dict(stride=2, k=4, pad=1, Cout=512, epilogue=2)])
def test_wide_channels_accepted(lib, kw, precision):
    """Up to 512 output channels on every path (the tensor-core tile splits N above
    256 and gives each stride-2 w-parity class its own tile above 128)."""
    st, h = create(lib, precision=precision, **kw)
    assert st == 0, lib.convt3d_last_error()
    lib.convt3d_plan_destroy(h)


@pytest.mark.parametrize("kw", [
    dict(per_dim=1, kdims=(3, 2, 4), strides=(1, 2, 2), pads=(1, 0, 2), out_pads=(0, 1, 1)),
    dict(dilation=(2, 1, 3), pad=1),
    dict(conv_groups=4, Cin=8, Cout=16),
    dict(per_dim=1, kdims=(2, 3, 3), strides=(2, 1, 2), pads=(0, 1, 1), out_pads=(1, 0, 0), dilation=(1, 2, 3)),
])
@pytest.mark.parametrize("precision", [0, 1])
def test_general_shapes_plan_facts(lib, kw, precision):
    st, h = create(lib, precision=precision, **kw)
    assert st == 0, lib.convt3d_last_error()
    try:
        d = make_desc(precision=precision, **kw)
        kk = tuple(d.kdims) if d.per_dim else (d.k,) * 3
        ss = tuple(d.strides) if d.per_dim else (d.stride,) * 3
        pp = tuple(d.pads) if d.per_dim else (d.pad,) * 3
        oo = tuple(d.out_pads) if d.per_dim else (d.out_pad,) * 3
        dd = tuple(v or 1 for v in d.dilation)
        G = d.conv_groups or 1
        outs = [oracle.output_size_dil(n, kk[a], ss[a], pp[a], oo[a], dd[a])
                for a, n in enumerate((d.Din, d.Hin, d.Win))]
        shp = (ctypes.c_int64 * 5)()
        assert lib.convt3d_output_shape(h, shp) == 0
        assert tuple(shp) == (d.N, d.Cout, *outs)
        inf = _lib.Info()
        assert lib.convt3d_plan_info(h, ctypes.byref(inf)) == 0
        assert inf.num_classes == ss[0] * ss[1] * ss[2]
        assert inf.gemm_k_total == d.Cin * kk[0] * kk[1] * kk[2]  # every tap once over the classes
        assert inf.useful_flop == 2.0 * d.N * d.Cout * (d.Cin // G) * kk[0] * kk[1] * kk[2] * d.Din * d.Hin * d.Win
    finally:
        lib.convt3d_plan_destroy(h)


@pytest.mark.parametrize("spec", workloads.ALL, ids=lambda s: s.name)
@pytest.mark.parametrize("precision", [0, 1, 4])
def test_plan_facts_for_workloads(lib, spec, precision):
    p = Plan.from_spec(spec, precision=precision)
    dims = [oracle.output_size(v, spec.k, spec.stride, spec.pad, spec.out_pad) for v in (spec.D, spec.H, spec.W)]
    if spec.epilogue in (workloads.EPI_SCALE_BATCHNORM_AVGPOOL, workloads.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL):
        assert p.out_shape == (spec.N, spec.Cout, 1, 1, 1)
    else:
        assert p.out_shape == (spec.N, spec.Cout, *dims)
    assert p.workspace_bytes > 0
    assert p.info["useful_flop"] == spec.useful_flop()
    assert p.info["gemm_m"] == spec.N * dims[0] * dims[1] * dims[2]
    assert p.info["num_classes"] == spec.stride ** 3
    # K summed over parity classes covers every tap exactly once
    assert p.info["gemm_k_total"] == spec.Cin * spec.k ** 3
    if spec.epilogue == workloads.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL:
        # no convolution: box sums of x, then one Cin*k^3 contraction per (n, c)
        assert p.info["issued_mma_flop"] == 2.0 * spec.N * spec.Cout * spec.Cin * spec.k ** 3
        assert p.info["launches_per_forward"] == 2
    else:
        assert p.info["issued_mma_flop"] >= p.info["useful_flop"] * (3 if precision in (0, 4) else 1) * 0.9


@pytest.mark.parametrize("spec", workloads.ALL, ids=lambda s: s.name)
def test_split_bf16_planes_are_half_the_split_tf32_planes(lib, spec):
    """Split BF16 keeps two 2-byte planes where split TF32 keeps two 4-byte
    planes: the same products are issued and the staged operands need half the
    workspace and half the GEMM's minimum traffic for them."""
    t, b = Plan.from_spec(spec, precision=0), Plan.from_spec(spec, precision=4)
    # a bf16 K step is 64 channels (128-byte rows): below 64 input channels the
    # padding doubles the elements and the bytes come out equal
    strict = spec.Cin % 64 == 0
    assert b.workspace_bytes < t.workspace_bytes if strict else b.workspace_bytes <= t.workspace_bytes
    if spec.epilogue != workloads.EPI_SCALE_BATCHNORM_EVAL_AVGPOOL:
        assert b.info["gemm_min_bytes"] <= t.info["gemm_min_bytes"]
        # bf16 K steps hold 64 channels: padding may add products, never remove them
        assert b.info["issued_mma_flop"] >= t.info["issued_mma_flop"]


def test_parity_classes_tile_every_output_once(lib):
    # 3-D outputs with odd extents: per-class q-grids must partition the output grid
    for (D, k, s, p, op) in [(5, 3, 2, 1, 0), (6, 4, 2, 1, 1), (4, 5, 1, 2, 0), (3, 3, 2, 0, 1)]:
        pl = Plan(1, 4, 16, D, D + 1, D + 2, k, s, p, op, precision=1)
        Do, Ho, Wo = pl.out_shape[2:]
        covered = 0
        for rd in range(s):
            for rh in range(s):
                for rw in range(s):
                    covered += len(range(rd, Do, s)) * len(range(rh, Ho, s)) * len(range(rw, Wo, s))
        assert covered == Do * Ho * Wo
        assert pl.info["tiles"] >= -(-Do * Ho * Wo // 64)


def test_host_validation_before_any_launch(lib):
    st, h = create(lib)
    assert st == 0
    try:
        V = ctypes.c_void_p
        # NULL weight / workspace / x: rejected on the host, nothing is launched
        assert lib.convt3d_pack_weights(h, None, V(1 << 20), 1 << 30, None) == 1
        assert lib.convt3d_pack_weights(h, V(1 << 20), None, 1 << 30, None) == 3
        assert lib.convt3d_pack_weights(h, V(1 << 20), V(1 << 20), 16, None) == 3
        assert lib.convt3d_forward(h, None, None, None, None, V(1 << 20), V(1 << 20), 1 << 30, None) == 1
        # misaligned buffers
        assert lib.convt3d_forward(h, V((1 << 20) + 4), None, None, None, V(1 << 21), V(1 << 22), 1 << 30, None) == 1
        # forward before pack_weights on this workspace
        assert lib.convt3d_forward(h, V(1 << 20), None, None, None, V(1 << 21), V(1 << 22), 1 << 30, None) == 7
        # profile_read without a profiled forward
        ms = ctypes.c_float()
        assert lib.convt3d_profile_read(h, ctypes.byref(ms)) == 1
    finally:
        lib.convt3d_plan_destroy(h)


def test_groupnorm_requires_affine(lib):
    st, h = create(lib, epilogue=1, groups=4)
    assert st == 0
    try:
        V = ctypes.c_void_p
        assert lib.convt3d_forward(h, V(1 << 20), None, None, None, V(1 << 21), V(1 << 22), 1 << 30, None) == 1
    finally:
        lib.convt3d_plan_destroy(h)


def test_sample_range_validation(lib):
    """convt3d_forward_samples / convt3d_forward_finish: the range and the epilogue
    are checked on the host before anything else; a valid range then stops at the
    unpacked workspace, as convt3d_forward does."""
    V = ctypes.c_void_p
    st, h = create(lib, N=4, epilogue=2, has_bias=1)  # training-mode BatchNorm
    assert st == 0
    try:
        rng = lambda n0, n1: lib.convt3d_forward_samples(h, V(1 << 20), V(1 << 23), V(1 << 21), V(1 << 22),  # noqa
                                                         1 << 30, n0, n1, None)
        for n0, n1 in ((-1, 2), (0, 5), (2, 2), (3, 1)):
            assert rng(n0, n1) == 1, (n0, n1)
        assert rng(1, 3) == 7
        assert lib.convt3d_forward_samples(h, None, None, V(1 << 21), V(1 << 22), 1 << 30, 0, 4, None) == 1
        # finish needs gamma and beta for BatchNorm
        assert lib.convt3d_forward_finish(h, V(1 << 23), None, None, V(1 << 21), V(1 << 22), 1 << 30, None) == 1
        assert lib.convt3d_forward_finish(h, V(1 << 23), V(1 << 24), V(1 << 25), V(1 << 21), V(1 << 22),
                                          1 << 30, None) == 7
    finally:
        lib.convt3d_plan_destroy(h)
    st, h = create(lib, N=4, epilogue=4, has_bias=1)  # evaluation-mode BatchNorm: one pass over the batch
    assert st == 0
    try:
        assert lib.convt3d_forward_samples(h, V(1 << 20), V(1 << 23), V(1 << 21), V(1 << 22), 1 << 30, 0, 4,
                                           None) == 2
        assert lib.convt3d_forward_finish(h, V(1 << 23), V(1 << 24), V(1 << 25), V(1 << 21), V(1 << 22),
                                          1 << 30, None) == 2
    finally:
        lib.convt3d_plan_destroy(h)


def test_running_stats_validation_and_eval_requirement(lib):
    st, h = create(lib, epilogue=4, has_bias=1)
    assert st == 0
    try:
        V = ctypes.c_void_p
        out = (ctypes.c_int64 * 5)()
        assert lib.convt3d_output_shape(h, out) == 0
        assert tuple(out) == (2, 16, 1, 1, 1)
        fwd = lambda: lib.convt3d_forward(h, V(1 << 20), V(1 << 23), V(1 << 24), V(1 << 25), V(1 << 21),  # noqa: E731
                                          V(1 << 22), 1 << 30, None)
        # evaluation mode reads the running statistics: forward refuses until they are set
        assert fwd() == 1
        assert lib.convt3d_set_running_stats(h, V(1 << 26), None, 0.1) == 1
        assert lib.convt3d_set_running_stats(h, V(1 << 26), V(1 << 27), 1.5) == 1
        assert lib.convt3d_set_running_stats(h, V(1 << 26), V(1 << 27), -0.1) == 1
        assert lib.convt3d_set_running_stats(h, V((1 << 26) + 2), V(1 << 27), 0.1) == 1
        assert lib.convt3d_set_running_stats(h, V(1 << 26), V(1 << 27), 0.1) == 0
        assert fwd() == 7  # past the running-statistics check; stops at the unpacked workspace
        assert lib.convt3d_set_running_stats(h, None, None, 0.1) == 0
        assert fwd() == 1
    finally:
        lib.convt3d_plan_destroy(h)
