"""PyTorch-facing binding of the convt3d C ABI.

Argument marshalling only: tensors are checked, their device pointers and the
current CUDA stream are handed to libconvt3d, and every step of the
computation runs in the library's kernels.  PyTorch supplies device memory and
streams.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (EPI_IDENTITY, EPI_RELU_GROUPNORM, EPI_SCALE_BATCHNORM_AVGPOOL,  # noqa: F401
                   EPI_SCALE_BATCHNORM_EVAL_AVGPOOL, EPI_SOFTMAX_SIGMOID, PREC_3XTF32, PREC_FFMA,
                   PREC_TF32, PREC_BF16, PREC_3XBF16, PREC_FP16, Convt3dError)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _triple(v):
    if isinstance(v, (tuple, list)):
        if len(v) != 3:
            raise ValueError("expected an int or 3 ints (d, h, w)")
        return tuple(int(a) for a in v)
    return (int(v),) * 3


def make_desc(N, Cin, Cout, D, H, W, k, stride=1, pad=0, out_pad=0, bias=False, epilogue=EPI_IDENTITY,
              groups=1, eps=1e-5, scale=1.0, precision=PREC_3XTF32, dilation=1, conv_groups=1,
              channels_last=False, io_bf16=False, io_fp16=False):
    """A convt3d_desc_t.  k, stride, pad, out_pad and dilation are an int or
    (d, h, w); conv_groups is the convolution's group count (weight
    [Cin, Cout/conv_groups, kd, kh, kw]); groups is GroupNorm's; channels_last
    selects NDHWC x and y; io_bf16 / io_fp16 make x, w and y 16-bit tensors."""
    kk, ss, pp, oo, dd = (_triple(v) for v in (k, stride, pad, out_pad, dilation))
    per_dim = any(len(set(t)) > 1 for t in (kk, ss, pp, oo))
    d = _lib.Desc(N, Cin, Cout, D, H, W, kk[0], ss[0], pp[0], oo[0], int(bool(bias)), int(epilogue), int(groups),
                  float(eps), float(scale), int(precision))
    d.per_dim = int(per_dim)
    for a in range(3):
        d.kdims[a], d.strides[a], d.pads[a], d.out_pads[a], d.dilation[a] = kk[a], ss[a], pp[a], oo[a], dd[a]
    d.conv_groups = int(conv_groups)
    d.channels_last = int(bool(channels_last))
    d.io_bf16 = int(bool(io_bf16))
    d.io_fp16 = int(bool(io_fp16))
    return d


class Plan:
    """A validated problem description (host-only; creating one needs no GPU)."""

    def __init__(self, N, Cin, Cout, D, H, W, k, stride=1, pad=0, out_pad=0, bias=False,
                 epilogue=EPI_IDENTITY, groups=1, eps=1e-5, scale=1.0, precision=PREC_3XTF32, dilation=1,
                 conv_groups=1, channels_last=False, io_bf16=False, io_fp16=False):
        self.lib = _lib.load()
        self.channels_last = bool(channels_last)
        # x, w and y
        self.io_dtype = torch.bfloat16 if io_bf16 else (torch.float16 if io_fp16 else torch.float32)
        self.desc = make_desc(N, Cin, Cout, D, H, W, k, stride, pad, out_pad, bias, epilogue, groups, eps, scale,
                              precision, dilation, conv_groups, channels_last, io_bf16, io_fp16)
        h = ctypes.c_void_p()
        _lib.check(self.lib.convt3d_plan_create(ctypes.byref(self.desc), ctypes.byref(h)), self.lib)
        self.handle = h
        shp = (ctypes.c_int64 * 5)()
        _lib.check(self.lib.convt3d_output_shape(self.handle, shp), self.lib)
        self.out_shape = tuple(int(v) for v in shp)  # logical [N, Cout, Do, Ho, Wo]
        # memory shape of y: NDHWC when channels_last (the pooled [N, Cout, 1, 1, 1] is the same either way)
        n_, c_, d_, h_, w_ = self.out_shape
        self.out_alloc_shape = (n_, d_, h_, w_, c_) if self.channels_last else self.out_shape
        self.workspace_bytes = int(self.lib.convt3d_workspace_bytes(self.handle))
        inf = _lib.Info()
        _lib.check(self.lib.convt3d_plan_info(self.handle, ctypes.byref(inf)), self.lib)
        self.info = {f: (tuple(getattr(inf, f)) if f == "out_shape" else getattr(inf, f))
                     for f, _ in _lib.Info._fields_}

    @classmethod
    def from_spec(cls, spec, precision=PREC_3XTF32):
        return cls(spec.N, spec.Cin, spec.Cout, spec.D, spec.H, spec.W, spec.k, spec.stride, spec.pad,
                   spec.out_pad, spec.bias, spec.epilogue, spec.groups, spec.eps, spec.scale, precision,
                   spec.dilation, spec.conv_groups, spec.channels_last, spec.io_bf16,
                   getattr(spec, "io_fp16", False))

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            self.lib.convt3d_plan_destroy(h)
            self.handle = None

    # -- device buffers --------------------------------------------------
    def new_workspace(self, device="cuda"):
        # 256-byte alignment: the caching allocator hands out 512-byte aligned blocks
        return torch.empty(max(self.workspace_bytes, 256), dtype=torch.uint8, device=device)

    def new_output(self, device="cuda"):
        return torch.empty(self.out_alloc_shape, dtype=self.io_dtype, device=device)

    @staticmethod
    def _dev(t, name, dtype=torch.float32):
        if t is None:
            return None
        if not (t.is_cuda and t.dtype == dtype and t.is_contiguous()):
            raise TypeError(f"{name} must be a contiguous {dtype} CUDA tensor")
        return t

    def _check_y(self, y):
        if tuple(y.shape) not in (self.out_shape, self.out_alloc_shape) and y.numel() != _numel(self.out_shape):
            raise ValueError(f"y has shape {tuple(y.shape)}, expected {self.out_alloc_shape}")

    # -- library calls ---------------------------------------------------
    def pack_weights(self, w, workspace, stream=None):
        self._dev(w, "w", self.io_dtype)
        _lib.check(self.lib.convt3d_pack_weights(self.handle, _ptr(w), _ptr(workspace),
                                                 workspace.numel(), _stream(stream)), self.lib)

    def forward(self, x, y, workspace, bias=None, gamma=None, beta=None, stream=None):
        self._dev(x, "x", self.io_dtype)
        self._dev(y, "y", self.io_dtype)
        for t, n in ((bias, "bias"), (gamma, "gamma"), (beta, "beta")):
            self._dev(t, n)
        self._check_y(y)
        _lib.check(self.lib.convt3d_forward(self.handle, _ptr(x), _ptr(bias), _ptr(gamma), _ptr(beta),
                                            _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream)),
                   self.lib)
        return y

    def forward_samples(self, x, y, workspace, n0, n1, bias=None, stream=None):
        """The per-sample part of forward for samples [n0, n1) of the batch: x and y
        are the whole batch's tensors, only those samples are read and written.
        Calls covering every sample once, then forward_finish, give forward's y."""
        self._dev(x, "x", self.io_dtype)
        self._dev(y, "y", self.io_dtype)
        self._dev(bias, "bias")
        self._check_y(y)
        if tuple(x.shape)[0] != self.desc.N:
            raise ValueError(f"x must hold the whole batch of N={self.desc.N} samples")
        _lib.check(self.lib.convt3d_forward_samples(self.handle, _ptr(x), _ptr(bias), _ptr(y), _ptr(workspace),
                                                    workspace.numel(), int(n0), int(n1), _stream(stream)),
                   self.lib)
        return y

    def forward_finish(self, y, workspace, bias=None, gamma=None, beta=None, stream=None):
        """The passes over the whole batch after forward_samples (GroupNorm's
        normalisation, BatchNorm's statistics and pooled output)."""
        self._dev(y, "y", self.io_dtype)
        for t, n in ((bias, "bias"), (gamma, "gamma"), (beta, "beta")):
            self._dev(t, n)
        self._check_y(y)
        _lib.check(self.lib.convt3d_forward_finish(self.handle, _ptr(bias), _ptr(gamma), _ptr(beta), _ptr(y),
                                                   _ptr(workspace), workspace.numel(), _stream(stream)), self.lib)
        return y

    def forward_static_workspace(self, w, x, y, bias=None, gamma=None, beta=None, stream=None):
        """Pack w and run the forward in the library's built-in 32 MiB device
        workspace, for callers that may not allocate device memory.  Calls that
        overlap on the GPU share that workspace and race."""
        for t, n in ((w, "w"), (x, "x"), (y, "y")):
            self._dev(t, n, self.io_dtype)
        for t, n in ((bias, "bias"), (gamma, "gamma"), (beta, "beta")):
            self._dev(t, n)
        _lib.check(self.lib.convt3d_forward_static_workspace(self.handle, _ptr(w), _ptr(x), _ptr(bias),
                                                             _ptr(gamma), _ptr(beta), _ptr(y), _stream(stream)),
                   self.lib)
        return y

    def set_running_stats(self, running_mean, running_var, momentum=0.1):
        """BatchNorm running statistics (Cout floats each on the device, or both
        None to clear).  The training-mode BatchNorm epilogue updates them in
        place on every forward; the evaluation-mode one normalises with them.
        The plan keeps references so the tensors outlive its use of them."""
        if (running_mean is None) != (running_var is None):
            raise ValueError("running_mean and running_var are set together")
        for t, n in ((running_mean, "running_mean"), (running_var, "running_var")):
            self._dev(t, n)
            if t is not None and t.numel() != self.desc.Cout:
                raise ValueError(f"{n} must hold Cout={self.desc.Cout} values")
        _lib.check(self.lib.convt3d_set_running_stats(self.handle, _ptr(running_mean), _ptr(running_var),
                                                      float(momentum)), self.lib)
        self._running = (running_mean, running_var)

    def check(self, workspace, stream=None):
        _lib.check(self.lib.convt3d_check(self.handle, _ptr(workspace), _stream(stream)), self.lib)

    def profile_enable(self, on=True):
        _lib.check(self.lib.convt3d_profile_enable(self.handle, int(bool(on))), self.lib)

    def profile_read(self) -> float:
        ms = ctypes.c_float()
        _lib.check(self.lib.convt3d_profile_read(self.handle, ctypes.byref(ms)), self.lib)
        return float(ms.value)


def _numel(shape):
    n = 1
    for v in shape:
        n *= v
    return n


def convt3d(x, w, bias=None, *, stride=1, pad=0, out_pad=0, dilation=1, conv_groups=1, epilogue=EPI_IDENTITY,
            groups=1, eps=1e-5, scale=1.0, gamma=None, beta=None, precision=PREC_3XTF32):
    """One-shot convenience: plan, pack, forward on the current stream; returns y.
    w is [Cin, Cout/conv_groups, kd, kh, kw]."""
    N, Cin, D, H, W = x.shape
    Cout, k = w.shape[1] * conv_groups, tuple(w.shape[2:])
    plan = Plan(N, Cin, Cout, D, H, W, k, stride, pad, out_pad, bias is not None, epilogue, groups, eps, scale,
                precision, dilation, conv_groups)
    ws = plan.new_workspace(x.device)
    y = plan.new_output(x.device)
    plan.pack_weights(w, ws)
    plan.forward(x, y, ws, bias, gamma, beta)
    return y


class HostPipeline:
    """Forward from host memory to host memory with the copies overlapped.

    The batch is split into chunks of samples; chunk i's host->device copy,
    chunk i-1's computation and chunk i-2's device->host copy run at once, each
    copy split over `copy_streams` streams per direction.  Epilogues whose result
    for a sample depends on that sample only (identity, ReLU+GroupNorm,
    softmax+sigmoid, evaluation-mode BatchNorm) run each chunk as a forward of a
    chunk-sized plan.  Training-mode BatchNorm, whose statistics cover the whole
    batch, runs one whole-batch plan: Plan.forward_samples on each chunk as its
    input arrives, then Plan.forward_finish, and copies the pooled y out at the
    end.  Host tensors should be pinned for the copies to be asynchronous.
    Device buffers, plans and streams are created once, here.
    """

    def __init__(self, N, Cin, Cout, D, H, W, k, stride=1, pad=0, out_pad=0, bias=False,
                 epilogue=EPI_IDENTITY, groups=1, eps=1e-5, scale=1.0, precision=PREC_3XTF32, chunks=4,
                 device="cuda", dilation=1, conv_groups=1, copy_streams=1, channels_last=False, io_bf16=False,
                 io_fp16=False):
        # training-mode BatchNorm: one whole-batch plan run in sample ranges
        self.ranges = epilogue == EPI_SCALE_BATCHNORM_AVGPOOL
        chunks = max(1, min(int(chunks), N))
        if N % chunks and not self.ranges:  # chunk-sized plans need equal chunks; ranges need not
            chunks = 1
        args = (Cin, Cout, D, H, W, k, stride, pad, out_pad, bias, epilogue, groups, eps, scale, precision,
                dilation, conv_groups, channels_last, io_bf16, io_fp16)
        self.plan = Plan(N if self.ranges else N // chunks, *args)
        if self.ranges and self.plan.info["main_kernel"] == 2:
            chunks = 1  # that kernel reads the whole batch in one launch
        self.chunks = chunks
        self.n_chunk = N // chunks
        dt = self.plan.io_dtype
        self.full_shape = (N,) + self.plan.out_alloc_shape[1:]
        dev = torch.device(device)
        self.x = torch.empty((N, D, H, W, Cin) if channels_last else (N, Cin, D, H, W), dtype=dt, device=dev)
        self.y = torch.empty(self.full_shape, dtype=dt, device=dev)
        self.w = torch.empty((Cin, Cout // conv_groups) + _triple(k), dtype=dt, device=dev)
        self.vec = {name: torch.empty(Cout, dtype=torch.float32, device=dev) for name in ("bias", "gamma", "beta")}
        self.ws = self.plan.new_workspace(dev)
        # each chunk's copies are split over `copy_streams` streams per direction, so
        # that several copy engines move it at once
        self.copy_streams = max(1, int(copy_streams))
        self.s_in = [torch.cuda.Stream(dev) for _ in range(self.copy_streams)]
        self.s_out = [torch.cuda.Stream(dev) for _ in range(self.copy_streams)]
        self.s_comp = torch.cuda.Stream(dev)
        # sample ranges alternate between two compute streams, so that a range's main
        # kernel fills the SMs that the previous range's last wave of tiles leaves idle
        self.s_comp2 = torch.cuda.Stream(dev)

    def set_running_stats(self, running_mean, running_var, momentum=0.1):
        """Device-resident BatchNorm running statistics, as Plan.set_running_stats."""
        self.plan.set_running_stats(running_mean, running_var, momentum)

    def __call__(self, x_host, w_host, y_host, bias=None, gamma=None, beta=None, stream=None):
        """Run on pinned host tensors; returns y_host.  The work is ordered after
        `stream` (default: current stream) and `stream` waits for its end."""
        caller = stream if stream is not None else torch.cuda.current_stream()
        for s in self.s_in + self.s_out + [self.s_comp, self.s_comp2]:
            s.wait_stream(caller)
        nc, k, N = self.n_chunk, self.copy_streams, self.x.shape[0]

        def pieces(dst, src):  # the same k contiguous slices of two equally shaped tensors
            d, s_ = dst.view(-1), src.reshape(-1)
            n = d.numel()
            for j in range(k):
                a, b = n * j // k, n * (j + 1) // k
                yield j, d[a:b], s_[a:b]

        with torch.cuda.stream(self.s_in[0]):
            self.w.copy_(w_host, non_blocking=True)
            dv = {}
            for name, t in (("bias", bias), ("gamma", gamma), ("beta", beta)):
                if t is not None:
                    self.vec[name].copy_(t, non_blocking=True)
                    dv[name] = self.vec[name]
                else:
                    dv[name] = None
            params_in = torch.cuda.Event()
            params_in.record(self.s_in[0])
        # the weight is packed while the first chunk of x is still on its way in
        comp = (self.s_comp, self.s_comp2) if self.ranges else (self.s_comp,)
        comp[0].wait_event(params_in)
        self.plan.pack_weights(self.w, self.ws, comp[0])
        if len(comp) > 1:
            packed = torch.cuda.Event()
            packed.record(comp[0])
            comp[1].wait_event(packed)
        # each chunk's compute is issued right after its copy, so that the GPU can start on
        # chunk 0 while the host is still issuing the later chunks
        for i in range(self.chunks):
            rows = slice(i * N // self.chunks, (i + 1) * N // self.chunks) if self.ranges else \
                slice(i * nc, (i + 1) * nc)
            s = comp[i % len(comp)]
            for j, d, s_ in pieces(self.x[rows], x_host[rows]):
                with torch.cuda.stream(self.s_in[j]):
                    d.copy_(s_, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(self.s_in[j])
                s.wait_event(ev)
            if self.ranges:
                # training-mode BatchNorm: the ranges touch disjoint samples of x, y, the staged
                # input and the per-tile statistics, so two of them may run at once on the two streams
                self.plan.forward_samples(self.x, self.y, self.ws, rows.start, rows.stop, dv["bias"], s)
                continue
            self.plan.forward(self.x[rows], self.y[rows], self.ws, dv["bias"], dv["gamma"], dv["beta"], s)
            ev = torch.cuda.Event()
            ev.record(s)
            for j, d, s_ in pieces(y_host[rows], self.y[rows]):
                self.s_out[j].wait_event(ev)
                with torch.cuda.stream(self.s_out[j]):
                    d.copy_(s_, non_blocking=True)
        if self.ranges:
            self.s_comp.wait_stream(self.s_comp2)
            self.plan.forward_finish(self.y, self.ws, dv["bias"], dv["gamma"], dv["beta"], self.s_comp)
            with torch.cuda.stream(self.s_comp):
                y_host.copy_(self.y, non_blocking=True)
        for s in self.s_out + [self.s_comp, self.s_comp2]:
            caller.wait_stream(s)
        return y_host
