"""ctypes wrapper and builder for the C oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: see the package docstring.  Arrays are numpy; the
wrapper checks dtypes and contiguity and nothing else -- every step of the
arithmetic is in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

EPI_IDENTITY = 0
EPI_RELU_GROUPNORM = 1
EPI_SCALE_BATCHNORM_AVGPOOL = 2
EPI_SOFTMAX_SIGMOID = 3
EPI_SCALE_BATCHNORM_EVAL_AVGPOOL = 4

_HERE = os.path.dirname(os.path.abspath(__file__))
# A different source may be named for mutation testing of the pins themselves.
_SRC = os.environ.get("CONVT3D_ORACLE_SRC") or os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.environ.get("CONVT3D_ORACLE_BUILD_DIR") or os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc + OpenMP into ``oracle/_build/liboracle.so``."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_output_size.restype = ctypes.c_long
        lib.oracle_output_size.argtypes = [ctypes.c_long] * 5
        lib.oracle_num_threads.restype = i
        lib.oracle_num_threads.argtypes = []
        lib.oracle_convt3d_scatter.restype = i
        lib.oracle_convt3d_scatter.argtypes = [i] * 10 + [P, P, P, P]
        lib.oracle_count_products.restype = None
        lib.oracle_count_products.argtypes = [i] * 10 + [P, P]
        lib.oracle_convt3d_forward.restype = i
        lib.oracle_convt3d_forward.argtypes = (
            [i] * 10 + [P, P, P, i, i, ctypes.c_double, ctypes.c_double, P, P, P, P, ctypes.c_double, P, P])
        lib.oracle_output_size_dil.restype = ctypes.c_long
        lib.oracle_output_size_dil.argtypes = [ctypes.c_long] * 6
        lib.oracle_convt3d_scatter_general.restype = i
        lib.oracle_convt3d_scatter_general.argtypes = [i] * 6 + [P] * 5 + [i] + [P] * 4
        lib.oracle_convt3d_forward_general.restype = i
        lib.oracle_convt3d_forward_general.argtypes = (
            [i] * 6 + [P] * 5 + [i] + [P, P, P, i, i, ctypes.c_double, ctypes.c_double, P, P, P, P,
                                      ctypes.c_double, P, P])
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a, name):
    if a is None:
        return None
    a = np.asarray(a)
    if a.dtype != np.float32 or not a.flags.c_contiguous:
        raise TypeError(f"{name} must be a C-contiguous float32 array")
    return a


def output_size(n_in: int, k: int, stride: int, pad: int, out_pad: int) -> int:
    return int(_load().oracle_output_size(n_in, k, stride, pad, out_pad))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def _shape(x, w, k, stride, pad, out_pad):
    N, Cin, Din, Hin, Win = x.shape
    if w.shape[0] != Cin or w.shape[2:] != (k, k, k):
        raise ValueError("w must be [Cin, Cout, k, k, k]")
    Cout = w.shape[1]
    Do, Ho, Wo = (output_size(d, k, stride, pad, out_pad) for d in (Din, Hin, Win))
    return N, Cin, Cout, Din, Hin, Win, Do, Ho, Wo


def convt3d_scatter(x, w, bias=None, *, stride=1, pad=0, out_pad=0):
    """fp64 scatter-form transposed convolution (+bias); returns [N,Cout,Do,Ho,Wo] float64."""
    x, w, bias = _f32(x, "x"), _f32(w, "w"), _f32(bias, "bias")
    k = w.shape[2]
    N, Cin, Cout, Din, Hin, Win, Do, Ho, Wo = _shape(x, w, k, stride, pad, out_pad)
    Y = np.empty((N, Cout, Do, Ho, Wo), np.float64)
    rc = _load().oracle_convt3d_scatter(N, Cin, Cout, Din, Hin, Win, k, stride, pad, out_pad,
                                        _ptr(x), _ptr(w), _ptr(bias), _ptr(Y))
    if rc:
        raise ValueError(f"oracle_convt3d_scatter failed ({rc})")
    return Y


def count_products(N, Cin, Cout, Din, Hin, Win, k, stride, pad, out_pad):
    """(in_range, total) products of the scatter loop nest."""
    a, b = ctypes.c_double(), ctypes.c_double()
    _load().oracle_count_products(N, Cin, Cout, Din, Hin, Win, k, stride, pad, out_pad,
                                  ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


def _triple(v, name):
    t = (int(v),) * 3 if np.isscalar(v) else tuple(int(a) for a in v)
    if len(t) != 3:
        raise ValueError(f"{name} must be an int or 3 ints (d, h, w)")
    return t


def _ints(t):
    return (ctypes.c_int * 3)(*t)


def output_size_dil(n_in: int, k: int, stride: int, pad: int, out_pad: int, dilation: int) -> int:
    return int(_load().oracle_output_size_dil(n_in, k, stride, pad, out_pad, dilation))


def _general_shape(x, w, stride, pad, out_pad, dilation, conv_groups):
    N, Cin, Din, Hin, Win = x.shape
    if w.ndim != 5 or w.shape[0] != Cin:
        raise ValueError("w must be [Cin, Cout/groups, kd, kh, kw]")
    kk = tuple(int(a) for a in w.shape[2:])
    ss, pp, oo, dd = (_triple(v, n) for v, n in ((stride, "stride"), (pad, "pad"), (out_pad, "out_pad"),
                                                  (dilation, "dilation")))
    Cout = w.shape[1] * int(conv_groups)
    outs = tuple(output_size_dil(i, kk[a], ss[a], pp[a], oo[a], dd[a]) for a, i in enumerate((Din, Hin, Win)))
    return N, Cin, Cout, (Din, Hin, Win), kk, ss, pp, oo, dd, outs


def convt3d_scatter_general(x, w, bias=None, *, stride=1, pad=0, out_pad=0, dilation=1, conv_groups=1):
    """fp64 scatter form with per-dimension shapes, dilation and groups; w is
    [Cin, Cout/groups, kd, kh, kw].  Returns [N,Cout,Do,Ho,Wo] float64."""
    x, w, bias = _f32(x, "x"), _f32(w, "w"), _f32(bias, "bias")
    N, Cin, Cout, ins, kk, ss, pp, oo, dd, outs = _general_shape(x, w, stride, pad, out_pad, dilation, conv_groups)
    Y = np.empty((N, Cout) + outs, np.float64)
    rc = _load().oracle_convt3d_scatter_general(N, Cin, Cout, *ins, _ints(kk), _ints(ss), _ints(pp), _ints(oo),
                                                _ints(dd), int(conv_groups), _ptr(x), _ptr(w), _ptr(bias), _ptr(Y))
    if rc:
        raise ValueError(f"oracle_convt3d_scatter_general failed ({rc})")
    return Y


def forward(x, w, bias=None, *, stride=1, pad=0, out_pad=0, dilation=1, conv_groups=1, epilogue=EPI_IDENTITY,
            groups=1, eps=1e-5, scale=1.0, gamma=None, beta=None, running_mean=None,
            running_var=None, momentum=0.1, want_f64=False):
    """Transposed convolution + epilogue, fp64 inside, fp32 result.

    stride / pad / out_pad / dilation: an int or (d, h, w); the kernel extents
    come from w, [Cin, Cout/conv_groups, kd, kh, kw].  ``groups`` is the
    GroupNorm group count.  Returns y (float32) or (y, y64) when ``want_f64``.
    Shapes: [N,Cout,Do,Ho,Wo], or [N,Cout,1,1,1] for the BN+pool epilogues.
    running_mean / running_var (float32 [Cout]) are read by the evaluation-mode
    epilogue and updated in place by the batch-statistics one.
    """
    x, w = _f32(x, "x"), _f32(w, "w")
    bias, gamma, beta = _f32(bias, "bias"), _f32(gamma, "gamma"), _f32(beta, "beta")
    running_mean, running_var = _f32(running_mean, "running_mean"), _f32(running_var, "running_var")
    N, Cin, Cout, ins, kk, ss, pp, oo, dd, outs = _general_shape(x, w, stride, pad, out_pad, dilation, conv_groups)
    pooled = epilogue in (EPI_SCALE_BATCHNORM_AVGPOOL, EPI_SCALE_BATCHNORM_EVAL_AVGPOOL)
    shape = (N, Cout, 1, 1, 1) if pooled else (N, Cout) + outs
    y = np.empty(shape, np.float32)
    y64 = np.empty(shape, np.float64) if want_f64 else None
    rc = _load().oracle_convt3d_forward_general(N, Cin, Cout, *ins, _ints(kk), _ints(ss), _ints(pp), _ints(oo),
                                                _ints(dd), int(conv_groups), _ptr(x), _ptr(w), _ptr(bias),
                                                int(epilogue), int(groups), float(eps), float(scale), _ptr(gamma),
                                                _ptr(beta), _ptr(running_mean), _ptr(running_var), float(momentum),
                                                _ptr(y), _ptr(y64))
    if rc:
        raise ValueError(f"oracle_convt3d_forward_general failed ({rc})")
    return (y, y64) if want_f64 else y
