"""ctypes declarations for libconvt3d.so (the C ABI in include/convt3d.h).

Loading fails loudly when the shared library is missing: there is no fallback
implementation anywhere in this package.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libconvt3d.so")

EPI_IDENTITY = 0
EPI_RELU_GROUPNORM = 1
EPI_SCALE_BATCHNORM_AVGPOOL = 2
EPI_SOFTMAX_SIGMOID = 3
EPI_SCALE_BATCHNORM_EVAL_AVGPOOL = 4

PREC_3XTF32 = 0
PREC_FFMA = 1
PREC_TF32 = 2
PREC_BF16 = 3
PREC_3XBF16 = 4
PREC_FP16 = 5

STATUS = {
    0: "CONVT3D_OK",
    1: "CONVT3D_ERR_INVALID_ARG",
    2: "CONVT3D_ERR_UNSUPPORTED",
    3: "CONVT3D_ERR_WORKSPACE",
    4: "CONVT3D_ERR_CUDA",
    5: "CONVT3D_ERR_TIMEOUT",
    6: "CONVT3D_ERR_DEVICE_ASSERT",
    7: "CONVT3D_ERR_NOT_PACKED",
}

# Every function include/convt3d.h declares (checked by the CPU tests).
EXPORTS = [
    "convt3d_plan_create", "convt3d_plan_destroy", "convt3d_output_shape", "convt3d_plan_info",
    "convt3d_workspace_bytes", "convt3d_pack_weights", "convt3d_forward", "convt3d_check",
    "convt3d_profile_enable", "convt3d_profile_read", "convt3d_status_string", "convt3d_last_error",
    "convt3d_version", "convt3d_forward_static_workspace", "convt3d_set_running_stats",
    "convt3d_forward_samples", "convt3d_forward_finish",
]


class Desc(ctypes.Structure):
    _fields_ = [
        ("N", ctypes.c_int), ("Cin", ctypes.c_int), ("Cout", ctypes.c_int),
        ("Din", ctypes.c_int), ("Hin", ctypes.c_int), ("Win", ctypes.c_int),
        ("k", ctypes.c_int), ("stride", ctypes.c_int), ("pad", ctypes.c_int), ("out_pad", ctypes.c_int),
        ("has_bias", ctypes.c_int), ("epilogue", ctypes.c_int), ("groups", ctypes.c_int),
        ("eps", ctypes.c_float), ("scale", ctypes.c_float), ("precision", ctypes.c_int),
        ("per_dim", ctypes.c_int), ("kdims", ctypes.c_int * 3), ("strides", ctypes.c_int * 3),
        ("pads", ctypes.c_int * 3), ("out_pads", ctypes.c_int * 3), ("dilation", ctypes.c_int * 3),
        ("conv_groups", ctypes.c_int), ("channels_last", ctypes.c_int), ("io_bf16", ctypes.c_int),
        ("io_fp16", ctypes.c_int),
    ]


class Info(ctypes.Structure):
    _fields_ = [
        ("out_shape", ctypes.c_int64 * 5), ("num_classes", ctypes.c_int), ("gemm_m", ctypes.c_int64),
        ("gemm_n", ctypes.c_int64), ("gemm_k_total", ctypes.c_int64), ("tiles", ctypes.c_int64),
        ("tile_m", ctypes.c_int), ("launches_per_forward", ctypes.c_int), ("launches_per_pack", ctypes.c_int),
        ("useful_flop", ctypes.c_double), ("issued_mma_flop", ctypes.c_double),
        ("gemm_min_bytes", ctypes.c_double), ("forward_min_bytes", ctypes.c_double),
        ("main_kernel", ctypes.c_int),
    ]


class Convt3dError(RuntimeError):
    def __init__(self, status: int, detail: str = ""):
        self.status = status
        super().__init__(f"{STATUS.get(status, status)}: {detail}")


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load libconvt3d.so; raise if it is not built."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"libconvt3d.so not found at {p}: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (there is no fallback path)")
        lib = ctypes.CDLL(p)
        V, P, I, S = ctypes.c_void_p, ctypes.POINTER, ctypes.c_int, ctypes.c_size_t
        lib.convt3d_plan_create.restype = I
        lib.convt3d_plan_create.argtypes = [P(Desc), P(V)]
        lib.convt3d_plan_destroy.restype = None
        lib.convt3d_plan_destroy.argtypes = [V]
        lib.convt3d_output_shape.restype = I
        lib.convt3d_output_shape.argtypes = [V, P(ctypes.c_int64)]
        lib.convt3d_plan_info.restype = I
        lib.convt3d_plan_info.argtypes = [V, P(Info)]
        lib.convt3d_workspace_bytes.restype = S
        lib.convt3d_workspace_bytes.argtypes = [V]
        lib.convt3d_pack_weights.restype = I
        lib.convt3d_pack_weights.argtypes = [V, V, V, S, V]
        lib.convt3d_forward.restype = I
        lib.convt3d_forward.argtypes = [V, V, V, V, V, V, V, S, V]
        lib.convt3d_check.restype = I
        lib.convt3d_check.argtypes = [V, V, V]
        lib.convt3d_profile_enable.restype = I
        lib.convt3d_profile_enable.argtypes = [V, I]
        lib.convt3d_profile_read.restype = I
        lib.convt3d_profile_read.argtypes = [V, P(ctypes.c_float)]
        lib.convt3d_status_string.restype = ctypes.c_char_p
        lib.convt3d_status_string.argtypes = [I]
        lib.convt3d_last_error.restype = ctypes.c_char_p
        lib.convt3d_last_error.argtypes = []
        lib.convt3d_version.restype = I
        lib.convt3d_version.argtypes = []
        lib.convt3d_forward_static_workspace.restype = I
        lib.convt3d_forward_static_workspace.argtypes = [V, V, V, V, V, V, V, V]
        lib.convt3d_set_running_stats.restype = I
        lib.convt3d_set_running_stats.argtypes = [V, V, V, ctypes.c_float]
        lib.convt3d_forward_samples.restype = I
        lib.convt3d_forward_samples.argtypes = [V, V, V, V, V, S, I, I, V]
        lib.convt3d_forward_finish.restype = I
        lib.convt3d_forward_finish.argtypes = [V, V, V, V, V, V, S, V]
        if path is None:
            _lib = lib
        return lib


def check(status: int, lib=None):
    if status != 0:
        lib = lib or load()
        raise Convt3dError(status, lib.convt3d_last_error().decode())
