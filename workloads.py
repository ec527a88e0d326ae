"""Seeded synthetic workloads shared by the tests, the smoke check and the benchmark.

This module holds shapes, distributions and seeds only -- none of the method's
arithmetic -- so that the CUDA library and the CPU oracle read identical input
bytes without either importing the other.

The workloads are the shapes of the three transcript pages (l2_p61
ReLU+GroupNorm, l2_p77 scale+BatchNorm+pool, l2_p49 stride-2 softmax+sigmoid),
a tiny parity case, a bare stride-2 k=4 identity case and the BatchNorm shape
in evaluation mode.  Values: x ~ N(0,1);
weight and bias ~ U(-b, b) with b = 1/sqrt(Cout/G * kd*kh*kw) (PyTorch's
ConvTranspose3d default bound; G = convolution groups); gamma ~ U(0.5, 1.5) and beta ~ U(-0.5, 0.5) where an affine
normalisation is present; BatchNorm running statistics from make_running_stats.
Drawn on the CPU in fp32 from one
torch.Generator seeded with 20261202 + workload index, in the order x, w, bias,
gamma, beta (absent tensors are not drawn).
"""
from __future__ import annotations

import dataclasses
import math

import torch

EPI_IDENTITY = 0
EPI_RELU_GROUPNORM = 1
EPI_SCALE_BATCHNORM_AVGPOOL = 2
EPI_SOFTMAX_SIGMOID = 3
EPI_SCALE_BATCHNORM_EVAL_AVGPOOL = 4

SEED_BASE = 20261202


@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    N: int
    Cin: int
    Cout: int
    D: int
    H: int
    W: int
    k: int
    stride: int = 1
    pad: int = 0
    out_pad: int = 0
    bias: bool = False
    epilogue: int = EPI_IDENTITY
    groups: int = 1
    eps: float = 1e-5
    scale: float = 1.0
    seed_index: int = 0
    dilation: object = 1     # int or (d, h, w); k, stride, pad, out_pad likewise
    conv_groups: int = 1
    channels_last: bool = False  # x and y in NDHWC memory order (make_inputs still returns NCDHW x)
    io_bf16: bool = False        # x, w and y as bf16 tensors (make_inputs still returns fp32 values)
    io_fp16: bool = False        # x, w and y as fp16 tensors (likewise)

    @property
    def kdims(self):
        return tuple(self.k) if isinstance(self.k, (tuple, list)) else (self.k,) * 3

    @property
    def kvol(self):
        a, b, c = self.kdims
        return a * b * c

    @property
    def affine(self) -> bool:
        return self.epilogue in (EPI_RELU_GROUPNORM, EPI_SCALE_BATCHNORM_AVGPOOL, EPI_SCALE_BATCHNORM_EVAL_AVGPOOL)

    def useful_flop(self) -> float:
        """2*N*Cout*(Cin/G)*kd*kh*kw*Din*Hin*Win: every product of the definition, no zero taps."""
        return 2.0 * self.N * self.Cout * (self.Cin // self.conv_groups) * self.kvol * self.D * self.H * self.W

    def replace(self, **kw) -> "Spec":
        return dataclasses.replace(self, **kw)


TINY = Spec("tiny_relu_groupnorm", N=2, Cin=8, Cout=16, D=8, H=8, W=8, k=3,
            epilogue=EPI_RELU_GROUPNORM, groups=4, seed_index=0)
GN = Spec("relu_groupnorm_16x64x32c_k3", N=16, Cin=64, Cout=128, D=32, H=32, W=32, k=3,
          epilogue=EPI_RELU_GROUPNORM, groups=8, seed_index=1)
BN = Spec("scale_batchnorm_avgpool_16x64x16x32x32_k5", N=16, Cin=64, Cout=128, D=16, H=32, W=32,
          k=5, bias=True, epilogue=EPI_SCALE_BATCHNORM_AVGPOOL, scale=2.0, seed_index=2)
SOFTMAX = Spec("softmax_sigmoid_16x32x16x32x32_k3s2", N=16, Cin=32, Cout=64, D=16, H=32, W=32,
               k=3, stride=2, pad=1, out_pad=1, bias=True, epilogue=EPI_SOFTMAX_SIGMOID,
               seed_index=3)
IDENTITY = Spec("identity_8x128x16x32x32_k4s2", N=8, Cin=128, Cout=128, D=16, H=32, W=32, k=4,
                stride=2, pad=1, out_pad=0, bias=True, epilogue=EPI_IDENTITY, seed_index=4)

# The BatchNorm shape with stored running statistics (evaluation mode).
BN_EVAL = Spec("scale_batchnorm_eval_avgpool_16x64x16x32x32_k5", N=16, Cin=64, Cout=128, D=16, H=32, W=32,
               k=5, bias=True, epilogue=EPI_SCALE_BATCHNORM_EVAL_AVGPOOL, scale=2.0, seed_index=5)

ALL = [TINY, GN, BN, SOFTMAX, IDENTITY, BN_EVAL]
BY_NAME = {s.name: s for s in ALL}


def make_inputs(spec: Spec, seed: int | None = None) -> dict:
    """CPU fp32 tensors x, w, bias, gamma, beta (None where absent)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(SEED_BASE + spec.seed_index if seed is None else seed)
    bound = 1.0 / math.sqrt(spec.Cout // spec.conv_groups * spec.kvol)
    x = torch.randn((spec.N, spec.Cin, spec.D, spec.H, spec.W), generator=g, dtype=torch.float32)
    w = torch.empty((spec.Cin, spec.Cout // spec.conv_groups) + spec.kdims, dtype=torch.float32)
    w.uniform_(-bound, bound, generator=g)
    bias = gamma = beta = None
    if spec.bias:
        bias = torch.empty(spec.Cout, dtype=torch.float32).uniform_(-bound, bound, generator=g)
    if spec.affine:
        gamma = torch.empty(spec.Cout, dtype=torch.float32).uniform_(0.5, 1.5, generator=g)
        beta = torch.empty(spec.Cout, dtype=torch.float32).uniform_(-0.5, 0.5, generator=g)
    return {"x": x, "w": w, "bias": bias, "gamma": gamma, "beta": beta}


def make_running_stats(spec: Spec, seed: int | None = None):
    """BatchNorm running mean ~ U(-0.2, 0.2) and running variance ~ U(0.5, 2.0),
    CPU fp32, Cout each, seeded with 20261202 + 1000 + workload index."""
    g = torch.Generator(device="cpu")
    g.manual_seed(SEED_BASE + 1000 + spec.seed_index if seed is None else seed)
    rm = torch.empty(spec.Cout, dtype=torch.float32).uniform_(-0.2, 0.2, generator=g)
    rv = torch.empty(spec.Cout, dtype=torch.float32).uniform_(0.5, 2.0, generator=g)
    return rm, rv


def sample_slice(inputs: dict, n0: int, n1: int) -> dict:
    """The same tensors restricted to batch samples [n0, n1) (weights unchanged)."""
    out = dict(inputs)
    out["x"] = inputs["x"][n0:n1].contiguous()
    return out
