"""convt3d: dense fp32 ConvTranspose3d with fused epilogues on one GB300 (sm_103a).

The computation lives in libconvt3d.so (C ABI, include/convt3d.h); this package
is its PyTorch-facing binding.  Importing the package does not load the
library; the first Plan does, and fails loudly if it has not been built.
"""
from .api import (EPI_IDENTITY, EPI_RELU_GROUPNORM, EPI_SCALE_BATCHNORM_AVGPOOL,  # noqa: F401
                  EPI_SCALE_BATCHNORM_EVAL_AVGPOOL, EPI_SOFTMAX_SIGMOID, PREC_3XTF32, PREC_FFMA, PREC_TF32,
                  PREC_BF16, PREC_3XBF16, PREC_FP16, Convt3dError, HostPipeline, Plan, convt3d)
