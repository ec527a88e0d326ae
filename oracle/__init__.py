"""convt3d oracle -- TEST INFRASTRUCTURE ONLY.

A plain CPU statement (fp64 accumulation, scatter form) of the dense 3-D
transposed convolution and its four epilogues, used to prove the GPU library
right.  Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline arm may import it; the product path never does.  It shares no code
with the CUDA library.

Functions whose pins live in ``tests/test_oracle_pins.py``:
  output_size      -- pinned by the page shapes and the 1-D examples
  convt3d_scatter  -- pinned by the 1-D worked examples (l2_p61), the stride-2
                      tap table (l2_p49), the stride-1 flipped-kernel identity,
                      the adjoint identity, linearity, the pooled-sum closed form
  forward          -- epilogues pinned by GN / softmax / BN invariants, the
                      BN+pool closed form (l2_p77), and PyTorch CPU fp64
                      batch_norm in evaluation mode and its running statistics
  count_products   -- pinned by the product count printed on page l2_p49
  convt3d_scatter_general, output_size_dil
                   -- per-dimension kernel/stride/padding, dilation and
                      grouped convolution: pinned by PyTorch CPU fp64
                      conv_transpose3d, the adjoint identity against an
                      independently written dilated grouped correlation, and
                      the block structure of grouped convolution
"""
from .oracle import (  # noqa: F401
    EPI_IDENTITY,
    EPI_RELU_GROUPNORM,
    EPI_SCALE_BATCHNORM_AVGPOOL,
    EPI_SCALE_BATCHNORM_EVAL_AVGPOOL,
    EPI_SOFTMAX_SIGMOID,
    build,
    convt3d_scatter,
    convt3d_scatter_general,
    count_products,
    forward,
    num_threads,
    output_size,
    output_size_dil,
)
