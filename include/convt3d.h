/*
 * convt3d -- dense fp32 3-D transposed convolution with fused epilogues for
 * one NVIDIA GB300 GPU (sm_103a).
 *
 * The operation (the three POPCORNBENCH "Kimi-K2.6" transcript pages
 * l2_p77, l2_p61 and l2_p49; each page's opening problem statement and its
 * derivation of the transposed-convolution index mapping):
 *
 *   Y[n,co,od,oh,ow] = bias[co] + sum over ci, kd, kh, kw of
 *                      x[n,ci,id,ih,iw] * w[ci,co,kd,kh,kw]
 *   where od = id*stride - pad + kd (likewise oh, ow), restricted to
 *   0 <= od < Do, and Do = (Din - 1)*stride - 2*pad + k + out_pad.
 *
 * General form (PyTorch's ConvTranspose3d; page l2_p61's shape analysis
 * writes the dilated extent): per-dimension kernel extent, stride, padding
 * and output padding, dilation (od = id*s - p + dil*kd, Do = (Din - 1)*s - 2p
 * + dil*(kd - 1) + op + 1) and G convolution groups (output channel co reads
 * the Cin/G input channels of its group; w is [Cin, Cout/G, kd, kh, kw]).
 *
 * followed by one epilogue:
 *   IDENTITY                  y = Y                                     (no page; bare op)
 *   RELU_GROUPNORM            v = max(Y,0); GroupNorm(groups) with biased
 *                             variance over (channels of the group, all
 *                             positions) per sample; affine gamma/beta    (page l2_p61)
 *   SCALE_BATCHNORM_AVGPOOL   z = scale*Y; BatchNorm3d with batch statistics
 *                             (biased variance over n and positions, per
 *                             channel); affine; mean over positions
 *                             -> [N, Cout, 1, 1, 1]                       (page l2_p77)
 *   SOFTMAX_SIGMOID           softmax over channels, then elementwise
 *                             sigmoid                                     (page l2_p49)
 *   SCALE_BATCHNORM_EVAL_AVGPOOL
 *                             z = scale*Y; BatchNorm3d in evaluation mode
 *                             (stored running mean/variance); affine; mean
 *                             over positions -> [N, Cout, 1, 1, 1]        (page l2_p77's
 *                                                                          submitted solution)
 *
 * Computation: an output-stationary implicit GEMM, M = output positions,
 * N = Cout, K = Cin x taps.  Stride 2 is split into the output-parity
 * classes (8 when all three strides are 2), each a dense stride-1
 * correlation over only the taps that reach it, so no zero-inserted taps are
 * multiplied.  Grouped convolution runs as the dense GEMM over a packed
 * weight that is zero outside the diagonal blocks.  CONVT3D_PREC_3XTF32 runs the
 * products on the tcgen05 tensor cores in split TF32 (a_hi*b_hi + a_hi*b_lo +
 * a_lo*b_hi, fp32 accumulation); CONVT3D_PREC_FFMA runs them as fp32 FMAs on
 * the CUDA cores (kept as an ablation).
 *
 * Conventions for every entry point:
 *   - Layouts: x [N,Cin,Din,Hin,Win], y [N,Cout,Do,Ho,Wo] (BN+pool: [N,Cout,1,1,1]),
 *     or channels-last x [N,Din,Hin,Win,Cin], y [N,Do,Ho,Wo,Cout] (desc.channels_last),
 *     w [Cin,Cout/G,kd,kh,kw] (PyTorch ConvTranspose3d), bias/gamma/beta [Cout];
 *     fp32 (x, w and y bf16 with desc.io_bf16, fp16 with desc.io_fp16), contiguous, device memory,
 *     16-byte aligned.
 *   - Ownership: the caller allocates and owns every device buffer (input,
 *     output, workspace).  The library never allocates or frees device memory
 *     and never synchronises a stream except in convt3d_check and
 *     convt3d_profile_read.  A plan owns host metadata only.
 *   - Streams: `stream` is a cudaStream_t (NULL = legacy default stream); all
 *     device work of a call is issued on it, in order.
 *   - Errors: a status code is returned, never an exception.  Arguments and
 *     shapes are validated on the host before anything is launched; nothing is
 *     launched when validation fails.  A failed launch returns
 *     CONVT3D_ERR_CUDA (convt3d_last_error gives the CUDA message).  Device-side
 *     conditions (a bounded wait that ran out) are recorded in the workspace
 *     and reported by convt3d_check.
 *   - y must not alias x.  Results are bitwise reproducible run to run (no
 *     floating-point atomics).
 *   - A plan caches launch state (encoded TMA descriptors keyed by the
 *     workspace address); do not call one plan from several host threads at
 *     once.  Different plans are independent.
 */
#ifndef CONVT3D_H
#define CONVT3D_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CONVT3D_EPI_IDENTITY = 0,
    CONVT3D_EPI_RELU_GROUPNORM = 1,
    CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL = 2,
    CONVT3D_EPI_SOFTMAX_SIGMOID = 3,
    CONVT3D_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL = 4
} convt3d_epilogue_t;

typedef enum {
    CONVT3D_PREC_3XTF32 = 0, /* tcgen05 tensor cores, split TF32 (default)             */
    CONVT3D_PREC_FFMA = 1,   /* CUDA-core fp32 FMA implicit GEMM (ablation)            */
    CONVT3D_PREC_TF32 = 2,   /* tcgen05 tensor cores, one TF32 product per term: inputs
                                rounded to TF32 (nearest), fp32 accumulation; results
                                within the 1e-2 tier of page l2_p49's harness quote */
    CONVT3D_PREC_BF16 = 3,   /* tcgen05 tensor cores, one BF16 product per term (kind::f16):
                                inputs rounded to bf16 (nearest even) when staged and
                                packed, fp32 accumulation and epilogue, fp32 I/O;
                                same 1e-2 tier                                        */
    CONVT3D_PREC_3XBF16 = 4, /* tcgen05 tensor cores, split BF16: each operand is
                                hi = bf16(v) + lo = bf16(v - hi) (nearest even, so
                                |v - hi - lo| <= 2^-16 |v|), three kind::f16 products
                                a_hi*b_hi + a_hi*b_lo + a_lo*b_hi per term, fp32
                                accumulation; fp32 I/O; the 1e-4 tier of 3XTF32 at
                                half its tensor-core time                              */
    CONVT3D_PREC_FP16 = 5    /* tcgen05 tensor cores, one FP16 product per term (kind::f16
                                with fp16 operands): inputs rounded to fp16 (nearest
                                even) when staged and packed, fp32 accumulation and
                                epilogue; the 1e-2 tier of page l2_p49's harness quote */
} convt3d_precision_t;

typedef enum {
    CONVT3D_OK = 0,
    CONVT3D_ERR_INVALID_ARG = 1,   /* NULL pointer, bad size, misaligned buffer       */
    CONVT3D_ERR_UNSUPPORTED = 2,   /* valid operation outside what this build runs    */
    CONVT3D_ERR_WORKSPACE = 3,     /* workspace NULL or smaller than workspace_bytes  */
    CONVT3D_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed                */
    CONVT3D_ERR_TIMEOUT = 5,       /* a device-side bounded wait ran out (check only)  */
    CONVT3D_ERR_DEVICE_ASSERT = 6, /* a device-side consistency check failed           */
    CONVT3D_ERR_NOT_PACKED = 7     /* forward before pack_weights on this workspace    */
} convt3d_status_t;

/* Problem description.  Enumerations are carried as int for a stable ABI. */
typedef struct {
    int N, Cin, Cout;     /* batch, input channels, output channels (>= 1)             */
    int Din, Hin, Win;    /* input extent (>= 1)                                        */
    int k;                /* cubic kernel size, 1..7                                    */
    int stride;           /* 1 or 2                                                     */
    int pad;              /* 0 <= pad <= dilation * (k - 1)                             */
    int out_pad;          /* 0 <= out_pad < max(stride, dilation)                       */
    int has_bias;         /* bias pointer is read iff non-zero                          */
    int epilogue;         /* convt3d_epilogue_t                                         */
    int groups;           /* GroupNorm groups; Cout % groups == 0 (RELU_GROUPNORM only) */
    float eps;            /* GroupNorm / BatchNorm epsilon (> 0)                        */
    float scale;          /* multiplier before BatchNorm (SCALE_BATCHNORM_AVGPOOL)      */
    int precision;        /* convt3d_precision_t                                        */
    /* General shapes (PyTorch ConvTranspose3d).  A zero-initialised tail gives
     * the cubic, undilated, dense case described by the fields above.        */
    int per_dim;          /* non-zero: kdims/strides/pads/out_pads replace k/stride/
                             pad/out_pad, index 0 = d, 1 = h, 2 = w               */
    int kdims[3];         /* kernel extent per dimension, 1..7                    */
    int strides[3];       /* 1 or 2 per dimension                                 */
    int pads[3];
    int out_pads[3];
    int dilation[3];      /* >= 1 per dimension; 0 means 1 (also without per_dim) */
    int conv_groups;      /* grouped convolution, Cin % G == Cout % G == 0; 0 = 1 */
    int channels_last;    /* non-zero: x is [N,Din,Hin,Win,Cin] and y [N,Do,Ho,Wo,Cout]
                             in memory (NDHWC); shapes are still reported as
                             [N,Cout,Do,Ho,Wo]; the pooled BN output is unchanged */
    int io_bf16;          /* non-zero: x, w and y are bf16 (2-byte) arrays; bias,
                             gamma, beta and the running statistics stay fp32;
                             requires precision CONVT3D_PREC_BF16                   */
    int io_fp16;          /* non-zero: x, w and y are fp16 (IEEE half) arrays, as
                             io_bf16 otherwise; requires precision CONVT3D_PREC_FP16 */
} convt3d_desc_t;

typedef struct convt3d_plan_s *convt3d_plan_t;

/* Plan facts, for callers that report or size things. */
typedef struct {
    int64_t out_shape[5];        /* y shape ([N,Cout,1,1,1] for the BN+pool epilogues)  */
    int num_classes;             /* output-parity classes (product of the strides)       */
    int64_t gemm_m;              /* output positions (N*Do*Ho*Wo)                        */
    int64_t gemm_n;              /* Cout                                                */
    int64_t gemm_k_total;        /* sum over classes of Cin * taps(class)                */
    int64_t tiles;               /* GEMM output tiles per forward                        */
    int tile_m;                  /* output positions per tile                            */
    int launches_per_forward;    /* kernels convt3d_forward launches                     */
    int launches_per_pack;       /* kernels convt3d_pack_weights launches                */
    double useful_flop;          /* 2*N*Cout*(Cin/G)*kd*kh*kw*Din*Hin*Win                */
    double issued_mma_flop;      /* tensor/FMA flop the main kernel issues per forward   */
    double gemm_min_bytes;       /* algorithmic HBM bytes of the main kernel             */
    double forward_min_bytes;    /* algorithmic HBM bytes of the whole forward           */
    int main_kernel;             /* 0: tensor-core GEMM on the staged channels-last copy
                                    of x; 1: FFMA kernel (requested, or the fallback for
                                    shapes the tensor-core loads cannot address: TMA
                                    im2col corners beyond [-16, 15]); 2: tensor-core GEMM
                                    reading NCDHW fp32 x itself, no staging pass (stride
                                    2 along w, Cin <= 32, Cout <= 64, BF16, 3XBF16 or FP16,
                                    identity or softmax+sigmoid, q-grid rows of 8..128
                                    positions dividing 128)                            */
} convt3d_info_t;

/* Validate `desc` and build a plan (host only: no CUDA call, no GPU needed).
 * Returns INVALID_ARG for malformed descriptions, UNSUPPORTED for valid ones
 * this build does not run (for example Cout > 512).  A tensor-core precision
 * whose loads cannot address the shape runs on the FFMA kernel instead
 * (convt3d_info_t.main_kernel).  *out is set to NULL on failure. */
convt3d_status_t convt3d_plan_create(const convt3d_desc_t *desc, convt3d_plan_t *out);

/* Release a plan (NULL is ignored). */
void convt3d_plan_destroy(convt3d_plan_t plan);

/* Output shape: [N,Cout,Do,Ho,Wo], or [N,Cout,1,1,1] for the BN+pool epilogues. Host only. */
convt3d_status_t convt3d_output_shape(convt3d_plan_t plan, int64_t shape[5]);

/* Plan facts (see convt3d_info_t). Host only. */
convt3d_status_t convt3d_plan_info(convt3d_plan_t plan, convt3d_info_t *info);

/* Bytes of device workspace the caller must provide to pack_weights and
 * forward (packed weights, the staged split input, statistics partials and a
 * status word).  0 on a NULL plan.  Host only. */
size_t convt3d_workspace_bytes(convt3d_plan_t plan);

/* Re-lay the weight w [Cin,Cout/G,kd,kh,kw] (G = conv_groups; [Cin,Cout,k,k,k]
 * in the cubic dense case) into the workspace: per parity class
 * and tap, Cout rows by Cin columns, split into TF32 hi and lo planes
 * (3XTF32) or kept fp32 (FFMA).  Call whenever w changes; forward reads only
 * the packed copy.  Also clears the workspace status word.  Asynchronous on
 * `stream`. */
convt3d_status_t convt3d_pack_weights(convt3d_plan_t plan, const void *w, void *workspace,
                                      size_t workspace_bytes, void *stream);

/* One forward pass: y = epilogue(convT(x, w) + bias).  bias may be NULL when
 * has_bias is 0; gamma/beta are required for RELU_GROUPNORM and
 * SCALE_BATCHNORM_AVGPOOL and ignored otherwise.  Uses the weights packed by
 * the last convt3d_pack_weights on the same workspace.  Asynchronous on
 * `stream`; y is complete when the stream reaches this point. */
convt3d_status_t convt3d_forward(convt3d_plan_t plan, const void *x, const float *bias,
                                 const float *gamma, const float *beta, void *y,
                                 void *workspace, size_t workspace_bytes, void *stream);

/* convt3d_forward in two parts, so that the main kernel can start on the first
 * samples of a batch while later ones are still being copied in.  No
 * counterpart on the pages: a scheduling convenience; the results are those
 * of convt3d_forward, bit for bit.
 *
 * convt3d_forward_samples runs the per-sample work for samples [n0, n1) of
 * the plan's batch: x and y are the WHOLE batch's tensors (sample n at its
 * usual offset), only samples n0..n1-1 of x are read and only those of y
 * (or of the per-tile statistics in the workspace) are written.  After calls
 * that together cover 0..N-1 once each, convt3d_forward_finish runs the passes
 * over the whole batch (GroupNorm's normalisation; BatchNorm's statistics,
 * pooled output and running-statistics update; nothing for IDENTITY and
 * SOFTMAX_SIGMOID) and y is then that of one convt3d_forward.  Ranges may go on
 * different streams when the caller orders each one before the finish call.
 * Errors: INVALID_ARG unless 0 <= n0 < n1 <= N, and as for convt3d_forward;
 * UNSUPPORTED for SCALE_BATCHNORM_EVAL_AVGPOOL (one pass over the batch) and,
 * unless [n0, n1) is the whole batch, for plans whose main kernel reads x
 * directly (convt3d_info_t.main_kernel 2).  gamma/beta as for convt3d_forward. */
convt3d_status_t convt3d_forward_samples(convt3d_plan_t plan, const void *x, const float *bias, void *y,
                                         void *workspace, size_t workspace_bytes, int n0, int n1,
                                         void *stream);
convt3d_status_t convt3d_forward_finish(convt3d_plan_t plan, const float *bias, const float *gamma,
                                        const float *beta, void *y, void *workspace, size_t workspace_bytes,
                                        void *stream);

/* BatchNorm running statistics, device pointers to Cout floats each (page
 * l2_p77: nn.BatchNorm3d with momentum 0.1, eps 1e-5).  With
 * SCALE_BATCHNORM_AVGPOOL, every later forward updates them in place from the
 * batch statistics: running_mean <- (1 - momentum) * running_mean + momentum *
 * mean, running_var likewise with the unbiased batch variance (n / (n - 1)
 * times the biased one, n = N * Do * Ho * Wo).  SCALE_BATCHNORM_EVAL_AVGPOOL
 * reads them and its forward fails with INVALID_ARG until they are set.  NULL
 * pointers clear the setting.  The plan keeps the pointers; the caller keeps
 * the memory valid.  Host only. */
convt3d_status_t convt3d_set_running_stats(convt3d_plan_t plan, float *running_mean, float *running_var,
                                           float momentum);

/* Synchronise `stream`, read and clear the workspace status word: returns OK,
 * TIMEOUT (a device-side bounded wait ran out) or DEVICE_ASSERT.  A NULL
 * workspace reads the built-in workspace of convt3d_forward_static_workspace
 * on the current device (the status of the last such call; the next call
 * clears it when it packs its weights). */
convt3d_status_t convt3d_check(convt3d_plan_t plan, void *workspace, void *stream);

/* Optional timing of the main GEMM kernel: when enabled, forward records two
 * CUDA events on `stream` around that launch; profile_read synchronises on
 * the second and returns the elapsed milliseconds of the last forward. */
convt3d_status_t convt3d_profile_enable(convt3d_plan_t plan, int enable);
convt3d_status_t convt3d_profile_read(convt3d_plan_t plan, float *gemm_ms);

/* A forward pass for callers that cannot provide a workspace, because they
 * are not allowed to allocate device memory (a plugin inside a host that owns
 * every device allocation) or cannot afford cudaMalloc's implicit device-wide
 * synchronisation.  No counterpart on the pages: this is a library
 * convenience, not part of the method.
 *
 * Packs w and runs the forward (the same kernels as convt3d_pack_weights +
 * convt3d_forward) using a 32 MiB workspace compiled into the library as a
 * device array; allocates nothing.  Each GPU that loads the library's device
 * code holds that array until the process exits.  Returns
 * CONVT3D_ERR_WORKSPACE, launching nothing, when convt3d_workspace_bytes(plan)
 * exceeds 32 MiB.  The first call on a device looks up the array's address
 * with that device current; make that first call outside any stream capture.
 * All calls share the one array: calls whose GPU work may overlap (other
 * streams, other threads) race on it and must be serialised by the caller.
 * Device-side conditions (a bounded wait that ran out) are recorded in the
 * array's status word: read them with convt3d_check(plan, NULL, stream) after
 * the call and before the next one, which clears the word.  The array's device
 * address is cached per device for the life of the process: do not call this
 * after cudaDeviceReset.  Arguments are as for convt3d_pack_weights and
 * convt3d_forward. */
convt3d_status_t convt3d_forward_static_workspace(convt3d_plan_t plan, const void *w, const void *x,
                                                  const float *bias, const float *gamma, const float *beta,
                                                  void *y, void *stream);

/* Static text for a status code. */
const char *convt3d_status_string(convt3d_status_t status);

/* Detail of the most recent failure in this thread (empty string if none). */
const char *convt3d_last_error(void);

/* Library version (major*10000 + minor*100 + patch). */
int convt3d_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CONVT3D_H */
