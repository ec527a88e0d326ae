/*
 * convt3d oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU statement of what the GPU library
 * computes: a dense 3-D transposed convolution in its scatter (adjoint) form,
 * accumulated in fp64, followed by one of five epilogues evaluated literally
 * in fp64 (identity, ReLU+GroupNorm, scale+BatchNorm with batch statistics
 * (optionally updating running statistics)+pool, softmax+sigmoid,
 * scale+BatchNorm in evaluation mode+pool).  Nothing in the product path may link, load or call this file; only
 * the test suite, the smoke check and the benchmark's CPU-baseline arm do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (three POPCORNBENCH agent transcripts, "Kimi-K2.6" pages):
 *   l2_p77  ConvTranspose3d(64->128,k=5) -> x2.0 -> BatchNorm3d -> AdaptiveAvgPool3d(1)
 *   l2_p61  ConvTranspose3d(64->128,k=3,bias=False) -> ReLU -> GroupNorm(8)
 *   l2_p49  ConvTranspose3d(32->64,k=3,s=2,p=1,op=1) -> Softmax(dim=1) -> Sigmoid
 *
 * Layouts (PyTorch conventions used by all three pages):
 *   x    [N, Cin, Din, Hin, Win]          fp32, contiguous (NCDHW)
 *   w    [Cin, Cout/G, kd, kh, kw]         fp32, contiguous (ConvTranspose3d weight;
 *                                          G = convolution groups, 1 on all three pages)
 *   bias [Cout] or NULL
 *   y    [N, Cout, Do, Ho, Wo]             (BN+pool epilogue: [N, Cout])
 *
 * Every function is pinned by tests that do not re-state its formula: the
 * worked 1-D examples and the stride-2 tap table printed on the pages, the
 * stride-1 flipped-kernel equivalence, the adjoint identity against an
 * independently written forward convolution, linearity, the pooled-sum closed
 * form, and the normalisation invariants of each epilogue.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_EPI_IDENTITY = 0, ORACLE_EPI_RELU_GROUPNORM = 1,
       ORACLE_EPI_SCALE_BATCHNORM_AVGPOOL = 2, ORACLE_EPI_SOFTMAX_SIGMOID = 3,
       ORACLE_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL = 4 };

/* Output extent of a transposed convolution along one dimension (dilation 1):
 * (in - 1) * stride - 2 * pad + k + out_pad.  Page l2_p49 states the general
 * form with output_padding in its shape analysis; page l2_p77 states the
 * stride-1 form (in + k - 1) when deriving [16,128,20,36,36]. */
long oracle_output_size(long in, long k, long stride, long pad, long out_pad) {
    return (in - 1) * stride - 2 * pad + k + out_pad;
}

/* The same with dilation (PyTorch's ConvTranspose3d; page l2_p61's shape
 * analysis writes the dilated form): (in - 1) * stride - 2 * pad
 * + dilation * (k - 1) + out_pad + 1. */
long oracle_output_size_dil(long in, long k, long stride, long pad, long out_pad, long dil) {
    return (in - 1) * stride - 2 * pad + dil * (k - 1) + out_pad + 1;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Scatter (adjoint) definition, page l2_p49's index derivation: every input
 * element x[n,ci,id,ih,iw] adds w[ci,co,kd,kh,kw]*x to the output element at
 * (id*s - p + kd, ih*s - p + kh, iw*s - p + kw); contributions that land
 * outside [0,Do)x[0,Ho)x[0,Wo) are dropped (that is how padding crops).  The
 * bias, when given, is added once to every output element.
 *
 * General form (PyTorch's ConvTranspose3d): per-dimension kernel extent k[],
 * stride s[], padding p[], output padding op[] and dilation dil[] (index 0 = d,
 * 1 = h, 2 = w), so tap kd lands at id*s[0] - p[0] + dil[0]*kd; with G groups
 * the input channels of group g = co / (Cout/G) are ci in [g*Cin/G, (g+1)*Cin/G)
 * and the weight is [Cin, Cout/G, k[0], k[1], k[2]].
 *
 * Y receives fp64 results, shape [N, Cout, Do, Ho, Wo].  Parallel over
 * (n, co): each thread owns one output channel volume, so there are no races.
 * Returns 0, or -1 on a bad argument. */
int oracle_convt3d_scatter_general(int N, int Cin, int Cout, int Din, int Hin, int Win,
                                   const int *kk, const int *ss, const int *pp, const int *opp,
                                   const int *dil, int G,
                                   const float *x, const float *w, const float *bias,
                                   double *Y) {
    if (N < 0 || Cin <= 0 || Cout <= 0 || G <= 0 || Cin % G || Cout % G) return -1;
    for (int a = 0; a < 3; ++a)
        if (kk[a] <= 0 || ss[a] <= 0 || pp[a] < 0 || opp[a] < 0 || dil[a] <= 0) return -1;
    const long Do = oracle_output_size_dil(Din, kk[0], ss[0], pp[0], opp[0], dil[0]);
    const long Ho = oracle_output_size_dil(Hin, kk[1], ss[1], pp[1], opp[1], dil[1]);
    const long Wo = oracle_output_size_dil(Win, kk[2], ss[2], pp[2], opp[2], dil[2]);
    if (Do <= 0 || Ho <= 0 || Wo <= 0) return -1;
    const long in_vol = (long)Din * Hin * Win;
    const long out_vol = Do * Ho * Wo;
    const long kvol = (long)kk[0] * kk[1] * kk[2];
    const long pairs = (long)N * Cout;
    const long Cin_g = Cin / G, Cout_g = Cout / G;

#pragma omp parallel for schedule(dynamic, 1)
    for (long pc = 0; pc < pairs; ++pc) {
        const long n = pc / Cout;
        const long co = pc % Cout;
        const long g = co / Cout_g, col = co % Cout_g;
        double *Yc = Y + (n * Cout + co) * out_vol;
        const double b = bias ? (double)bias[co] : 0.0;
        for (long o = 0; o < out_vol; ++o) Yc[o] = 0.0;
        for (long ci = g * Cin_g; ci < (g + 1) * Cin_g; ++ci) {
            const float *xc = x + (n * Cin + ci) * in_vol;
            const float *wc = w + (ci * Cout_g + col) * kvol;
            for (long id = 0; id < Din; ++id)
            for (long ih = 0; ih < Hin; ++ih)
            for (long iw = 0; iw < Win; ++iw) {
                const double xv = (double)xc[(id * Hin + ih) * Win + iw];
                for (long kd = 0; kd < kk[0]; ++kd) {
                    const long od = id * ss[0] - pp[0] + dil[0] * kd;
                    if (od < 0 || od >= Do) continue;
                    for (long kh = 0; kh < kk[1]; ++kh) {
                        const long oh = ih * ss[1] - pp[1] + dil[1] * kh;
                        if (oh < 0 || oh >= Ho) continue;
                        for (long kw = 0; kw < kk[2]; ++kw) {
                            const long ow = iw * ss[2] - pp[2] + dil[2] * kw;
                            if (ow < 0 || ow >= Wo) continue;
                            Yc[(od * Ho + oh) * Wo + ow] +=
                                xv * (double)wc[(kd * kk[1] + kh) * kk[2] + kw];
                        }
                    }
                }
            }
        }
        for (long o = 0; o < out_vol; ++o) Yc[o] += b;
    }
    return 0;
}

/* The cubic, dense, undilated case (all three pages). */
int oracle_convt3d_scatter(int N, int Cin, int Cout, int Din, int Hin, int Win,
                           int k, int s, int p, int op,
                           const float *x, const float *w, const float *bias,
                           double *Y) {
    const int kk[3] = {k, k, k}, ss[3] = {s, s, s}, pp[3] = {p, p, p}, opp[3] = {op, op, op};
    const int dil[3] = {1, 1, 1};
    return oracle_convt3d_scatter_general(N, Cin, Cout, Din, Hin, Win, kk, ss, pp, opp, dil, 1, x, w, bias, Y);
}

/* Products visited by the scatter loop nest, split into those that land in
 * the output and those cropped by padding.  Both factor per dimension, so
 * this walks (i, k) pairs of one dimension at a time.  Page l2_p49 prints
 * the total for its workload (N*Cout*Cin*27*Din*Hin*Win). */
void oracle_count_products(int N, int Cin, int Cout, int Din, int Hin, int Win,
                           int k, int s, int p, int op,
                           double *in_range, double *total) {
    const int dims[3] = {Din, Hin, Win};
    double in_r = (double)N * Cin * Cout, tot = (double)N * Cin * Cout;
    for (int d = 0; d < 3; ++d) {
        const long out = oracle_output_size(dims[d], k, s, p, op);
        long hit = 0;
        for (long i = 0; i < dims[d]; ++i)
            for (long t = 0; t < k; ++t) {
                const long o = i * s - p + t;
                if (o >= 0 && o < out) ++hit;
            }
        in_r *= (double)hit;
        tot *= (double)dims[d] * k;
    }
    *in_range = in_r;
    *total = tot;
}

/* ReLU then GroupNorm (page l2_p61): v = max(Y, 0); for each (n, group g)
 * over its Cout/G channels and all output positions, mean and biased
 * ("population") variance, both in two passes; then
 * out = (v - mean) / sqrt(var + eps) * gamma[c] + beta[c]. */
static void epi_relu_groupnorm(int N, int C, long vol, int G, double eps,
                               const float *gamma, const float *beta,
                               double *Y) {
    const int cpg = C / G;
    const long cnt = (long)cpg * vol;
#pragma omp parallel for schedule(dynamic, 1)
    for (long ng = 0; ng < (long)N * G; ++ng) {
        const long n = ng / G, g = ng % G;
        double *base = Y + (n * C + g * cpg) * vol;
        for (long e = 0; e < cnt; ++e) base[e] = base[e] > 0.0 ? base[e] : 0.0;
        double sum = 0.0;
        for (long e = 0; e < cnt; ++e) sum += base[e];
        const double mean = sum / (double)cnt;
        double ss = 0.0;
        for (long e = 0; e < cnt; ++e) { const double d = base[e] - mean; ss += d * d; }
        const double var = ss / (double)cnt;
        const double inv = 1.0 / sqrt(var + eps);
        for (int cl = 0; cl < cpg; ++cl) {
            const long c = g * cpg + cl;
            const double ga = gamma ? (double)gamma[c] : 1.0;
            const double be = beta ? (double)beta[c] : 0.0;
            double *row = base + (long)cl * vol;
            for (long o = 0; o < vol; ++o) row[o] = (row[o] - mean) * inv * ga + be;
        }
    }
}

/* Channel softmax then elementwise sigmoid (page l2_p49): per (n, position)
 * m = max_c Y, e_c = exp(Y_c - m), S = sum_c e_c, out_c = 1 / (1 + exp(-e_c / S)). */
static void epi_softmax_sigmoid(int N, int C, long vol, double *Y) {
#pragma omp parallel for schedule(static)
    for (long np = 0; np < (long)N * vol; ++np) {
        const long n = np / vol, o = np % vol;
        double *col = Y + n * C * vol + o;
        double m = col[0];
        for (int c = 1; c < C; ++c) if (col[(long)c * vol] > m) m = col[(long)c * vol];
        double S = 0.0;
        for (int c = 0; c < C; ++c) S += exp(col[(long)c * vol] - m);
        for (int c = 0; c < C; ++c) {
            const double t = exp(col[(long)c * vol] - m) / S;
            col[(long)c * vol] = 1.0 / (1.0 + exp(-t));
        }
    }
}

/* Multiply by scale, BatchNorm3d with batch statistics, AdaptiveAvgPool3d(1)
 * (page l2_p77): z = scale * Y; per channel c over (n, positions) the mean and
 * the biased variance (two passes); every element normalised
 * (z - mean) / sqrt(var + eps) * gamma + beta; then the spatial mean per (n, c).
 * Written element by element so that the algebraic shortcut the page derives
 * is an independent check, not a restatement.  out is [N, C]. */
static void epi_scale_bn_avgpool(int N, int C, long vol, double scale, double eps,
                                 const float *gamma, const float *beta,
                                 const double *Y, double *out) {
    const double cnt = (double)N * (double)vol;
#pragma omp parallel for schedule(dynamic, 1)
    for (long c = 0; c < C; ++c) {
        double sum = 0.0;
        for (long n = 0; n < N; ++n) {
            const double *row = Y + (n * C + c) * vol;
            for (long o = 0; o < vol; ++o) sum += scale * row[o];
        }
        const double mean = sum / cnt;
        double ss = 0.0;
        for (long n = 0; n < N; ++n) {
            const double *row = Y + (n * C + c) * vol;
            for (long o = 0; o < vol; ++o) { const double d = scale * row[o] - mean; ss += d * d; }
        }
        const double var = ss / cnt;
        const double inv = 1.0 / sqrt(var + eps);
        const double ga = gamma ? (double)gamma[c] : 1.0;
        const double be = beta ? (double)beta[c] : 0.0;
        for (long n = 0; n < N; ++n) {
            const double *row = Y + (n * C + c) * vol;
            double acc = 0.0;
            for (long o = 0; o < vol; ++o) acc += (scale * row[o] - mean) * inv * ga + be;
            out[n * C + c] = acc / (double)vol;
        }
    }
}

/* Multiply by scale, BatchNorm3d in evaluation mode, AdaptiveAvgPool3d(1)
 * (page l2_p77's submitted solution assumes evaluation mode): each element is
 * normalised with the stored running statistics,
 * (z - running_mean[c]) / sqrt(running_var[c] + eps) * gamma + beta, then the
 * spatial mean per (n, c).  Written element by element.  out is [N, C]. */
static void epi_scale_bn_eval_avgpool(int N, int C, long vol, double scale, double eps,
                                      const float *gamma, const float *beta,
                                      const float *rmean, const float *rvar,
                                      const double *Y, double *out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (long nc = 0; nc < (long)N * C; ++nc) {
        const long c = nc % C;
        const double inv = 1.0 / sqrt((double)rvar[c] + eps);
        const double ga = gamma ? (double)gamma[c] : 1.0;
        const double be = beta ? (double)beta[c] : 0.0;
        const double *row = Y + nc * vol;
        double acc = 0.0;
        for (long o = 0; o < vol; ++o) acc += (scale * row[o] - (double)rmean[c]) * inv * ga + be;
        out[nc] = acc / (double)vol;
    }
}

/* BatchNorm3d's running-statistics update in training mode (page l2_p77,
 * "momentum=0.1"): with the batch mean and the biased batch variance of
 * z = scale * Y over the n = N * vol elements of each channel,
 * running_mean <- (1 - m) * running_mean + m * mean and
 * running_var  <- (1 - m) * running_var  + m * var * n / (n - 1). */
static void bn_update_running(int N, int C, long vol, double scale, double momentum, const double *Y,
                              float *rmean, float *rvar) {
    const double cnt = (double)N * (double)vol;
#pragma omp parallel for schedule(dynamic, 1)
    for (long c = 0; c < C; ++c) {
        double sum = 0.0;
        for (long n = 0; n < N; ++n)
            for (long o = 0; o < vol; ++o) sum += scale * Y[(n * C + c) * vol + o];
        const double mean = sum / cnt;
        double ss = 0.0;
        for (long n = 0; n < N; ++n)
            for (long o = 0; o < vol; ++o) {
                const double d = scale * Y[(n * C + c) * vol + o] - mean;
                ss += d * d;
            }
        const double var_unbiased = cnt > 1.0 ? ss / (cnt - 1.0) : 0.0;
        rmean[c] = (float)((1.0 - momentum) * (double)rmean[c] + momentum * mean);
        rvar[c] = (float)((1.0 - momentum) * (double)rvar[c] + momentum * var_unbiased);
    }
}

/* Full forward: scatter-form transposed convolution (+bias), then the
 * epilogue, all in fp64; results are rounded once to fp32 (round to nearest
 * even) into y.  If y64 is not NULL the fp64 results are also written there.
 * For the BN+pool epilogues y / y64 hold [N, Cout]; otherwise
 * [N, Cout, Do, Ho, Wo].  running_mean / running_var: read by the
 * evaluation-mode epilogue; updated in place by the batch-statistics epilogue
 * when both are given (NULL skips the update).  Shape arguments as in
 * oracle_convt3d_scatter_general.  Returns 0, -1 on a bad argument, -2 if out
 * of memory. */
int oracle_convt3d_forward_general(int N, int Cin, int Cout, int Din, int Hin, int Win,
                                   const int *kk, const int *ss, const int *pp, const int *opp,
                                   const int *dil, int conv_groups,
                                   const float *x, const float *w, const float *bias,
                                   int epilogue, int groups, double eps, double scale,
                                   const float *gamma, const float *beta,
                                   float *running_mean, float *running_var, double momentum,
                                   float *y, double *y64) {
    const long Do = oracle_output_size_dil(Din, kk[0], ss[0], pp[0], opp[0], dil[0]);
    const long Ho = oracle_output_size_dil(Hin, kk[1], ss[1], pp[1], opp[1], dil[1]);
    const long Wo = oracle_output_size_dil(Win, kk[2], ss[2], pp[2], opp[2], dil[2]);
    if (N <= 0 || Do <= 0 || Ho <= 0 || Wo <= 0) return -1;
    if (epilogue == ORACLE_EPI_RELU_GROUPNORM && (groups <= 0 || Cout % groups)) return -1;
    if (epilogue < 0 || epilogue > 4) return -1;
    if (epilogue == ORACLE_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL && (!running_mean || !running_var)) return -1;
    const long vol = Do * Ho * Wo;
    const long total = (long)N * Cout * vol;
    double *Y = (double *)malloc(sizeof(double) * (size_t)total);
    if (!Y) return -2;
    int rc = oracle_convt3d_scatter_general(N, Cin, Cout, Din, Hin, Win, kk, ss, pp, opp, dil, conv_groups, x, w,
                                            bias, Y);
    if (rc) { free(Y); return rc; }
    if (epilogue == ORACLE_EPI_SCALE_BATCHNORM_AVGPOOL || epilogue == ORACLE_EPI_SCALE_BATCHNORM_EVAL_AVGPOOL) {
        double *pooled = (double *)malloc(sizeof(double) * (size_t)N * Cout);
        if (!pooled) { free(Y); return -2; }
        if (epilogue == ORACLE_EPI_SCALE_BATCHNORM_AVGPOOL) {
            epi_scale_bn_avgpool(N, Cout, vol, scale, eps, gamma, beta, Y, pooled);
            if (running_mean && running_var)
                bn_update_running(N, Cout, vol, scale, momentum, Y, running_mean, running_var);
        } else {
            epi_scale_bn_eval_avgpool(N, Cout, vol, scale, eps, gamma, beta, running_mean, running_var, Y,
                                      pooled);
        }
        for (long i = 0; i < (long)N * Cout; ++i) {
            y[i] = (float)pooled[i];
            if (y64) y64[i] = pooled[i];
        }
        free(pooled);
        free(Y);
        return 0;
    }
    if (epilogue == ORACLE_EPI_RELU_GROUPNORM)
        epi_relu_groupnorm(N, Cout, vol, groups, eps, gamma, beta, Y);
    else if (epilogue == ORACLE_EPI_SOFTMAX_SIGMOID)
        epi_softmax_sigmoid(N, Cout, vol, Y);
#pragma omp parallel for schedule(static)
    for (long i = 0; i < total; ++i) {
        y[i] = (float)Y[i];
        if (y64) y64[i] = Y[i];
    }
    free(Y);
    return 0;
}

/* The cubic, dense, undilated case (all three pages). */
int oracle_convt3d_forward(int N, int Cin, int Cout, int Din, int Hin, int Win,
                           int k, int s, int p, int op,
                           const float *x, const float *w, const float *bias,
                           int epilogue, int groups, double eps, double scale,
                           const float *gamma, const float *beta,
                           float *running_mean, float *running_var, double momentum,
                           float *y, double *y64) {
    const int kk[3] = {k, k, k}, ss[3] = {s, s, s}, pp[3] = {p, p, p}, opp[3] = {op, op, op};
    const int dil[3] = {1, 1, 1};
    return oracle_convt3d_forward_general(N, Cin, Cout, Din, Hin, Win, kk, ss, pp, opp, dil, 1, x, w, bias,
                                          epilogue, groups, eps, scale, gamma, beta, running_mean, running_var,
                                          momentum, y, y64);
}
