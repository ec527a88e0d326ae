// Statistics finalisation and the GroupNorm normalise pass.
//
// The GEMM epilogues leave statistics partials in fp64 in the workspace:
// partials[(n * T + t) * P + 3 * j + {0, 1, 2}] = (count, sum, M2) of group or
// channel j over partial row t of sample n (T rows per sample: one per tile, or
// one per epilogue warp of a tile), M2 being the sum of squared deviations from
// that row's own mean.  Rows combine by the pairwise update for the variance of
// a union of sets (Chan, Golub and LeVeque): with mean mu of the union,
// M2 = sum_t (M2_t + n_t (S_t / n_t - mu)^2), computed in two fixed-order passes
// (the sums, then the squared deviations), so results are bitwise reproducible
// and no one-pass E[v^2] - mean^2 cancellation arises however large the mean.
//
// GroupNorm (page l2_p61): per (n, g) mean and biased variance over
// Cout/G channels x all positions; GroupNorm's statistics span the whole
// sample, so a second pass rewrites y in place as (v - mean) * rstd * gamma
// + beta -- the page's own plan also needs two passes over global memory
// because a group does not fit in shared memory.  The GEMM leaves r = v - b in
// y (b the channel's bias), so the pass computes (r + (b - mean)) * rstd *
// gamma + beta with b - mean formed in fp64: no value of the bias's magnitude
// is rounded to fp32 (or to 16 bits) on the way.
// BatchNorm + pool (page l2_p77): per-channel batch mean/biased variance of
// z = scale*(conv + bias) over (n, positions); the pooled output is
// gamma * (S[n,c]/V - mean) * rstd + beta with S the per-sample spatial sum,
// the algebra the page derives for folding the average pool into the
// normalisation.
#include "convt3d_internal.h"

namespace convt3d {
namespace {

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One block per (n, g): 256 threads stride over the sample's partial rows,
// then a fixed-order tree reduction (fp64).
constexpr int kFinThreads = 256;

__device__ __forceinline__ void block_sum2(double &a, double &b, double (*red)[kFinThreads / 32]) {
    a = warp_sum(a);
    b = warp_sum(b);
    const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (lane == 0) {
        red[0][w] = a;
        red[1][w] = b;
    }
    __syncthreads();
    if (w == 0) {
        a = lane < kFinThreads / 32 ? red[0][lane] : 0.0;
        b = lane < kFinThreads / 32 ? red[1][lane] : 0.0;
        a = warp_sum(a);
        b = warp_sum(b);
    }
}

// The squared deviations of one partial row (count n, sum S, M2) from mean mu.
__device__ __forceinline__ double row_m2(const double *p, double mu) {
    if (p[0] <= 0.0) return 0.0;
    const double d = p[1] - p[0] * mu;
    return p[2] + d * d / p[0];
}

// A row's count (a non-negative whole number held as a double) read from its bits with
// integer operations, sparing the fp64 pipe (a small fraction of the fp32 rate on this
// GPU): the value for counts below 2^21, -1 above (the caller then uses the double).
__device__ __forceinline__ int row_count(double n) {
    const long long b = __double_as_longlong(n);
    if (b <= 0) return 0;  // +0.0: an empty row
    const int e = (int)(b >> 52) - 1023;
    if (e > 20) return -1;
    return (int)(((b & 0xFFFFFFFFFFFFFLL) | (1LL << 52)) >> (52 - e));
}

// As row_m2, dividing by the row's count through a table of reciprocals (counts
// above the table divide).
constexpr int kRcpTable = 129;
__device__ __forceinline__ double row_m2_rcp(const double *p, double mu, const double *rcp) {
    const double n = p[0];
    const int k = row_count(n);
    if (k == 0) return 0.0;
    const double d = fma(-n, mu, p[1]);  // S - n mu
    return k > 0 && k < kRcpTable ? fma(d * d, rcp[k], p[2]) : p[2] + d * d / n;
}

__global__ void __launch_bounds__(kFinThreads) gn_finalize_kernel(const double *__restrict__ partials,
                                                                  double *__restrict__ stats, int N, int G, int T,
                                                                  double eps) {
    __shared__ double red[2][kFinThreads / 32];
    __shared__ double s_mu;
    const int ng = blockIdx.x;
    const int n = ng / G, g = ng % G;
    const double *rows = partials + (int64_t)n * T * 3 * G + 3 * g;
    double cnt = 0.0, s1 = 0.0;
    for (int t = threadIdx.x; t < T; t += kFinThreads) {
        cnt += rows[(int64_t)t * 3 * G];
        s1 += rows[(int64_t)t * 3 * G + 1];
    }
    block_sum2(cnt, s1, red);
    if (threadIdx.x == 0) s_mu = cnt > 0.0 ? s1 / cnt : 0.0;
    __syncthreads();
    const double mu = s_mu;
    double m2 = 0.0, unused = 0.0;
    for (int t = threadIdx.x; t < T; t += kFinThreads) m2 += row_m2(rows + (int64_t)t * 3 * G, mu);
    __syncthreads();  // red is reused
    block_sum2(m2, unused, red);
    if (threadIdx.x == 0) {
        const double var = cnt > 0.0 ? m2 / cnt : 0.0;
        stats[2 * ng] = mu;
        stats[2 * ng + 1] = 1.0 / sqrt(var + eps);
    }
}

// Per (n, c): the scale a = rstd * gamma and the shift b - mean that the
// normalise pass applies to r = v - b.
__device__ __forceinline__ void gn_coeffs(const double *stats, const float *gamma, const float *bias, int n, int c,
                                          int C, int G, float &a, float &shift) {
    const int sg = n * G + c / (C / G);
    const double mean = stats[2 * sg], rstd = stats[2 * sg + 1];
    a = (float)(rstd * (double)gamma[c]);
    shift = (float)((bias ? (double)bias[c] : 0.0) - mean);
}

// y <- (y + shift[n,c]) * a[n,c] + beta[c].
// blockIdx.y is the (n, c) plane, blockIdx.x a chunk of it; each thread
// streams kVec float4s (16-byte loads and stores) when the plane is 16-byte
// aligned, scalars otherwise.
constexpr int kNormThreads = 256;
constexpr int kNormVec = 4;

__global__ void __launch_bounds__(kNormThreads) gn_normalize_kernel(float *__restrict__ y,
                                                                    const double *__restrict__ stats,
                                                                    const float *__restrict__ gamma,
                                                                    const float *__restrict__ beta,
                                                                    const float *__restrict__ bias, int C, int G,
                                                                    int64_t V, int planes) {
  for (int plane = blockIdx.y; plane < planes; plane += gridDim.y) {
    const int c = plane % C, n = plane / C;
    float a, sh;
    gn_coeffs(stats, gamma, bias, n, c, C, G, a, sh);
    const float b = beta[c];
    float *yp = y + (int64_t)plane * V;
    if ((V & 3) == 0) {
        float4 *y4 = reinterpret_cast<float4 *>(yp);
        const int64_t V4 = V >> 2;
        const int64_t base = (int64_t)blockIdx.x * kNormThreads * kNormVec + threadIdx.x;
        float4 v[kNormVec];
#pragma unroll
        for (int j = 0; j < kNormVec; ++j) {
            const int64_t i = base + (int64_t)j * kNormThreads;
            if (i < V4) v[j] = y4[i];
        }
#pragma unroll
        for (int j = 0; j < kNormVec; ++j) {
            const int64_t i = base + (int64_t)j * kNormThreads;
            if (i < V4) {
                v[j].x = fmaf(v[j].x + sh, a, b);
                v[j].y = fmaf(v[j].y + sh, a, b);
                v[j].z = fmaf(v[j].z + sh, a, b);
                v[j].w = fmaf(v[j].w + sh, a, b);
                y4[i] = v[j];
            }
        }
    } else {
        const int64_t base = (int64_t)blockIdx.x * kNormThreads * kNormVec * 4 + threadIdx.x;
        for (int j = 0; j < kNormVec * 4; ++j) {
            const int64_t i = base + (int64_t)j * kNormThreads;
            if (i < V) yp[i] = fmaf(yp[i] + sh, a, b);
        }
    }
  }
}

// Phase 1: per (n, c, row split) the (count, sum, M2) of a contiguous range
// of the sample's partial rows.  Block = 32 channels x 8 row lanes; grid
// (channel blocks, N, splits) -- the splits give the reduction enough blocks to
// fill the GPU.  Two passes: the range's mean, then the squared deviations.
__global__ void bn_reduce_kernel(const double *__restrict__ partials, double *__restrict__ sums, int N, int C,
                                 int T, int splits) {
    __shared__ double red[2][8][33];
    __shared__ double s_mu[32];
    // 1 / k for the rows' counts (at most one tile's rows, 128): this GPU's fp64 division is
    // slow, and a row's squared deviation needs one per (row, channel)
    __shared__ double s_rcp[kRcpTable];
    for (int i = threadIdx.y * 32 + threadIdx.x; i < kRcpTable; i += 256) s_rcp[i] = i > 0 ? 1.0 / i : 0.0;
    const int n = blockIdx.y, split = blockIdx.z;
    const int c = blockIdx.x * 32 + threadIdx.x;
    const int lane_t = threadIdx.y;
    const int t0 = (int)((int64_t)T * split / splits), t1 = (int)((int64_t)T * (split + 1) / splits);
    const double *rows = partials + (int64_t)n * T * 3 * C + 3 * c;
    long long cnt_i = 0;  // counts are whole numbers: summed exactly in integers
    double s1 = 0.0;
    if (c < C)
        for (int t = t0 + lane_t; t < t1; t += 8) {
            const double n = rows[(int64_t)t * 3 * C];
            const int k = row_count(n);
            cnt_i += k >= 0 ? (long long)k : (long long)n;
            s1 += rows[(int64_t)t * 3 * C + 1];
        }
    const double cnt = (double)cnt_i;
    red[0][lane_t][threadIdx.x] = cnt;
    red[1][lane_t][threadIdx.x] = s1;
    __syncthreads();
    if (lane_t == 0) {
        double a = 0.0, b = 0.0;
        for (int j = 0; j < 8; ++j) {
            a += red[0][j][threadIdx.x];
            b += red[1][j][threadIdx.x];
        }
        red[0][0][threadIdx.x] = a;
        red[1][0][threadIdx.x] = b;
        s_mu[threadIdx.x] = a > 0.0 ? b / a : 0.0;
    }
    __syncthreads();
    const double n_all = red[0][0][threadIdx.x], s_all = red[1][0][threadIdx.x], mu = s_mu[threadIdx.x];
    __syncthreads();  // red is reused
    double m2 = 0.0;
    if (c < C)
        for (int t = t0 + lane_t; t < t1; t += 8) m2 += row_m2_rcp(rows + (int64_t)t * 3 * C, mu, s_rcp);
    red[0][lane_t][threadIdx.x] = m2;
    __syncthreads();
    if (lane_t == 0 && c < C) {
        double a = 0.0;
        for (int j = 0; j < 8; ++j) a += red[0][j][threadIdx.x];
        double *o = sums + (((int64_t)n * splits + split) * C + c) * 3;
        o[0] = n_all;
        o[1] = s_all;
        o[2] = a;
    }
}

// Phase 2: per channel, batch mean and biased variance from the (count, sum,
// M2) of every (sample, split), then the pooled output from each sample's sum;
// optionally the running statistics' update (unbiased variance).  One warp per
// channel: lanes stride over the rows, butterfly sums in a fixed order.
constexpr int kBnFinWarps = 4;

__global__ void __launch_bounds__(32 * kBnFinWarps) bn_finalize_kernel(
    const double *__restrict__ sums, const float *__restrict__ gamma, const float *__restrict__ beta,
    float *__restrict__ y, int N, int C, int splits, double V, double eps, float *__restrict__ rmean,
    float *__restrict__ rvar, double momentum, int y16) {
    const int c = blockIdx.x * kBnFinWarps + threadIdx.x / 32, lane = threadIdx.x % 32;
    if (c >= C) return;  // whole warps leave together
    const int R = N * splits;
    double cnt = 0.0, S = 0.0;
    for (int r = lane; r < R; r += 32) {
        cnt += sums[((int64_t)r * C + c) * 3];
        S += sums[((int64_t)r * C + c) * 3 + 1];
    }
    cnt = warp_sum(cnt);
    S = warp_sum(S);
    const double mean = cnt > 0.0 ? S / cnt : 0.0;
    double m2 = 0.0;
    for (int r = lane; r < R; r += 32) m2 += row_m2(sums + ((int64_t)r * C + c) * 3, mean);
    m2 = warp_sum(m2);
    const double var = cnt > 0.0 ? m2 / cnt : 0.0;
    const double rstd = 1.0 / sqrt(var + eps);
    for (int n = lane; n < N; n += 32) {
        double Sn = 0.0;
        for (int k = 0; k < splits; ++k) Sn += sums[(((int64_t)n * splits + k) * C + c) * 3 + 1];
        const float out = (float)((double)gamma[c] * (Sn / V - mean) * rstd + (double)beta[c]);
        if (y16)  // 16-bit output of that kind
            reinterpret_cast<uint16_t *>(y)[(int64_t)n * C + c] = cvt16(out, y16);
        else
            y[(int64_t)n * C + c] = out;
    }
    if (lane == 0 && rmean && rvar) {
        const double unbiased = cnt > 1.0 ? var * cnt / (cnt - 1.0) : 0.0;
        rmean[c] = (float)((1.0 - momentum) * (double)rmean[c] + momentum * mean);
        rvar[c] = (float)((1.0 - momentum) * (double)rvar[c] + momentum * unbiased);
    }
}

// Channels-last variant: the per-channel scale and shift of one sample sit in
// shared memory; each thread rescales 4 consecutive elements of the sample's
// [V][C] block (128-bit when C % 4 == 0).  grid: (blocks over V*C, N).
__global__ void __launch_bounds__(kNormThreads) gn_normalize_cl_kernel(float *__restrict__ y,
                                                                       const double *__restrict__ stats,
                                                                       const float *__restrict__ gamma,
                                                                       const float *__restrict__ beta,
                                                                       const float *__restrict__ bias, int C, int G,
                                                                       int64_t V) {
    __shared__ float sa[kMaxCout], sh[kMaxCout], sb[kMaxCout];
    const int n = blockIdx.y;
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        gn_coeffs(stats, gamma, bias, n, c, C, G, sa[c], sh[c]);
        sb[c] = beta[c];
    }
    __syncthreads();
    float *yn = y + (int64_t)n * V * C;
    const int64_t total = V * C;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * 4;
    for (int64_t e = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; e < total; e += stride) {
        if ((C & 3) == 0) {  // e % 4 == 0, so the 4 elements share a row and start 16-byte aligned
            const int c = (int)(e % C);
            float4 v = *reinterpret_cast<float4 *>(yn + e);
            v.x = fmaf(v.x + sh[c], sa[c], sb[c]);
            v.y = fmaf(v.y + sh[c + 1], sa[c + 1], sb[c + 1]);
            v.z = fmaf(v.z + sh[c + 2], sa[c + 2], sb[c + 2]);
            v.w = fmaf(v.w + sh[c + 3], sa[c + 3], sb[c + 3]);
            *reinterpret_cast<float4 *>(yn + e) = v;
        } else {
            for (int64_t i = e; i < e + 4 && i < total; ++i) {
                const int c = (int)(i % C);
                yn[i] = fmaf(yn[i] + sh[c], sa[c], sb[c]);
            }
        }
    }
}

// 16-bit output (bf16 or fp16, `kind`), NCDHW: one (n, c) plane per
// blockIdx.y, pairs of elements (4-byte loads and stores) along the plane; an
// odd plane length leaves one last element for the x = 0 block.
__global__ void __launch_bounds__(kNormThreads) gn_normalize_16_kernel(uint16_t *__restrict__ y,
                                                                       const double *__restrict__ stats,
                                                                       const float *__restrict__ gamma,
                                                                       const float *__restrict__ beta,
                                                                       const float *__restrict__ bias, int C, int G,
                                                                       int64_t V, int planes, int kind) {
    for (int plane = blockIdx.y; plane < planes; plane += gridDim.y) {
        const int c = plane % C, n = plane / C;
        float a, sh;
        gn_coeffs(stats, gamma, bias, n, c, C, G, a, sh);
        const float b = beta[c];
        uint16_t *yp = y + (int64_t)plane * V;
        const bool even_base = ((int64_t)plane * V) % 2 == 0;  // 4-byte alignment of the pairs
        const int64_t first = even_base ? 0 : 1;
        if (!even_base && blockIdx.x == 0 && threadIdx.x == 0) yp[0] = cvt16(fmaf(ld16(yp, 0, kind) + sh, a, b), kind);
        const int64_t npairs = (V - first) / 2;
        uint32_t *y2 = reinterpret_cast<uint32_t *>(yp + first);
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < npairs;
             i += (int64_t)gridDim.x * blockDim.x) {
            const float2 v = ld16x2(y2[i], kind);
            y2[i] = cvt16x2(fmaf(v.x + sh, a, b), fmaf(v.y + sh, a, b), kind);
        }
        const int64_t last = first + 2 * npairs;
        if (last < V && blockIdx.x == 0 && threadIdx.x == 0)
            yp[last] = cvt16(fmaf(ld16(yp, last, kind) + sh, a, b), kind);
    }
}

// 16-bit output, channels-last: per-channel scale and shift of one sample in
// shared memory; each thread rescales element pairs (c, c+1) of the sample's
// [V][C] block, channel by invariant-divisor division (C even), else singly.
__global__ void __launch_bounds__(kNormThreads) gn_normalize_16_cl_kernel(uint16_t *__restrict__ y,
                                                                          const double *__restrict__ stats,
                                                                          const float *__restrict__ gamma,
                                                                          const float *__restrict__ beta,
                                                                          const float *__restrict__ bias, int C,
                                                                          int G, int64_t V, FastDiv divc, int kind) {
    __shared__ float sa[kMaxCout], sh[kMaxCout], sb[kMaxCout];
    const int n = blockIdx.y;
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        gn_coeffs(stats, gamma, bias, n, c, C, G, sa[c], sh[c]);
        sb[c] = beta[c];
    }
    __syncthreads();
    uint16_t *yn = y + (int64_t)n * V * C;
    const uint32_t total = (uint32_t)(V * C);  // < 2^31 elements per sample
    const uint32_t stride = gridDim.x * blockDim.x;
    if ((C & 1) == 0) {
        uint32_t *y2 = reinterpret_cast<uint32_t *>(yn);
        for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total / 2; i += stride) {
            const uint32_t e = 2 * i;
            const int c = (int)(e - fastdiv(e, divc) * (uint32_t)C);
            const float2 v = ld16x2(y2[i], kind);
            y2[i] = cvt16x2(fmaf(v.x + sh[c], sa[c], sb[c]), fmaf(v.y + sh[c + 1], sa[c + 1], sb[c + 1]), kind);
        }
    } else {
        for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
            const int c = (int)(e - fastdiv(e, divc) * (uint32_t)C);
            yn[e] = cvt16(fmaf(ld16(yn, e, kind) + sh[c], sa[c], sb[c]), kind);
        }
    }
}

}  // namespace

cudaError_t launch_gn_finalize(const convt3d_plan_s &p, const double *partials, double *stats, cudaStream_t s) {
    const int N = p.g.N, G = p.d.groups;
    gn_finalize_kernel<<<N * G, kFinThreads, 0, s>>>(partials, stats, N, G, p.tiles_per_sample * p.stat_rows_per_tile,
                                                     (double)p.d.eps);
    return cudaGetLastError();
}

cudaError_t launch_gn_normalize(const convt3d_plan_s &p, const double *stats, const float *gamma, const float *beta,
                                const float *bias, float *y, cudaStream_t s) {
    const int64_t V = (int64_t)p.g.Do * p.g.Ho * p.g.Wo;
    if (p.io16) {
        uint16_t *yh = reinterpret_cast<uint16_t *>(y);
        if (p.cl) {
            const int64_t want = (V * p.g.Cout / 2 + 8 * kNormThreads - 1) / (8 * kNormThreads);
            dim3 grid((unsigned)(want < 4096 ? (want > 0 ? want : 1) : 4096), (unsigned)p.g.N);
            gn_normalize_16_cl_kernel<<<grid, kNormThreads, 0, s>>>(yh, stats, gamma, beta, bias, p.g.Cout, p.d.groups, V,
                                                                     make_fastdiv((uint32_t)p.g.Cout), p.io16);
        } else {
            const int planes = p.g.N * p.g.Cout;
            const int64_t want = (V / 2 + 8 * kNormThreads - 1) / (8 * kNormThreads);  // ~8 pairs per thread
            dim3 grid((unsigned)(want < 1024 ? (want > 0 ? want : 1) : 1024), (unsigned)(planes < 65535 ? planes : 65535));
            gn_normalize_16_kernel<<<grid, kNormThreads, 0, s>>>(yh, stats, gamma, beta, bias, p.g.Cout, p.d.groups, V,
                                                                  planes, p.io16);
        }
        return cudaGetLastError();
    }
    if (p.cl) {
        const int64_t per_sample = V * p.g.Cout;
        const int64_t want = (per_sample / 4 + kNormThreads - 1) / kNormThreads;
        dim3 grid((unsigned)(want < 4096 ? (want > 0 ? want : 1) : 4096), (unsigned)p.g.N);
        gn_normalize_cl_kernel<<<grid, kNormThreads, 0, s>>>(y, stats, gamma, beta, bias, p.g.Cout, p.d.groups, V);
        return cudaGetLastError();
    }
    const int64_t per_block = (int64_t)kNormThreads * kNormVec * 4;  // floats per block
    const int planes = p.g.N * p.g.Cout;
    dim3 grid((unsigned)((V + per_block - 1) / per_block), (unsigned)(planes < 65535 ? planes : 65535));
    gn_normalize_kernel<<<grid, kNormThreads, 0, s>>>(y, stats, gamma, beta, bias, p.g.Cout, p.d.groups, V, planes);
    return cudaGetLastError();
}

cudaError_t launch_bn_finalize(const convt3d_plan_s &p, const double *partials, double *sums, const float *gamma,
                               const float *beta, float *y, cudaStream_t s) {
    const int N = p.g.N, C = p.g.Cout;
    dim3 grid((C + 31) / 32, N, p.bn_splits);
    bn_reduce_kernel<<<grid, dim3(32, 8), 0, s>>>(partials, sums, N, C, p.tiles_per_sample * p.stat_rows_per_tile,
                                                  p.bn_splits);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const double V = (double)p.g.Do * p.g.Ho * p.g.Wo;
    bn_finalize_kernel<<<(C + kBnFinWarps - 1) / kBnFinWarps, 32 * kBnFinWarps, 0, s>>>(
        sums, gamma, beta, y, N, C, p.bn_splits, V, (double)p.d.eps, p.run_mean, p.run_var, (double)p.momentum,
        p.io16);
    return cudaGetLastError();
}

}  // namespace convt3d
