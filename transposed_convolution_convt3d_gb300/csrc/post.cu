// Statistics finalisation and the GroupNorm normalise pass.
//
// The GEMM epilogues leave partial (sum, sum of squares) in fp64 in the
// workspace: partials[(n * T + t) * P + j], T partial rows per sample (one per
// tile, or one per epilogue warp of a tile), P values per row.  Reductions here run in a fixed order (no atomics), so results
// are bitwise reproducible.
//
// GroupNorm (page l2_p61): per (n, g) mean and biased variance over
// Cout/G channels x all positions; GroupNorm's statistics span the whole
// sample, so a second pass rewrites y in place as (v - mean) * rstd * gamma
// + beta -- the page's own plan also needs two passes over global memory
// because a group does not fit in shared memory.
// BatchNorm + pool (page l2_p77): per-channel batch mean/biased variance of
// z = scale*(conv + bias) over (n, positions); the pooled output is
// gamma * (S[n,c]/V - mean) * rstd + beta with S the per-sample spatial sum,
// the algebra the page derives for folding the average pool into the
// normalisation.
#include <cuda_bf16.h>

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

__global__ void __launch_bounds__(kFinThreads) gn_finalize_kernel(const double *__restrict__ partials,
                                                                  double *__restrict__ stats, int N, int G, int T,
                                                                  double count, double eps) {
    __shared__ double red[2][kFinThreads / 32];
    const int ng = blockIdx.x;
    const int n = ng / G, g = ng % G;
    double s1 = 0.0, s2 = 0.0;
    for (int t = threadIdx.x; t < T; t += kFinThreads) {
        const double *p = partials + ((int64_t)n * T + t) * 2 * G + 2 * g;
        s1 += p[0];
        s2 += p[1];
    }
    block_sum2(s1, s2, red);
    if (threadIdx.x == 0) {
        const double mean = s1 / count;
        double var = s2 / count - mean * mean;
        var = var > 0.0 ? var : 0.0;
        stats[2 * ng] = mean;
        stats[2 * ng + 1] = 1.0 / sqrt(var + eps);
    }
}

// y <- y * a[n,c] + b[n,c] with a = rstd*gamma, b = beta - mean*rstd*gamma.
// blockIdx.y is the (n, c) plane, blockIdx.x a chunk of it; each thread
// streams kVec float4s (16-byte loads and stores) when the plane is 16-byte
// aligned, scalars otherwise.
constexpr int kNormThreads = 256;
constexpr int kNormVec = 4;

__global__ void __launch_bounds__(kNormThreads) gn_normalize_kernel(float *__restrict__ y,
                                                                    const double *__restrict__ stats,
                                                                    const float *__restrict__ gamma,
                                                                    const float *__restrict__ beta, int C, int G,
                                                                    int64_t V, int planes) {
  for (int plane = blockIdx.y; plane < planes; plane += gridDim.y) {
    const int c = plane % C, n = plane / C;
    const int sg = n * G + c / (C / G);
    const double rstd = stats[2 * sg + 1], mean = stats[2 * sg];
    const float a = (float)(rstd * gamma[c]);
    const float b = (float)(beta[c] - mean * rstd * gamma[c]);
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
                v[j].x = fmaf(v[j].x, a, b);
                v[j].y = fmaf(v[j].y, a, b);
                v[j].z = fmaf(v[j].z, a, b);
                v[j].w = fmaf(v[j].w, a, b);
                y4[i] = v[j];
            }
        }
    } else {
        const int64_t base = (int64_t)blockIdx.x * kNormThreads * kNormVec * 4 + threadIdx.x;
        for (int j = 0; j < kNormVec * 4; ++j) {
            const int64_t i = base + (int64_t)j * kNormThreads;
            if (i < V) yp[i] = fmaf(yp[i], a, b);
        }
    }
  }
}

// Phase 1: per (n, c) the spatial sum S and the sum of squares over the
// sample's partial rows.  Block = 32 channels x 8 row lanes of one sample.
__global__ void bn_reduce_kernel(const double *__restrict__ partials, double *__restrict__ sums, int N, int C,
                                 int T) {
    __shared__ double red[2][8][33];
    const int n = blockIdx.y;
    const int c = blockIdx.x * 32 + threadIdx.x;
    const int lane_t = threadIdx.y;
    double s1 = 0.0, s2 = 0.0;
    if (c < C) {
        for (int t = lane_t; t < T; t += 8) {
            const double *p = partials + ((int64_t)n * T + t) * 2 * C + 2 * c;
            s1 += p[0];
            s2 += p[1];
        }
    }
    red[0][lane_t][threadIdx.x] = s1;
    red[1][lane_t][threadIdx.x] = s2;
    __syncthreads();
    if (lane_t == 0 && c < C) {
        double a = 0.0, b = 0.0;
        for (int j = 0; j < 8; ++j) {
            a += red[0][j][threadIdx.x];
            b += red[1][j][threadIdx.x];
        }
        sums[((int64_t)n * C + c) * 2] = a;
        sums[((int64_t)n * C + c) * 2 + 1] = b;
    }
}

// Phase 2: per channel, batch mean and biased variance, then the pooled output;
// optionally the running statistics' update (unbiased variance).
__global__ void bn_finalize_kernel(const double *__restrict__ sums, const float *__restrict__ gamma,
                                   const float *__restrict__ beta, float *__restrict__ y, int N, int C, double V,
                                   double eps, float *__restrict__ rmean, float *__restrict__ rvar,
                                   double momentum, int y16) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= C) return;
    double S = 0.0, Q = 0.0;
    for (int n = 0; n < N; ++n) {
        S += sums[((int64_t)n * C + c) * 2];
        Q += sums[((int64_t)n * C + c) * 2 + 1];
    }
    const double cnt = (double)N * V;
    const double mean = S / cnt;
    double var = Q / cnt - mean * mean;
    var = var > 0.0 ? var : 0.0;
    const double rstd = 1.0 / sqrt(var + eps);
    for (int n = 0; n < N; ++n) {
        const double Sn = sums[((int64_t)n * C + c) * 2];
        const float out = (float)((double)gamma[c] * (Sn / V - mean) * rstd + (double)beta[c]);
        if (y16)
            reinterpret_cast<__nv_bfloat16 *>(y)[(int64_t)n * C + c] = __float2bfloat16_rn(out);
        else
            y[(int64_t)n * C + c] = out;
    }
    if (rmean && rvar) {
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
                                                                       const float *__restrict__ beta, int C, int G,
                                                                       int64_t V) {
    __shared__ float sa[256], sb[256];
    const int n = blockIdx.y;
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        const int sg = n * G + c / (C / G);
        const double rstd = stats[2 * sg + 1], mean = stats[2 * sg];
        sa[c] = (float)(rstd * gamma[c]);
        sb[c] = (float)(beta[c] - mean * rstd * gamma[c]);
    }
    __syncthreads();
    float *yn = y + (int64_t)n * V * C;
    const int64_t total = V * C;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * 4;
    for (int64_t e = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; e < total; e += stride) {
        if ((C & 3) == 0) {  // e % 4 == 0, so the 4 elements share a row and start 16-byte aligned
            const int c = (int)(e % C);
            float4 v = *reinterpret_cast<float4 *>(yn + e);
            v.x = fmaf(v.x, sa[c], sb[c]);
            v.y = fmaf(v.y, sa[c + 1], sb[c + 1]);
            v.z = fmaf(v.z, sa[c + 2], sb[c + 2]);
            v.w = fmaf(v.w, sa[c + 3], sb[c + 3]);
            *reinterpret_cast<float4 *>(yn + e) = v;
        } else {
            for (int64_t i = e; i < e + 4 && i < total; ++i) {
                const int c = (int)(i % C);
                yn[i] = fmaf(yn[i], sa[c], sb[c]);
            }
        }
    }
}

// bf16 output, NCDHW: one (n, c) plane per blockIdx.y, pairs of elements
// (4-byte bf16x2 loads and stores) along the plane; an odd plane length leaves
// one last element for the x = 0 block.
__global__ void __launch_bounds__(kNormThreads) gn_normalize_bf16_kernel(__nv_bfloat16 *__restrict__ y,
                                                                         const double *__restrict__ stats,
                                                                         const float *__restrict__ gamma,
                                                                         const float *__restrict__ beta, int C, int G,
                                                                         int64_t V, int planes) {
    for (int plane = blockIdx.y; plane < planes; plane += gridDim.y) {
        const int c = plane % C, n = plane / C;
        const int sg = n * G + c / (C / G);
        const double rstd = stats[2 * sg + 1], mean = stats[2 * sg];
        const float a = (float)(rstd * gamma[c]);
        const float b = (float)(beta[c] - mean * rstd * gamma[c]);
        __nv_bfloat16 *yp = y + (int64_t)plane * V;
        const bool even_base = ((int64_t)plane * V) % 2 == 0;  // 4-byte alignment of the pairs
        const int64_t first = even_base ? 0 : 1;
        if (!even_base && blockIdx.x == 0 && threadIdx.x == 0)
            yp[0] = __float2bfloat16_rn(fmaf(__bfloat162float(yp[0]), a, b));
        const int64_t npairs = (V - first) / 2;
        __nv_bfloat162 *y2 = reinterpret_cast<__nv_bfloat162 *>(yp + first);
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < npairs;
             i += (int64_t)gridDim.x * blockDim.x) {
            const float2 v = __bfloat1622float2(y2[i]);
            y2[i] = __floats2bfloat162_rn(fmaf(v.x, a, b), fmaf(v.y, a, b));
        }
        const int64_t last = first + 2 * npairs;
        if (last < V && blockIdx.x == 0 && threadIdx.x == 0)
            yp[last] = __float2bfloat16_rn(fmaf(__bfloat162float(yp[last]), a, b));
    }
}

// bf16 output, channels-last: per-channel scale and shift of one sample in
// shared memory; each thread rescales element pairs (c, c+1) of the sample's
// [V][C] block, channel by invariant-divisor division (C even), else singly.
__global__ void __launch_bounds__(kNormThreads) gn_normalize_bf16_cl_kernel(__nv_bfloat16 *__restrict__ y,
                                                                            const double *__restrict__ stats,
                                                                            const float *__restrict__ gamma,
                                                                            const float *__restrict__ beta, int C,
                                                                            int G, int64_t V, FastDiv divc) {
    __shared__ float sa[256], sb[256];
    const int n = blockIdx.y;
    for (int c = threadIdx.x; c < C; c += blockDim.x) {
        const int sg = n * G + c / (C / G);
        const double rstd = stats[2 * sg + 1], mean = stats[2 * sg];
        sa[c] = (float)(rstd * gamma[c]);
        sb[c] = (float)(beta[c] - mean * rstd * gamma[c]);
    }
    __syncthreads();
    __nv_bfloat16 *yn = y + (int64_t)n * V * C;
    const uint32_t total = (uint32_t)(V * C);  // < 2^31 elements per sample
    const uint32_t stride = gridDim.x * blockDim.x;
    if ((C & 1) == 0) {
        __nv_bfloat162 *y2 = reinterpret_cast<__nv_bfloat162 *>(yn);
        for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total / 2; i += stride) {
            const uint32_t e = 2 * i;
            const int c = (int)(e - fastdiv(e, divc) * (uint32_t)C);
            const float2 v = __bfloat1622float2(y2[i]);
            y2[i] = __floats2bfloat162_rn(fmaf(v.x, sa[c], sb[c]), fmaf(v.y, sa[c + 1], sb[c + 1]));
        }
    } else {
        for (uint32_t e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
            const int c = (int)(e - fastdiv(e, divc) * (uint32_t)C);
            yn[e] = __float2bfloat16_rn(fmaf(__bfloat162float(yn[e]), sa[c], sb[c]));
        }
    }
}

}  // namespace

cudaError_t launch_gn_finalize(const convt3d_plan_s &p, const double *partials, double *stats, cudaStream_t s) {
    const int N = p.g.N, G = p.d.groups;
    const double V = (double)p.g.Do * p.g.Ho * p.g.Wo;
    const double count = V * (p.g.Cout / G);
    gn_finalize_kernel<<<N * G, kFinThreads, 0, s>>>(partials, stats, N, G, p.tiles_per_sample * p.stat_rows_per_tile,
                                                     count, (double)p.d.eps);
    return cudaGetLastError();
}

cudaError_t launch_gn_normalize(const convt3d_plan_s &p, const double *stats, const float *gamma, const float *beta,
                                float *y, cudaStream_t s) {
    const int64_t V = (int64_t)p.g.Do * p.g.Ho * p.g.Wo;
    if (p.io16) {
        __nv_bfloat16 *yh = reinterpret_cast<__nv_bfloat16 *>(y);
        if (p.cl) {
            const int64_t want = (V * p.g.Cout / 2 + 8 * kNormThreads - 1) / (8 * kNormThreads);
            dim3 grid((unsigned)(want < 4096 ? (want > 0 ? want : 1) : 4096), (unsigned)p.g.N);
            gn_normalize_bf16_cl_kernel<<<grid, kNormThreads, 0, s>>>(yh, stats, gamma, beta, p.g.Cout, p.d.groups, V,
                                                                       make_fastdiv((uint32_t)p.g.Cout));
        } else {
            const int planes = p.g.N * p.g.Cout;
            const int64_t want = (V / 2 + 8 * kNormThreads - 1) / (8 * kNormThreads);  // ~8 pairs per thread
            dim3 grid((unsigned)(want < 1024 ? (want > 0 ? want : 1) : 1024), (unsigned)(planes < 65535 ? planes : 65535));
            gn_normalize_bf16_kernel<<<grid, kNormThreads, 0, s>>>(yh, stats, gamma, beta, p.g.Cout, p.d.groups, V,
                                                                    planes);
        }
        return cudaGetLastError();
    }
    if (p.cl) {
        const int64_t per_sample = V * p.g.Cout;
        const int64_t want = (per_sample / 4 + kNormThreads - 1) / kNormThreads;
        dim3 grid((unsigned)(want < 4096 ? (want > 0 ? want : 1) : 4096), (unsigned)p.g.N);
        gn_normalize_cl_kernel<<<grid, kNormThreads, 0, s>>>(y, stats, gamma, beta, p.g.Cout, p.d.groups, V);
        return cudaGetLastError();
    }
    const int64_t per_block = (int64_t)kNormThreads * kNormVec * 4;  // floats per block
    const int planes = p.g.N * p.g.Cout;
    dim3 grid((unsigned)((V + per_block - 1) / per_block), (unsigned)(planes < 65535 ? planes : 65535));
    gn_normalize_kernel<<<grid, kNormThreads, 0, s>>>(y, stats, gamma, beta, p.g.Cout, p.d.groups, V, planes);
    return cudaGetLastError();
}

cudaError_t launch_bn_finalize(const convt3d_plan_s &p, const double *partials, double *sums, const float *gamma,
                               const float *beta, float *y, cudaStream_t s) {
    const int N = p.g.N, C = p.g.Cout;
    dim3 grid((C + 31) / 32, N);
    bn_reduce_kernel<<<grid, dim3(32, 8), 0, s>>>(partials, sums, N, C, p.tiles_per_sample * p.stat_rows_per_tile);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const double V = (double)p.g.Do * p.g.Ho * p.g.Wo;
    bn_finalize_kernel<<<(C + 127) / 128, 128, 0, s>>>(sums, gamma, beta, y, N, C, V, (double)p.d.eps, p.run_mean,
                                                        p.run_var, (double)p.momentum, p.io16);
    return cudaGetLastError();
}

}  // namespace convt3d
