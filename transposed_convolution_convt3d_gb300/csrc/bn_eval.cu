// Scale + BatchNorm3d in evaluation mode + global average pool, without the
// convolution (page l2_p77's module run with stored running statistics).
//
// With fixed statistics the normalisation is an affine map per channel, so it
// commutes with the average over positions:
//   out[n,c] = gamma[c] * (scale * mean_pos(Y[n,c]) - rm[c]) / sqrt(rv[c] + eps) + beta[c].
// mean_pos(Y[n,c]) = b[c] + S[n,c] / V with V = Do*Ho*Wo and
//   S[n,c] = sum_{ci, tap} w[ci, c, tap] * B[n, ci, tap],
// where B is the sum of x[n, ci] over the input box whose scatter through that
// tap lands inside the output (ConvTranspose3d scatters input i through tap t
// to o = stride*i - pad + dilation*t per dimension).  Grouped convolution needs
// nothing more: the packed weight is zero between channels of different groups.  The box is a product of one
// interval per dimension, so B is three passes of 1-D interval sums:
//   boxsum_kernel    one block per (n, ci): x once along d into k accumulators
//                    per (h, w) column, then intervals along h (prefix sums,
//                    one difference per interval), then along w;
//   bn_eval_out_kernel  one block per (c, 16 samples): the Cin*k^3 contraction
//                    with the packed weight, then the formula above in fp64.
// The work is O(N*Cin*D*H*W*k + N*Cout*Cin*k^3), a read of x and of the weight.
#include <cuda_bf16.h>

#include "convt3d_internal.h"

namespace convt3d {
namespace {

constexpr int kMaxK = 7;

__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Inputs i whose output s*i - p + dil*t lies in [0, out - 1], clamped to [0, in - 1].
struct Interval {
    int lo, hi;
};

__device__ __forceinline__ Interval tap_interval(int t, int s, int p, int dil, int in, int out) {
    Interval r;
    r.lo = -floor_div(-(p - dil * t), s);           // ceil((p - dil*t) / s)
    r.hi = floor_div(out - 1 + p - dil * t, s);
    r.lo = r.lo > 0 ? r.lo : 0;
    r.hi = r.hi < in - 1 ? r.hi : in - 1;
    return r;
}

struct BoxParams {
    const float *x;
    float *box;  // [kd*kh*kw][Cin][N]: the samples of one (tap, ci) side by side
    int N, Cin, D, H, W, Do, Ho, Wo;
    int cl;      // channels-last x
    int x16;     // x is a bf16 array
    int kd, kh, kw, sd, sh, sw, pd, ph, pw, dd, dh, dw;  // kernel, stride, pad, dilation per dimension
};

// One block per (n, ci).  fp32 sums: at most D*H*W terms of the input each,
// far inside the tolerance the contraction's result is held to.
__global__ void __launch_bounds__(256) boxsum_kernel(const BoxParams P) {
    extern __shared__ float sm[];
    const int H = P.H, W = P.W, HW = H * W;
    float *a1 = sm;                        // [kd][H][W]: sums along d
    float *a2 = sm + (size_t)P.kd * HW;    // [kd][kh][W]: then along h
    const int n = blockIdx.x / P.Cin, ci = blockIdx.x % P.Cin;
    // element (d, col) of this (n, ci) slab: NCDHW contiguous, or channels-last with stride Cin
    const float *xp = P.cl ? P.x + (size_t)n * P.D * HW * P.Cin + ci : P.x + (size_t)blockIdx.x * P.D * HW;
    const size_t es = P.cl ? (size_t)P.Cin : 1;

    int dlo[kMaxK], dhi[kMaxK];
#pragma unroll
    for (int t = 0; t < kMaxK; ++t) {
        const Interval iv = t < P.kd ? tap_interval(t, P.sd, P.pd, P.dd, P.D, P.Do) : Interval{1, 0};
        dlo[t] = iv.lo;
        dhi[t] = iv.hi;
    }
    if (HW % 4 == 0 && !P.cl && !P.x16) {
        // 128-bit loads: the slab of (n, ci) starts on a 16-byte boundary when H*W % 4 == 0
        for (int c4 = threadIdx.x; c4 < HW / 4; c4 += blockDim.x) {
            float4 acc[kMaxK];
#pragma unroll
            for (int t = 0; t < kMaxK; ++t) acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
            for (int d = 0; d < P.D; ++d) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(xp + (size_t)d * HW) + c4);
#pragma unroll
                for (int t = 0; t < kMaxK; ++t)
                    if (d >= dlo[t] && d <= dhi[t]) {
                        acc[t].x += v.x;
                        acc[t].y += v.y;
                        acc[t].z += v.z;
                        acc[t].w += v.w;
                    }
            }
#pragma unroll
            for (int t = 0; t < kMaxK; ++t)
                if (t < P.kd) reinterpret_cast<float4 *>(a1 + (size_t)t * HW)[c4] = acc[t];
        }
    } else {
        for (int col = threadIdx.x; col < HW; col += blockDim.x) {
            float acc[kMaxK];
#pragma unroll
            for (int t = 0; t < kMaxK; ++t) acc[t] = 0.f;
            for (int d = 0; d < P.D; ++d) {
                const size_t xi = ((size_t)d * HW + col) * es;
                const float v = P.x16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(P.x)[(xp - P.x) + xi])
                                      : __ldg(xp + xi);
#pragma unroll
                for (int t = 0; t < kMaxK; ++t)
                    if (d >= dlo[t] && d <= dhi[t]) acc[t] += v;
            }
#pragma unroll
            for (int t = 0; t < kMaxK; ++t)
                if (t < P.kd) a1[(size_t)t * HW + col] = acc[t];
        }
    }
    __syncthreads();
    // along h: inclusive prefix sums of each (td, w) column, then one difference per interval
    for (int col = threadIdx.x; col < P.kd * W; col += blockDim.x) {
        float *c = a1 + (size_t)(col / W) * HW + col % W;
        float run = 0.f;
        for (int h = 0; h < H; ++h) {
            run += c[(size_t)h * W];
            c[(size_t)h * W] = run;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < P.kd * P.kh * W; i += blockDim.x) {
        const int w = i % W, th = (i / W) % P.kh, td = i / (W * P.kh);
        const Interval iv = tap_interval(th, P.sh, P.ph, P.dh, H, P.Ho);
        const float *c = a1 + (size_t)td * HW + w;
        a2[i] = iv.hi < iv.lo ? 0.f : c[(size_t)iv.hi * W] - (iv.lo > 0 ? c[(size_t)(iv.lo - 1) * W] : 0.f);
    }
    __syncthreads();
    const int k3 = P.kd * P.kh * P.kw;
    for (int i = threadIdx.x; i < k3; i += blockDim.x) {
        const int tw = i % P.kw, tdh = i / P.kw;  // i = (td*kh + th)*kw + tw
        const Interval iv = tap_interval(tw, P.sw, P.pw, P.dw, W, P.Wo);
        float acc = 0.f;
        for (int w = iv.lo; w <= iv.hi; ++w) acc += a2[(size_t)tdh * W + w];
        P.box[((size_t)i * P.Cin + ci) * P.N + n] = acc;
    }
}

struct TapTable {
    int16_t widx[kMaxTaps];
};

constexpr int kOutSamples = 16;  // samples per contraction block

struct OutParams {
    const float *box;
    const float *w_a, *w_b;  // tensor-core layout: TF32 hi/lo planes [tap][cout_pad][cin_pad]; FFMA: [tap][cin_pad][cout_pad]
    const float *bias, *gamma, *beta, *rmean, *rvar;
    float *y;
    int N, Cin, Cout, cin_pad, cout_pad, ntaps, k3, kmajor, wbf16, y16;
    double inv_vol, scale, eps;
};

// One block of 512 threads per (c, group of 16 samples): each weight element
// is read once per block and multiplied into the 16 samples' box sums;
// per-thread fp32 partial sums, then a block reduction.
constexpr int kOutThreads = 512;

__global__ void __launch_bounds__(kOutThreads) bn_eval_out_kernel(const OutParams P,
                                                          const __grid_constant__ TapTable taps) {
    const int c = blockIdx.x, n0 = blockIdx.y * kOutSamples;
    const int nn = P.N - n0 < kOutSamples ? P.N - n0 : kOutSamples;
    // 16 samples' box sums of one (tap, ci) are consecutive: four 16-byte loads
    const bool vec = nn == kOutSamples && P.N % 4 == 0;
    const int total = P.ntaps * P.Cin;
    float acc[kOutSamples];
#pragma unroll
    for (int q = 0; q < kOutSamples; ++q) acc[q] = 0.f;
#pragma unroll 4
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int j = i / P.Cin, ci = i - j * P.Cin;
        float wv;
        if (P.kmajor) {
            const size_t o = ((size_t)j * P.cout_pad + c) * P.cin_pad + ci;
            if (P.wbf16)  // bf16 planes: hi (+ lo, split bf16)
                wv = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(P.w_a)[o]) +
                     (P.w_b ? __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(P.w_b)[o]) : 0.f);
            else  // hi + lo: the fp32 weight, exactly (or its TF32 rounding)
                wv = P.w_b ? P.w_a[o] + P.w_b[o] : P.w_a[o];
        } else {
            wv = P.w_a[((size_t)j * P.cin_pad + ci) * P.cout_pad + c];
        }
        const float *b = P.box + ((size_t)taps.widx[j] * P.Cin + ci) * P.N + n0;
        if (vec) {
#pragma unroll
            for (int q4 = 0; q4 < kOutSamples / 4; ++q4) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(b) + q4);
                acc[4 * q4] = fmaf(wv, v.x, acc[4 * q4]);
                acc[4 * q4 + 1] = fmaf(wv, v.y, acc[4 * q4 + 1]);
                acc[4 * q4 + 2] = fmaf(wv, v.z, acc[4 * q4 + 2]);
                acc[4 * q4 + 3] = fmaf(wv, v.w, acc[4 * q4 + 3]);
            }
        } else {
#pragma unroll
            for (int q = 0; q < kOutSamples; ++q)
                if (q < nn) acc[q] = fmaf(wv, b[q], acc[q]);
        }
    }
    __shared__ float red[kOutSamples][kOutThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int q = 0; q < kOutSamples; ++q) {
        float v = acc[q];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) red[q][warp] = v;
    }
    __syncthreads();
    if (threadIdx.x < nn) {
        const int q = threadIdx.x;
        double S = 0.0;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) S += (double)red[q][i];
        const double mean_y = S * P.inv_vol + (P.bias ? (double)P.bias[c] : 0.0);
        const double rstd = 1.0 / sqrt((double)P.rvar[c] + P.eps);
        const float out =
            (float)((double)P.gamma[c] * (P.scale * mean_y - (double)P.rmean[c]) * rstd + (double)P.beta[c]);
        if (P.y16)
            reinterpret_cast<__nv_bfloat16 *>(P.y)[(size_t)(n0 + q) * P.Cout + c] = __float2bfloat16_rn(out);
        else
            P.y[(size_t)(n0 + q) * P.Cout + c] = out;
    }
}

}  // namespace

size_t bn_eval_smem_bytes(const convt3d_plan_s &p) {
    const size_t kd = p.g.kk[0], kh = p.g.kk[1];
    return (kd * p.g.Hin * p.g.Win + kd * kh * p.g.Win) * sizeof(float);
}

cudaError_t launch_bn_eval(const convt3d_plan_s &p, const float *x, const float *w_a, const float *w_b,
                           const float *bias, const float *gamma, const float *beta, float *box, float *y,
                           cudaStream_t s) {
    const Geometry &g = p.g;
    BoxParams bp{x,        box,      g.N,      g.Cin,    g.Din,    g.Hin,    g.Win,    g.Do,     g.Ho,     g.Wo,
                 p.cl,     p.io16,   g.kk[0],  g.kk[1],  g.kk[2],  g.ss[0],  g.ss[1],  g.ss[2],  g.pp[0],
                 g.pp[1],  g.pp[2],  g.dil[0], g.dil[1], g.dil[2]};
    const size_t smem = bn_eval_smem_bytes(p);
    cudaError_t e = cudaFuncSetAttribute(boxsum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    boxsum_kernel<<<(unsigned)(g.N * g.Cin), 256, smem, s>>>(bp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    TapTable t;
    for (int j = 0; j < kMaxTaps; ++j) t.widx[j] = j < g.ntaps ? g.taps[j].widx : 0;
    OutParams op;
    op.box = box;
    op.w_a = w_a;
    op.w_b = w_b;
    op.bias = bias;
    op.gamma = gamma;
    op.beta = beta;
    op.rmean = p.run_mean;
    op.rvar = p.run_var;
    op.y = y;
    op.N = g.N;
    op.Cin = g.Cin;
    op.Cout = g.Cout;
    op.cin_pad = p.cin_pad;
    op.cout_pad = p.cout_pad;
    op.ntaps = g.ntaps;
    op.k3 = g.kvol;
    op.kmajor = p.tc;
    op.wbf16 = p.bf16;
    op.y16 = p.io16;
    op.inv_vol = 1.0 / ((double)g.Do * g.Ho * g.Wo);
    op.scale = (double)p.d.scale;
    op.eps = (double)p.d.eps;
    dim3 grid((unsigned)g.Cout, (unsigned)((g.N + kOutSamples - 1) / kOutSamples));
    bn_eval_out_kernel<<<grid, kOutThreads, 0, s>>>(op, t);
    return cudaGetLastError();
}

}  // namespace convt3d
