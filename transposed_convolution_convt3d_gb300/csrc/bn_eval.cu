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
// to o = stride*i - pad + t per dimension).  The box is a product of one
// interval per dimension, so B is three passes of 1-D interval sums:
//   boxsum_kernel    one block per (n, ci): x once along d into k accumulators
//                    per (h, w) column, then intervals along h, then along w;
//   bn_eval_out_kernel  one block per (n, c): the Cin*k^3 contraction with the
//                    packed weight, fp64 accumulation, then the formula above.
// The work is O(N*Cin*D*H*W*k + N*Cout*Cin*k^3), a read of x and of the weight.
#include "convt3d_internal.h"

namespace convt3d {
namespace {

constexpr int kMaxK = 7;

__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Inputs i whose output s*i - p + t lies in [0, out - 1], clamped to [0, in - 1].
struct Interval {
    int lo, hi;
};

__device__ __forceinline__ Interval tap_interval(int t, int s, int p, int in, int out) {
    Interval r;
    r.lo = -floor_div(-(p - t), s);           // ceil((p - t) / s)
    r.hi = floor_div(out - 1 + p - t, s);
    r.lo = r.lo > 0 ? r.lo : 0;
    r.hi = r.hi < in - 1 ? r.hi : in - 1;
    return r;
}

struct BoxParams {
    const float *x;
    double *box;  // [N][k^3][Cin]
    int Cin, D, H, W, k, s, p, Do, Ho, Wo;
};

__global__ void __launch_bounds__(256) boxsum_kernel(const BoxParams P) {
    extern __shared__ double sm[];
    const int k = P.k, H = P.H, W = P.W, HW = H * W;
    double *a1 = sm;                 // [k][H][W]: sums along d
    double *a2 = sm + (size_t)k * HW;  // [k][k][W]: then along h
    const int n = blockIdx.x / P.Cin, ci = blockIdx.x % P.Cin;
    const float *xp = P.x + (size_t)blockIdx.x * P.D * HW;

    int dlo[kMaxK], dhi[kMaxK];
#pragma unroll
    for (int t = 0; t < kMaxK; ++t) {
        const Interval iv = t < k ? tap_interval(t, P.s, P.p, P.D, P.Do) : Interval{1, 0};
        dlo[t] = iv.lo;
        dhi[t] = iv.hi;
    }
    for (int col = threadIdx.x; col < HW; col += blockDim.x) {
        double acc[kMaxK];
#pragma unroll
        for (int t = 0; t < kMaxK; ++t) acc[t] = 0.0;
        for (int d = 0; d < P.D; ++d) {
            const double v = (double)__ldg(xp + (size_t)d * HW + col);
#pragma unroll
            for (int t = 0; t < kMaxK; ++t)
                if (d >= dlo[t] && d <= dhi[t]) acc[t] += v;
        }
#pragma unroll
        for (int t = 0; t < kMaxK; ++t)
            if (t < k) a1[(size_t)t * HW + col] = acc[t];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < k * k * W; i += blockDim.x) {
        const int w = i % W, th = (i / W) % k, td = i / (W * k);
        const Interval iv = tap_interval(th, P.s, P.p, H, P.Ho);
        double acc = 0.0;
        for (int h = iv.lo; h <= iv.hi; ++h) acc += a1[(size_t)td * HW + h * W + w];
        a2[i] = acc;
    }
    __syncthreads();
    const int k3 = k * k * k;
    for (int i = threadIdx.x; i < k3; i += blockDim.x) {
        const int tw = i % k, tdh = i / k;  // i = (td*k + th)*k + tw
        const Interval iv = tap_interval(tw, P.s, P.p, W, P.Wo);
        double acc = 0.0;
        for (int w = iv.lo; w <= iv.hi; ++w) acc += a2[(size_t)tdh * W + w];
        P.box[((size_t)n * k3 + i) * P.Cin + ci] = acc;
    }
}

struct TapTable {
    int16_t widx[kMaxTaps];
};

struct OutParams {
    const double *box;
    const float *w_a, *w_b;  // tensor-core layout: TF32 hi/lo planes [tap][cout_pad][cin_pad]; FFMA: [tap][cin_pad][cout_pad]
    const float *bias, *gamma, *beta, *rmean, *rvar;
    float *y;
    int Cin, Cout, cin_pad, cout_pad, ntaps, k3, kmajor;
    double inv_vol, scale, eps;
};

__global__ void __launch_bounds__(256) bn_eval_out_kernel(const OutParams P,
                                                          const __grid_constant__ TapTable taps) {
    const int n = blockIdx.x / P.Cout, c = blockIdx.x % P.Cout;
    const double *bx = P.box + (size_t)n * P.k3 * P.Cin;
    const int total = P.ntaps * P.Cin;
    double acc = 0.0;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int j = i / P.Cin, ci = i % P.Cin;
        float wv;
        if (P.kmajor) {
            const size_t o = ((size_t)j * P.cout_pad + c) * P.cin_pad + ci;
            wv = P.w_a[o] + P.w_b[o];  // hi + lo: the fp32 weight, exactly
        } else {
            wv = P.w_a[((size_t)j * P.cin_pad + ci) * P.cout_pad + c];
        }
        acc += (double)wv * bx[(size_t)taps.widx[j] * P.Cin + ci];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    __shared__ double red[8];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        double S = 0.0;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) S += red[i];
        const double mean_y = S * P.inv_vol + (P.bias ? (double)P.bias[c] : 0.0);
        const double rstd = 1.0 / sqrt((double)P.rvar[c] + P.eps);
        P.y[(size_t)n * P.Cout + c] =
            (float)((double)P.gamma[c] * (P.scale * mean_y - (double)P.rmean[c]) * rstd + (double)P.beta[c]);
    }
}

}  // namespace

size_t bn_eval_smem_bytes(const convt3d_plan_s &p) {
    const size_t k = p.g.k;
    return (k * p.g.Hin * p.g.Win + k * k * p.g.Win) * sizeof(double);
}

cudaError_t launch_bn_eval(const convt3d_plan_s &p, const float *x, const float *w_a, const float *w_b,
                           const float *bias, const float *gamma, const float *beta, double *box, float *y,
                           cudaStream_t s) {
    const Geometry &g = p.g;
    BoxParams bp{x, box, g.Cin, g.Din, g.Hin, g.Win, g.k, g.stride, g.pad, g.Do, g.Ho, g.Wo};
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
    op.Cin = g.Cin;
    op.Cout = g.Cout;
    op.cin_pad = p.cin_pad;
    op.cout_pad = p.cout_pad;
    op.ntaps = g.ntaps;
    op.k3 = g.k * g.k * g.k;
    op.kmajor = p.tc;
    op.inv_vol = 1.0 / ((double)g.Do * g.Ho * g.Wo);
    op.scale = (double)p.d.scale;
    op.eps = (double)p.d.eps;
    bn_eval_out_kernel<<<(unsigned)(g.N * g.Cout), 256, 0, s>>>(op, t);
    return cudaGetLastError();
}

}  // namespace convt3d
