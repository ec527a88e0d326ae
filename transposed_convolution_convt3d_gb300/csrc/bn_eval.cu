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
//   boxsum_kernel    one block per (n, ci): x once along d into one
//                    accumulator per distinct d-interval (taps whose intervals
//                    coincide share it) per (h, w) column, then intervals along
//                    h (prefix sums, one difference per interval), then along w;
//   bn_eval_out_kernel  blocks per (c, 16 samples, K split): the Cin*k^3
//                    contraction with the packed weight; the last block of a
//                    (c, samples) pair to finish adds the splits' fp64 partial
//                    sums in split order and applies the formula above.
// The work is O(N*Cin*D*H*W*k + N*Cout*Cin*k^3), a read of x and of the weight.
#include <cuda_bf16.h>

#include <type_traits>

#include "convt3d_internal.h"

namespace convt3d {
namespace {

constexpr int kMaxK = 7;

__host__ __device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

// Inputs i whose output s*i - p + dil*t lies in [0, out - 1], clamped to [0, in - 1].
struct Interval {
    int lo, hi;
};

__host__ __device__ __forceinline__ Interval tap_interval(int t, int s, int p, int dil, int in, int out) {
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
    int x16;     // x is a 16-bit array of that kind (kBF16 / kF16), 0: fp32
    int kd, kh, kw, sd, sh, sw, pd, ph, pw, dd, dh, dw;  // kernel, stride, pad, dilation per dimension
    // distinct d-intervals of the taps along d: nud of them, tap td uses ud_of[td]
    int nud;
    int ud_lo[kMaxK], ud_hi[kMaxK], ud_of[kMaxK];
};

// One block per (n, ci); NUD = the number of distinct d-intervals (a
// compile-time count, so that each load feeds exactly that many accumulators).
// fp32 sums: at most D*H*W terms of the input each, far inside the tolerance
// the contraction's result is held to.
template <int NUD>
__global__ void __launch_bounds__(256) boxsum_kernel(const BoxParams P) {
    extern __shared__ float sm[];
    const int H = P.H, W = P.W, HW = H * W;
    float *a1 = sm;                        // [nud][H][W]: sums along d, one plane per distinct interval
    float *a2 = sm + (size_t)P.nud * HW;   // [kd][kh][W]: then along h
    const int n = blockIdx.x / P.Cin, ci = blockIdx.x % P.Cin;
    // element (d, col) of this (n, ci) slab: NCDHW contiguous, or channels-last with stride Cin
    const float *xp = P.cl ? P.x + (size_t)n * P.D * HW * P.Cin + ci : P.x + (size_t)blockIdx.x * P.D * HW;
    const size_t es = P.cl ? (size_t)P.Cin : 1;

    int dlo[NUD], dhi[NUD];
#pragma unroll
    for (int t = 0; t < NUD; ++t) {
        dlo[t] = P.ud_lo[t];
        dhi[t] = P.ud_hi[t];
    }
    if (HW % 4 == 0 && !P.cl && !P.x16) {
        // 128-bit loads: the slab of (n, ci) starts on a 16-byte boundary when H*W % 4 == 0
        for (int c4 = threadIdx.x; c4 < HW / 4; c4 += blockDim.x) {
            float4 acc[NUD];
#pragma unroll
            for (int t = 0; t < NUD; ++t) acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
            for (int d = 0; d < P.D; ++d) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(xp + (size_t)d * HW) + c4);
#pragma unroll
                for (int t = 0; t < NUD; ++t)
                    if (d >= dlo[t] && d <= dhi[t]) {
                        acc[t].x += v.x;
                        acc[t].y += v.y;
                        acc[t].z += v.z;
                        acc[t].w += v.w;
                    }
            }
#pragma unroll
            for (int t = 0; t < NUD; ++t) reinterpret_cast<float4 *>(a1 + (size_t)t * HW)[c4] = acc[t];
        }
    } else {
        for (int col = threadIdx.x; col < HW; col += blockDim.x) {
            float acc[NUD];
#pragma unroll
            for (int t = 0; t < NUD; ++t) acc[t] = 0.f;
            for (int d = 0; d < P.D; ++d) {
                const size_t xi = ((size_t)d * HW + col) * es;
                const float v = P.x16 ? ld16(P.x, (xp - P.x) + xi, P.x16) : __ldg(xp + xi);
#pragma unroll
                for (int t = 0; t < NUD; ++t)
                    if (d >= dlo[t] && d <= dhi[t]) acc[t] += v;
            }
#pragma unroll
            for (int t = 0; t < NUD; ++t) a1[(size_t)t * HW + col] = acc[t];
        }
    }
    __syncthreads();
    // along h: inclusive prefix sums of each (interval, w) column, then one difference per interval
    for (int col = threadIdx.x; col < P.nud * W; col += blockDim.x) {
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
        const float *c = a1 + (size_t)P.ud_of[td] * HW + w;
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
    double *part;         // [ks][N][Cout] partial sums when the contraction is split (ks > 1)
    unsigned *counters;   // [N/16 blocks][Cout] blocks finished, reset to 0 by the last one
    int ks;
    const float *w_a, *w_b;  // tensor-core layout: TF32 hi/lo planes [tap][cout_pad][cin_pad]; FFMA: [tap][cin_pad][cout_pad]
    const float *bias, *gamma, *beta, *rmean, *rvar;
    float *y;
    int N, Cin, Cout, cin_pad, cout_pad, ntaps, k3, kmajor, w16, y16;  // w16 / y16: 16-bit kinds (0: fp32)
    double inv_vol, scale, eps;
};

// Blocks of 256 threads per (c, group of 16 samples, K split): each weight
// element is read once per block and multiplied into the 16 samples' box
// sums; per-thread fp32 partial sums, then a block reduction.  With K split
// (ks > 1) the last block of a (c, samples) pair to finish adds the splits'
// fp64 sums in split order.
constexpr int kOutThreads = 256;

__global__ void __launch_bounds__(kOutThreads) bn_eval_out_kernel(const OutParams P,
                                                          const __grid_constant__ TapTable taps) {
    const int c = blockIdx.x, n0 = blockIdx.y * kOutSamples;
    const int nn = P.N - n0 < kOutSamples ? P.N - n0 : kOutSamples;
    // 16 samples' box sums of one (tap, ci) are consecutive: four 16-byte loads
    const bool vec = nn == kOutSamples && P.N % 4 == 0;
    const int total = P.ntaps * P.Cin;
    const int ks = blockIdx.z;  // this block's share of the K = taps x Cin products
    const int i_begin = (int)((int64_t)total * ks / P.ks), i_end = (int)((int64_t)total * (ks + 1) / P.ks);
    float acc[kOutSamples];
#pragma unroll
    for (int q = 0; q < kOutSamples; ++q) acc[q] = 0.f;
    // The loop over this thread's products, specialised on the box-row access (four
    // 16-byte loads, or scalars for a partial sample block) and the weight layout
    // (0: tensor-core fp32 planes, 1: tensor-core bf16 planes, 2: FFMA layout, 3: tensor-core
    // fp16 plane), with
    // the (tap, ci) index stepped instead of divided per product.
    auto contract = [&](auto vec_t, auto wm_t) {
        constexpr bool kVec = decltype(vec_t)::value;
        constexpr int kWm = decltype(wm_t)::value;
        const int i0 = i_begin + (int)threadIdx.x;
        int j = i0 / P.Cin, ci = i0 - j * P.Cin;
        const int dj = (int)blockDim.x / P.Cin, dci = (int)blockDim.x - dj * P.Cin;
#pragma unroll 4
        for (int i = i0; i < i_end; i += blockDim.x) {
            float wv;
            if constexpr (kWm == 2) {
                wv = P.w_a[((size_t)j * P.cin_pad + ci) * P.cout_pad + c];
            } else {
                const size_t o = ((size_t)j * P.cout_pad + c) * P.cin_pad + ci;
                if constexpr (kWm == 1)  // bf16 planes: hi (+ lo, split bf16)
                    wv = ld16(P.w_a, (int64_t)o, kBF16) + (P.w_b ? ld16(P.w_b, (int64_t)o, kBF16) : 0.f);
                else if constexpr (kWm == 3)  // one fp16 plane
                    wv = ld16(P.w_a, (int64_t)o, kF16);
                else  // hi + lo: the fp32 weight, exactly (or its TF32 rounding)
                    wv = P.w_b ? P.w_a[o] + P.w_b[o] : P.w_a[o];
            }
            const float *b = P.box + ((size_t)taps.widx[j] * P.Cin + ci) * P.N + n0;
            if constexpr (kVec) {
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
                    if (q < nn) acc[q] = fmaf(wv, __ldg(b + q), acc[q]);
            }
            j += dj;
            ci += dci;
            if (ci >= P.Cin) {
                ci -= P.Cin;
                ++j;
            }
        }
    };
    using T_ = std::true_type;
    using F_ = std::false_type;
    using W0 = std::integral_constant<int, 0>;
    using W1 = std::integral_constant<int, 1>;
    using W2 = std::integral_constant<int, 2>;
    using W3 = std::integral_constant<int, 3>;
    if (!P.kmajor)
        vec ? contract(T_{}, W2{}) : contract(F_{}, W2{});
    else if (P.w16 == kF16)
        vec ? contract(T_{}, W3{}) : contract(F_{}, W3{});
    else if (P.w16)
        vec ? contract(T_{}, W1{}) : contract(F_{}, W1{});
    else
        vec ? contract(T_{}, W0{}) : contract(F_{}, W0{});
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
    double S = 0.0;
    if (threadIdx.x < nn)
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) S += (double)red[threadIdx.x][i];
    if (P.ks > 1) {
        // publish this split's sums; the block that finishes last for (c, samples)
        // adds all splits in split order (a fixed order: results are reproducible)
        __shared__ bool last;
        if (threadIdx.x < nn) P.part[((size_t)ks * P.N + n0 + threadIdx.x) * P.Cout + c] = S;
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned *cnt = P.counters + (size_t)blockIdx.y * P.Cout + c;
            last = atomicAdd(cnt, 1u) == (unsigned)P.ks - 1u;
            if (last) *cnt = 0u;  // ready for the next forward
        }
        __syncthreads();
        if (!last) return;
        __threadfence();
        if (threadIdx.x < nn) {
            S = 0.0;
            for (int k = 0; k < P.ks; ++k)
                S += __ldcg(P.part + ((size_t)k * P.N + n0 + threadIdx.x) * P.Cout + c);
        }
    }
    if (threadIdx.x < nn) {
        const int q = threadIdx.x;
        const double mean_y = S * P.inv_vol + (P.bias ? (double)P.bias[c] : 0.0);
        const double rstd = 1.0 / sqrt((double)P.rvar[c] + P.eps);
        const float out =
            (float)((double)P.gamma[c] * (P.scale * mean_y - (double)P.rmean[c]) * rstd + (double)P.beta[c]);
        if (P.y16)  // 16-bit output of that kind
            reinterpret_cast<uint16_t *>(P.y)[(size_t)(n0 + q) * P.Cout + c] = cvt16(out, P.y16);
        else
            P.y[(size_t)(n0 + q) * P.Cout + c] = out;
    }
}

}  // namespace

// Distinct d-intervals of the taps (host): taps whose input intervals along d
// coincide (for example every tap when no padding crops the output) share one
// accumulator in boxsum_kernel.
static int unique_d_intervals(const Geometry &g, int lo[kMaxK], int hi[kMaxK], int of[kMaxK]) {
    int n = 0;
    for (int t = 0; t < kMaxK; ++t) {
        of[t] = 0;
        if (t >= g.kk[0]) continue;
        const Interval iv = tap_interval(t, g.ss[0], g.pp[0], g.dil[0], g.Din, g.Do);
        int u = 0;
        while (u < n && !(lo[u] == iv.lo && hi[u] == iv.hi)) ++u;
        if (u == n) {
            lo[n] = iv.lo;
            hi[n] = iv.hi;
            ++n;
        }
        of[t] = u;
    }
    for (int u = n; u < kMaxK; ++u) lo[u] = 1, hi[u] = 0;
    return n;
}

size_t bn_eval_smem_bytes(const convt3d_plan_s &p) {
    int lo[kMaxK], hi[kMaxK], of[kMaxK];
    const size_t nud = (size_t)unique_d_intervals(p.g, lo, hi, of);
    const size_t kd = p.g.kk[0], kh = p.g.kk[1];
    return (nud * p.g.Hin * p.g.Win + kd * kh * p.g.Win) * sizeof(float);
}

// K splits of the contraction: about 2,048 products per block, at most 16 splits.
int bn_eval_ksplits(int ntaps, int Cin) {
    const int total = ntaps * Cin;
    const int ks = (total + 2047) / 2048;
    return ks < 1 ? 1 : (ks > 16 ? 16 : ks);
}

cudaError_t launch_bn_eval(const convt3d_plan_s &p, const float *x, const float *w_a, const float *w_b,
                           const float *bias, const float *gamma, const float *beta, float *box, double *part,
                           unsigned *counters, float *y, cudaStream_t s) {
    const Geometry &g = p.g;
    BoxParams bp{x,        box,      g.N,      g.Cin,    g.Din,    g.Hin,    g.Win,    g.Do,     g.Ho,     g.Wo,
                 p.cl,     p.io16,   g.kk[0],  g.kk[1],  g.kk[2],  g.ss[0],  g.ss[1],  g.ss[2],  g.pp[0],
                 g.pp[1],  g.pp[2],  g.dil[0], g.dil[1], g.dil[2]};
    bp.nud = unique_d_intervals(g, bp.ud_lo, bp.ud_hi, bp.ud_of);
    const size_t smem = bn_eval_smem_bytes(p);
    void (*kern)(const BoxParams) = nullptr;
    switch (bp.nud) {
        case 1: kern = boxsum_kernel<1>; break;
        case 2: kern = boxsum_kernel<2>; break;
        case 3: kern = boxsum_kernel<3>; break;
        case 4: kern = boxsum_kernel<4>; break;
        case 5: kern = boxsum_kernel<5>; break;
        case 6: kern = boxsum_kernel<6>; break;
        case 7: kern = boxsum_kernel<7>; break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(g.N * g.Cin), 256, smem, s>>>(bp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    TapTable t;
    for (int j = 0; j < kMaxTaps; ++j) t.widx[j] = j < g.ntaps ? g.taps[j].widx : 0;
    OutParams op;
    op.box = box;
    op.part = part;
    op.counters = counters;
    op.ks = p.ev_ks;
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
    op.w16 = p.bf16 ? (p.half ? kF16 : kBF16) : kF32;
    op.y16 = p.io16;
    op.inv_vol = 1.0 / ((double)g.Do * g.Ho * g.Wo);
    op.scale = (double)p.d.scale;
    op.eps = (double)p.d.eps;
    dim3 grid((unsigned)g.Cout, (unsigned)((g.N + kOutSamples - 1) / kOutSamples), (unsigned)p.ev_ks);
    bn_eval_out_kernel<<<grid, kOutThreads, 0, s>>>(op, t);
    return cudaGetLastError();
}

}  // namespace convt3d
