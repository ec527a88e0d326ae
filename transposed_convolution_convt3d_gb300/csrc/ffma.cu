// CUDA-core (fp32 FMA) output-stationary implicit GEMM with the fused
// epilogues -- the ablation beside the tensor-core path.
//
// One block computes a tile of 64 output positions of one parity class
// (consecutive positions of the class's q-grid within one sample) by all
// output channels.  K runs over (tap of the class, 8 input channels); the
// activation slice is gathered from NCDHW x with the class's tap offsets
// (input index i = q + delta, out-of-range reads are zero), the weight slice
// comes from the [tap][Cin_pad][Cout_pad] packed copy.  256 threads hold a
// 4 x CPT register tile each.  The accumulated tile (+bias) then passes
// through shared memory to the epilogue:
//   identity         store;
//   softmax+sigmoid  per position over all channels, store;
//   relu+groupnorm   per-group (count, sum, M2) partials of v = ReLU(conv + b), store v - b;
//   scale+bn+pool    scale, per-channel (count, sum, M2) partials, no store.
#include <string.h>

#include "convt3d_internal.h"

namespace convt3d {
namespace {

constexpr int kThreads = 256;
constexpr int kBM = kFfmaTileM;  // 64
constexpr int kBK = 8;

struct TileInfo {
    int n, gi, t, cls, slot;
};

__device__ __forceinline__ TileInfo decode_tile(const FfmaParams &P, int bid) {
    TileInfo ti;
    ti.n = bid / P.tiles_per_sample;
    const int r = bid % P.tiles_per_sample;
    int gi = 0;
    for (int i = 1; i < P.ngroups; ++i)
        if (r >= P.grp[i].tile_prefix) gi = i;
    ti.gi = gi;
    ti.t = r - P.grp[gi].tile_prefix;
    ti.cls = P.grp[gi].cls[0];
    ti.slot = bid;  // == n * tiles_per_sample + r
    return ti;
}

// ReLU(a + b) in fp64 for the GroupNorm statistics, b = bias[c] (0 without a bias).
__device__ __forceinline__ double relu_biased(float a, const float *bias, int c) {
    const float t = a + (bias ? bias[c] : 0.0f);
    return t > 0.0f ? (double)a + (bias ? (double)bias[c] : 0.0) : 0.0;
}

template <int CPT>
__global__ void __launch_bounds__(kThreads) ffma_conv_kernel(const __grid_constant__ FfmaParams P) {
    extern __shared__ __align__(16) float smem[];
    const int cpad = P.cout_pad;                     // == 16 * CPT
    float *As = smem;                                 // [2][kBK][kBM]
    float *Bs = smem + 2 * kBK * kBM;                 // [2][kBK][cpad]
    float *E = smem;                                  // epilogue tile [kBM][cpad + 1] (aliases)
    __shared__ int rowoff[kBM];

    const int tid = threadIdx.x;
    const TileInfo ti = decode_tile(P, P.tile_base + blockIdx.x);
    const ClassDesc &cl = P.cls[ti.cls];
    const int Qhw = cl.Qh * cl.Qw;
    const int vol = cl.Qd * Qhw;
    const int64_t Sin = (int64_t)P.Din * P.Hin * P.Win;
    const int64_t Sout = (int64_t)P.Do * P.Ho * P.Wo;

    // Positions this thread loads: m = lane and lane + 32 of the tile.
    int lq[2][3];
    bool lvalid[2];
    const int lk = tid / 32;  // channel within the K step
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int q = ti.t * kBM + (tid % 32) + 32 * r;
        lvalid[r] = q < vol;
        lq[r][0] = q / Qhw;
        lq[r][1] = (q / cl.Qw) % cl.Qh;
        lq[r][2] = q % cl.Qw;
    }
    const float *xn = P.x + (int64_t)ti.n * P.Cin * Sin;
    const int kc = P.cin_pad / kBK;
    const int nsteps = cl.ntaps * kc;

    float acc[4][CPT];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < CPT; ++j) acc[i][j] = 0.0f;

    int64_t sp[2] = {-1, -1};
    int cur_tap = -1;
    float areg[2];
    constexpr int kBRegs = (kBK * 16 * CPT / 4 + kThreads - 1) / kThreads;  // float4s per thread per weight slice
    float4 breg[kBRegs];
    const int nb4 = kBK * cpad / 4;  // float4s in one weight slice

    auto load_step = [&](int step) {
        const int j = step / kc;
        const int ci0 = (step % kc) * kBK;
        if (j != cur_tap) {
            cur_tap = j;
            const TapDesc td = P.taps[cl.tap_begin + j];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int id = lq[r][0] + td.dd, ih = lq[r][1] + td.dh, iw = lq[r][2] + td.dw;
                const bool ok = lvalid[r] && id >= 0 && id < P.Din && ih >= 0 && ih < P.Hin && iw >= 0 && iw < P.Win;
                sp[r] = ok ? ((int64_t)id * P.Hin + ih) * P.Win + iw : -1;
            }
        }
        const int ci = ci0 + lk;
#pragma unroll
        for (int r = 0; r < 2; ++r)
            areg[r] = (sp[r] >= 0 && ci < P.Cin) ? __ldg(xn + (int64_t)ci * P.xcs + sp[r] * P.xps) : 0.0f;
        const float4 *wsrc = reinterpret_cast<const float4 *>(
            P.wpk + ((int64_t)(cl.tap_begin + j) * P.cin_pad + ci0) * cpad);
#pragma unroll
        for (int r = 0; r < kBRegs; ++r) {
            const int idx = tid + r * kThreads;
            if (idx < nb4) breg[r] = __ldg(wsrc + idx);
        }
    };
    auto store_step = [&](int buf) {
        float *A = As + buf * kBK * kBM;
        A[lk * kBM + (tid % 32)] = areg[0];
        A[lk * kBM + (tid % 32) + 32] = areg[1];
        float4 *B = reinterpret_cast<float4 *>(Bs + buf * kBK * cpad);
#pragma unroll
        for (int r = 0; r < kBRegs; ++r) {
            const int idx = tid + r * kThreads;
            if (idx < nb4) B[idx] = breg[r];
        }
    };

    const int tx = tid % 16, ty = tid / 16;
    if (nsteps > 0) {
        load_step(0);
        store_step(0);
        __syncthreads();
        for (int step = 0; step < nsteps; ++step) {
            const int buf = step & 1;
            if (step + 1 < nsteps) load_step(step + 1);
            const float *A = As + buf * kBK * kBM;
            const float *B = Bs + buf * kBK * cpad;
#pragma unroll
            for (int kk = 0; kk < kBK; ++kk) {
                const float4 a = *reinterpret_cast<const float4 *>(A + kk * kBM + ty * 4);
                float b[CPT];
#pragma unroll
                for (int j = 0; j < CPT; ++j) b[j] = B[kk * cpad + tx * CPT + j];
                const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < CPT; ++j) acc[i][j] = fmaf(av[i], b[j], acc[i][j]);
            }
            if (step + 1 < nsteps) store_step(buf ^ 1);
            __syncthreads();
        }
    }

    // ---- epilogue ------------------------------------------------------
    const int es = cpad + 1;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int c = tx * CPT + j;
            const float b = (P.bias && c < P.Cout) ? P.bias[c] : 0.0f;
            // GroupNorm keeps the accumulator: its statistics add the bias, and the stored
            // value is relative to it (see below)
            E[(ty * 4 + i) * es + c] = P.epilogue == CONVT3D_EPI_RELU_GROUPNORM ? acc[i][j] : acc[i][j] + b;
        }
    if (tid < kBM) {
        const int q = ti.t * kBM + tid;
        int off = -1;
        if (q < vol) {
            const int od = P.sd * (q / Qhw) + cl.rd;
            const int oh = P.sh * ((q / cl.Qw) % cl.Qh) + cl.rh;
            const int ow = P.sw * (q % cl.Qw) + cl.rw;
            if (od < P.Do && oh < P.Ho && ow < P.Wo) off = (od * P.Ho + oh) * P.Wo + ow;
        }
        rowoff[tid] = off;
    }
    __syncthreads();

    const int C = P.Cout;
    float *yn = P.y + (int64_t)ti.n * C * Sout;
    if (P.epilogue == CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL) {
        // per channel over the tile's valid positions: (count, sum, M2) in fp64, M2 about the tile's mean
        double *part = P.partials + (int64_t)ti.slot * 3 * C;
        for (int c = tid; c < C; c += kThreads) {
            double n = 0.0, s1 = 0.0;
            for (int m = 0; m < kBM; ++m) {
                if (rowoff[m] < 0) continue;
                n += 1.0;
                s1 += (double)P.scale * (double)E[m * es + c];
            }
            const double mu = n > 0.0 ? s1 / n : 0.0;
            double m2 = 0.0;
            for (int m = 0; m < kBM; ++m) {
                if (rowoff[m] < 0) continue;
                const double d = (double)P.scale * (double)E[m * es + c] - mu;
                m2 += d * d;
            }
            part[3 * c] = n;
            part[3 * c + 1] = s1;
            part[3 * c + 2] = m2;
        }
        return;
    }
    if (P.epilogue == CONVT3D_EPI_SOFTMAX_SIGMOID) {
        if (tid < kBM && rowoff[tid] >= 0) {
            float *row = E + tid * es;
            float mx = row[0];
            for (int c = 1; c < C; ++c) mx = fmaxf(mx, row[c]);
            float sum = 0.0f;
            for (int c = 0; c < C; ++c) sum += expf(row[c] - mx);
            const float inv = 1.0f / sum;
            for (int c = 0; c < C; ++c) {
                const float t = expf(row[c] - mx) * inv;
                row[c] = 1.0f / (1.0f + expf(-t));
            }
        }
        __syncthreads();
    }
    if (P.epilogue == CONVT3D_EPI_RELU_GROUPNORM) {
        // E holds the accumulator a; the GroupNorm input is v = ReLU(a + b), and y keeps
        // r = v - b (a itself where the ReLU passes, else -b) for the normalise pass
        // per-group (count, sum, M2) over the tile's valid positions in fp64, M2 about
        // the tile's group mean: one warp per group
        const int G = P.groups, cpg = C / G;
        const int warp = tid / 32, lane = tid % 32;
        double *part = P.partials + (int64_t)ti.slot * 3 * G;
        for (int g = warp; g < G; g += kThreads / 32) {
            double n = 0.0, s1 = 0.0;
            for (int m = lane; m < kBM; m += 32) {
                if (rowoff[m] < 0) continue;
                const float *row = E + m * es + g * cpg;
                n += cpg;
                for (int c = 0; c < cpg; ++c) s1 += relu_biased(row[c], P.bias, g * cpg + c);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                n += __shfl_xor_sync(0xffffffffu, n, o);
                s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            }
            const double mu = n > 0.0 ? s1 / n : 0.0;
            double m2 = 0.0;
            for (int m = lane; m < kBM; m += 32) {
                if (rowoff[m] < 0) continue;
                const float *row = E + m * es + g * cpg;
                for (int c = 0; c < cpg; ++c) {
                    const double d = relu_biased(row[c], P.bias, g * cpg + c) - mu;
                    m2 += d * d;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m2 += __shfl_xor_sync(0xffffffffu, m2, o);
            if (lane == 0) {
                part[3 * g] = n;
                part[3 * g + 1] = s1;
                part[3 * g + 2] = m2;
            }
        }
        __syncthreads();
        for (int idx = tid; idx < kBM * C; idx += kThreads) {
            const int m = idx % kBM, c = idx / kBM;
            const float a = E[m * es + c], b = P.bias ? P.bias[c] : 0.0f;
            E[m * es + c] = a + b > 0.0f ? a : -b;
        }
        __syncthreads();
    }
    // store (identity, softmax+sigmoid, relu output before normalisation)
    for (int idx = tid; idx < kBM * C; idx += kThreads) {
        const int m = idx % kBM, c = idx / kBM;
        const int off = rowoff[m];
        if (off >= 0) yn[(int64_t)c * P.ycs + off * P.yps] = E[m * es + c];
    }
}

template <int CPT>
cudaError_t launch_cpt(const FfmaParams &P, int blocks, cudaStream_t s) {
    const int cpad = 16 * CPT;
    const size_t loop_smem = (size_t)(2 * kBK * kBM + 2 * kBK * cpad) * sizeof(float);
    const size_t epi_smem = (size_t)kBM * (cpad + 1) * sizeof(float);
    const size_t smem = loop_smem > epi_smem ? loop_smem : epi_smem;
    cudaError_t e = cudaFuncSetAttribute(ffma_conv_kernel<CPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    ffma_conv_kernel<CPT><<<blocks, kThreads, smem, s>>>(P);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffma(const convt3d_plan_s &p, const float *x, const float *wpk, const float *bias, float *y,
                        double *partials, int n0, int n1, cudaStream_t s) {
    FfmaParams P;
    memset(&P, 0, sizeof(P));
    P.x = x; P.wpk = wpk; P.bias = bias; P.y = y; P.partials = partials;
    P.N = p.g.N; P.Cin = p.g.Cin; P.cin_pad = p.cin_pad; P.Cout = p.g.Cout; P.cout_pad = p.cout_pad;
    P.Din = p.g.Din; P.Hin = p.g.Hin; P.Win = p.g.Win; P.Do = p.g.Do; P.Ho = p.g.Ho; P.Wo = p.g.Wo;
    P.sd = p.g.ss[0];
    P.sh = p.g.ss[1];
    P.sw = p.g.ss[2];
    const int64_t Sin = (int64_t)p.g.Din * p.g.Hin * p.g.Win, Sout = (int64_t)p.g.Do * p.g.Ho * p.g.Wo;
    P.xcs = p.cl ? 1 : Sin;
    P.xps = p.cl ? p.g.Cin : 1;
    P.ycs = p.cl ? 1 : Sout;
    P.yps = p.cl ? p.g.Cout : 1;
    P.epilogue = p.d.epilogue;
    P.groups = p.d.groups;
    P.scale = p.d.scale;
    P.ngroups = p.ngroups;
    P.tiles_per_sample = p.tiles_per_sample;
    for (int i = 0; i < kMaxGroups; ++i) P.grp[i] = p.grp[i];
    for (int i = 0; i < kMaxClasses; ++i) P.cls[i] = p.g.cls[i];
    for (int i = 0; i < kMaxTaps; ++i) P.taps[i] = p.g.taps[i];
    // one block per tile, the tiles of samples [n0, n1) (tiles are ordered sample by sample)
    P.tile_base = n0 * p.tiles_per_sample;
    const int blocks = (n1 - n0) * p.tiles_per_sample;
    if (blocks <= 0) return cudaSuccess;
    switch (p.cout_pad) {
        case 16: return launch_cpt<1>(P, blocks, s);
        case 32: return launch_cpt<2>(P, blocks, s);
        case 64: return launch_cpt<4>(P, blocks, s);
        case 128: return launch_cpt<8>(P, blocks, s);
        case 256: return launch_cpt<16>(P, blocks, s);
        case 512: return launch_cpt<32>(P, blocks, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace convt3d
