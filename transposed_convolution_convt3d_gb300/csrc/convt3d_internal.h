// Internal definitions shared by the host plan and the kernels of libconvt3d.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "convt3d.h"

namespace convt3d {

constexpr int kMaxClasses = 8;   // stride <= 2  ->  at most 2^3 output-parity classes
constexpr int kMaxGroups = 8;
constexpr int kMaxTaps = 343;    // k <= 7
constexpr int kFfmaTileM = 64;   // output positions per FFMA tile
constexpr int kTcTileM = 128;    // output positions per tensor-core tile (TMEM lanes)
constexpr int kTcChunk = 32;     // fp32 input channels per K step of the tensor-core path (128 B)
constexpr int kTcRowBytes = 128; // bytes of one operand row per K step (the 128-byte swizzle span)
constexpr int kTcStatRows = 4;   // partial-statistics rows per tensor-core tile (one per TMEM lane quarter)
constexpr int kMaxCout = 512;    // output channels: the tensor-memory columns of one accumulator
constexpr int kTcMaxSliceN = 256;  // largest N of one tcgen05.mma (and one TMA box row count)

// 16-bit element kinds of tensors at the boundary and of operand planes.
enum : int { kF32 = 0, kBF16 = 1, kF16 = 2 };

// Element i of a 16-bit array of the given kind (kBF16 or kF16), as fp32.
__device__ __forceinline__ float ld16(const void *p, int64_t i, int kind) {
    const uint16_t b = reinterpret_cast<const uint16_t *>(p)[i];
    return kind == kF16 ? __half2float(__ushort_as_half(b)) : __bfloat162float(__ushort_as_bfloat16(b));
}

// v rounded to nearest even in the given 16-bit kind, as its bit pattern.
__device__ __forceinline__ uint16_t cvt16(float v, int kind) {
    return kind == kF16 ? __half_as_ushort(__float2half_rn(v)) : __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// Two values as one 32-bit pair (a in the low half).
__device__ __forceinline__ uint32_t cvt16x2(float a, float b, int kind) {
    return (uint32_t)cvt16(a, kind) | ((uint32_t)cvt16(b, kind) << 16);
}

__device__ __forceinline__ float2 ld16x2(uint32_t bits, int kind) {
    const uint16_t lo = (uint16_t)(bits & 0xFFFFu), hi = (uint16_t)(bits >> 16);
    if (kind == kF16) return make_float2(__half2float(__ushort_as_half(lo)), __half2float(__ushort_as_half(hi)));
    return make_float2(__bfloat162float(__ushort_as_bfloat16(lo)), __bfloat162float(__ushort_as_bfloat16(hi)));
}

// Status word layout at the start of the workspace.
enum : uint32_t { kErrNone = 0, kErrTimeout = 1, kErrAssert = 2 };
constexpr size_t kStatusBytes = 256;

// One tap of a parity class: input offset along each dimension
// (i = q + delta) and the flat index kd*k*k + kh*k + kw into the weight.
struct TapDesc {
    int8_t dd, dh, dw, pad_;
    int16_t widx, pad2_;
};

// One output-parity class: output positions o = stride*q + r per dimension,
// q in [0, Q).  Its taps are taps[tap_begin .. tap_begin + ntaps).
struct ClassDesc {
    int rd, rh, rw;
    int Qd, Qh, Qw;
    int ntaps, tap_begin;
    int lo_d, lo_h, lo_w;   // smallest delta per dimension
    int nt_d, nt_h, nt_w;   // taps per dimension
    int step_d;             // delta decrease between consecutive d-slices (the d dilation)
};

// Unsigned division by an invariant divisor d >= 1 as a multiply-high, a
// subtract and two shifts, exact for every 32-bit dividend (Granlund and
// Montgomery, "Division by Invariant Integers using Multiplication", 1994,
// their unsigned algorithm with l = ceil(log2 d)).
struct FastDiv {
    uint32_t m;
    uint16_t s1, s2;
};

inline FastDiv make_fastdiv(uint32_t d) {
    int l = 0;
    while (l < 32 && (1ull << l) < d) ++l;
    FastDiv f;
    f.m = (uint32_t)((((1ull << l) - d) << 32) / d + 1);
    f.s1 = (uint16_t)(l < 1 ? l : 1);
    f.s2 = (uint16_t)(l > 1 ? l - 1 : 0);
    return f;
}

__host__ __device__ __forceinline__ uint32_t fastdiv(uint32_t n, FastDiv f) {
#ifdef __CUDA_ARCH__
    const uint32_t t = __umulhi(f.m, n);
#else
    const uint32_t t = (uint32_t)(((uint64_t)f.m * n) >> 32);
#endif
    return (t + ((n - t) >> f.s1)) >> f.s2;
}

// A unit of GEMM work: one class (FFMA, or stride 1), or the two classes
// differing only in w-parity (tensor-core path, stride 2), enumerated over a
// common q-grid of Qd x Qh x Qw positions per sample.
struct GroupDesc {
    int ncls;
    int cls[2];
    int Qd, Qh, Qw;
    int vol;                // Qd*Qh*Qw
    int tiles;              // tiles per sample
    int tile_prefix;        // tiles of earlier groups within one sample
    int ksteps;             // K steps per tile (all classes of the group)
    FastDiv div_qw, div_qhw;  // division by Qw and by Qh * Qw (q-grid position of a row)
    // Merged w-taps of a w-parity pair (tensor-core path): for each distinct w
    // offset, which classes have it (bit c) and the tap's index among class c's
    // w-taps; entries that both classes have come first.
    int nm;
    int8_t mdw[8];
    uint8_t mmask[8];
    int8_t me[8][2];
    // The merged walk flattened (tensor-core launch): K steps step0.. in (d-slice,
    // h-tap, merged w-tap) order, steps_per_a per d-slice, so a tile's trimmed
    // d-slice range is one contiguous run of steps.
    int step0, steps_per_a;
};

// Taps a tile issues.  Along d, a class's taps have decreasing input offsets
// delta = hi, hi - step, ..., hi - (nt_d-1)*step (taps are enumerated d-major in
// increasing kernel index, delta = (r + p - dil*t)/stride, and consecutive taps
// of a class are stride/gcd(stride, dil) apart, so step is the dilation for the
// supported shapes), so the d-slices whose input plane q + delta lies inside
// [0, Din) for some row of the tile form one contiguous range [a0, a1].  The
// tile issues taps [a0 * nhw, (a1+1) * nhw) of the class (nhw = taps per
// d-slice), or just tap 0 when no slice is live -- that zero-filled product
// still initialises the accumulator.
struct TapRange {
    int begin, end;
    int a0, a1;  // the d-slices [a0, a1] (slice 0 alone when none is live)
};

__host__ __device__ inline TapRange tile_taps(const GroupDesc &G, const ClassDesc &C, int t, int tile_m, int Din) {
    const int q0 = t * tile_m;
    const int q1 = (q0 + tile_m < G.vol ? q0 + tile_m : G.vol) - 1;
    const int d0 = (int)fastdiv((uint32_t)q0, G.div_qhw), d1 = (int)fastdiv((uint32_t)q1, G.div_qhw);
    const int step = C.step_d;
    const int hi = C.lo_d + (C.nt_d - 1) * step;  // offset of d-slice 0
    // live slices a: hi + d0 - (Din - 1) <= a * step <= hi + d1
    int a0 = d0 + hi - (Din - 1), a1 = d1 + hi;
    if (step != 1) {
        a0 = a0 > 0 ? (a0 + step - 1) / step : 0;
        a1 = a1 >= 0 ? a1 / step : -1;
    }
    a0 = a0 > 0 ? a0 : 0;
    a1 = a1 < C.nt_d - 1 ? a1 : C.nt_d - 1;
    const int nhw = C.nt_h * C.nt_w;
    TapRange r;
    if (a0 > a1 || C.ntaps == 0) {
        r.begin = 0;
        r.end = C.ntaps > 0 ? 1 : 0;
        r.a0 = r.a1 = 0;
    } else {
        r.begin = a0 * nhw;
        r.end = (a1 + 1) * nhw;
        r.a0 = a0;
        r.a1 = a1;
    }
    return r;
}

struct Geometry {
    int N, Cin, Cout, Din, Hin, Win;
    int kk[3], ss[3], pp[3], op[3], dil[3];  // per dimension (d, h, w): kernel, stride, pad, out pad, dilation
    int kvol;                                // kk[0] * kk[1] * kk[2]
    int G;                                   // convolution groups
    int Do, Ho, Wo;
    int nclasses;
    int ntaps;
    ClassDesc cls[kMaxClasses];
    TapDesc taps[kMaxTaps];
};

// Parameters of the FFMA implicit-GEMM kernel (passed by value).
struct FfmaParams {
    const float *x;
    const float *wpk;       // [ntaps][cin_pad][cout_pad]
    const float *bias;
    float *y;
    double *partials;
    int N, Cin, cin_pad, Cout, cout_pad, Din, Hin, Win, Do, Ho, Wo, sd, sh, sw;
    int64_t xcs, xps, ycs, yps;  // element strides of a channel and of a position within a sample (x, y)
    int epilogue, groups;
    float scale;
    int ngroups, tiles_per_sample;
    int tile_base;           // this launch's first tile (block b runs tile tile_base + b)
    GroupDesc grp[kMaxGroups];
    ClassDesc cls[kMaxClasses];
    TapDesc taps[kMaxTaps];
};

}  // namespace convt3d

struct convt3d_plan_s {
    convt3d_desc_t d;
    convt3d::Geometry g;
    int tc;                 // 1: tensor-core path, 0: FFMA
    int direct;             // tensor-core path reading NCDHW fp32 x directly (no staged copy; direct.cu)
    int planes;             // tensor-core operand planes: 2 = split TF32 (hi, lo), 1 = TF32 or BF16
    int cl;                 // channels-last x and y (NDHWC)
    int io16;               // x, w and y are 16-bit arrays: kBF16 or kF16 (0: fp32)
    int merged;             // w-parity pairs share activation loads and MMAs (see GroupDesc::nm)
    int bf16;               // tensor-core operands are 16-bit (kind::f16 MMA): bf16, or fp16 when half
    int half;               // the 16-bit operands are fp16
    int chunk;              // input channels per K step (one 128-byte operand row)
    int elem_bytes;         // bytes per staged / packed operand element
    int cin_pad, cout_pad;
    int nslices;            // tensor-core path: N slices of cout_pad / nslices (<= 256) columns per tile
    int tile_m;
    int ngroups;
    convt3d::GroupDesc grp[convt3d::kMaxGroups];
    int tiles_per_sample;
    int64_t tiles;
    int stat_rows_per_tile;  // partial-statistics rows each tile writes (tensor-core: one per epilogue warp)
    int bn_splits;           // BatchNorm: row ranges per sample the first reduction splits into
    // workspace layout (byte offsets, 256-aligned)
    size_t off_wpk_hi, off_wpk_lo, off_xs_hi, off_xs_lo, off_partials, off_stats, ws_total;
    size_t wpk_elems, xs_elems, partial_doubles, stat_doubles;
    // GEMM timing
    int prof_enabled;
    int prof_valid;
    cudaEvent_t ev0, ev1;
    int ev_created;
    const void *packed_ws;  // workspace that pack_weights last filled for this plan
    void *tc_cache;         // tensor-core launch state (tc.cu)
    void *direct_cache;     // direct-input tensor-core launch state (direct.cu)
    float *run_mean;        // BatchNorm running statistics (device, Cout each) or NULL
    float *run_var;
    float momentum;
    size_t off_box;         // evaluation-mode BatchNorm: per-tap input box sums
    int ev_ks;              // evaluation-mode BatchNorm: K splits of the contraction (1 = none)
    size_t off_evpart;      //   fp64 partial sums [ks][n][c] when ev_ks > 1
    size_t off_evcnt;       //   per (c, sample block) arrival counters, zeroed by pack_weights
};

// Kernel launchers (defined in the .cu files); each returns cudaGetLastError().
namespace convt3d {
cudaError_t launch_pack_weights(const convt3d_plan_s &p, const float *w, float *hi, float *lo,
                                int kmajor, cudaStream_t s);
// The per-sample launches take the samples [n0, n1) of the batch (all of it: 0, N).
cudaError_t launch_stage_input(const convt3d_plan_s &p, const float *x, float *hi, float *lo, int n0, int n1,
                               cudaStream_t s);
cudaError_t launch_ffma(const convt3d_plan_s &p, const float *x, const float *wpk, const float *bias,
                        float *y, double *partials, int n0, int n1, cudaStream_t s);
cudaError_t launch_tc(convt3d_plan_s &p, const float *xs_hi, const float *xs_lo,
                      const float *w_hi, const float *w_lo, const float *bias, float *y,
                      double *partials, uint32_t *status, int n0, int n1, cudaStream_t s);
cudaError_t launch_gn_finalize(const convt3d_plan_s &p, const double *partials, double *stats,
                               cudaStream_t s);
cudaError_t launch_gn_normalize(const convt3d_plan_s &p, const double *stats, const float *gamma,
                                const float *beta, const float *bias, float *y, cudaStream_t s);
cudaError_t launch_bn_finalize(const convt3d_plan_s &p, const double *partials, double *sums,
                               const float *gamma, const float *beta, float *y, cudaStream_t s);
cudaError_t launch_bn_eval(const convt3d_plan_s &p, const float *x, const float *w_a, const float *w_b,
                           const float *bias, const float *gamma, const float *beta, float *box, double *part,
                           unsigned *counters, float *y, cudaStream_t s);
size_t bn_eval_smem_bytes(const convt3d_plan_s &p);
int bn_eval_ksplits(int ntaps, int Cin);
void tc_cache_free(void *cache);
cudaError_t launch_direct(convt3d_plan_s &p, const float *x, const void *wdir, const float *bias, float *y,
                          uint32_t *status, cudaStream_t s);
cudaError_t launch_direct_pack(convt3d_plan_s &p, const float *w, void *dst, cudaStream_t s);
bool direct_supported(const convt3d_plan_s &p);
size_t direct_weight_bytes(const convt3d_plan_s &p);
void direct_cache_free(void *cache);
void *static_workspace_address();
void report_error(const char *fmt, ...);
}  // namespace convt3d
