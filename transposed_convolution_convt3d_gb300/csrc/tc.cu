// Tensor-core implicit GEMM for the transposed convolution: tcgen05 MMA in
// split TF32 ("3xTF32": a_hi*b_hi + a_hi*b_lo + a_lo*b_hi, fp32 accumulation
// in tensor memory), single TF32 (one product of TF32-rounded operands) or
// BF16 (kind::f16, one product of bf16 operands, 64 channels per 128-byte
// row), TMA-fed, with the epilogues fused.
//
// GEMM view (output-stationary): M = output positions of one parity class,
// N = Cout, K = Cin x taps of that class.  A 128-row tile is 128 consecutive
// positions of the class's q-grid within one sample; for each K step
// (tap, 32 input channels) the TMA im2col unit gathers the 128 x 32 activation
// slice straight from the channels-last staged input (input index
// i = q + delta per dimension; out-of-range pixels arrive as zeros), and a
// tiled TMA load brings the Cout x 32 weight slice.  Both land K-major with the
// 128-byte (or, for 16-channel steps, 64-byte) swizzle that the tcgen05
// shared-memory descriptors describe.
// With stride 2 along w the two classes that differ only in w-parity share a CTA tile
// (two accumulators), so the identity and ReLU epilogues write each output
// row as contiguous pairs.
//
// CTA roles (persistent, one CTA per SM):
//   warp 0      TMA producer (one thread): fills a ring of shared-memory stages
//   warp 1      MMA issuer (one thread) + tensor-memory allocation
//   warps 2..   epilogue, one warp per tensor-memory lane quarter (two for
//               softmax+sigmoid, splitting the channels): tensor memory ->
//               registers -> fused epilogue -> HBM
// Accumulators are double-buffered in tensor memory so the epilogue of one
// tile overlaps the main loop of the next.  Every wait is bounded; a wait that
// runs out records CONVT3D_ERR_TIMEOUT in the workspace status word, all roles
// drain and the kernel returns.
#include <stdio.h>
#include <string.h>

#include <new>

#include <cuda_bf16.h>

#include "convt3d_internal.h"
#include "epimath.cuh"
#include "ptx.cuh"

// Order of the per-dimension arrays the TMA im2col interfaces take.
#ifndef CONVT3D_CORNERS_DHW
#define CONVT3D_CORNERS_DHW 0
#endif
#ifndef CONVT3D_OFFSETS_DHW
#define CONVT3D_OFFSETS_DHW 0
#endif

// Epilogue warps of the softmax kernel: 4, 8 or 16 (1, 2 or 4 per lane quarter).
#ifndef CONVT3D_SOFTMAX_EPI_WARPS
#define CONVT3D_SOFTMAX_EPI_WARPS 8
#endif

namespace convt3d {
namespace {

// Epilogue warps per CTA: softmax+sigmoid is arithmetic-heavy and gets two warps
// per tensor-memory lane quarter (each taking half of the channels); the other
// epilogues use one, which leaves the producer and MMA warps more issue slots.
template <int EPI>
struct EpiCfg {
    static constexpr int warps = EPI == CONVT3D_EPI_SOFTMAX_SIGMOID ? CONVT3D_SOFTMAX_EPI_WARPS : 4;
    static constexpr int threads = 64 + 32 * warps;  // producer warp, MMA warp, epilogue warps
};

// Softmax: 16-channel chunks per epilogue warp whose exponentials stay in
// registers between the sum and the output pass (the register budget per
// thread halves when the warp count doubles).
constexpr int kSoftmaxKeepChunks = CONVT3D_SOFTMAX_EPI_WARPS >= 16 ? 1 : 2;

// Shared-memory floats of the softmax (max, sum) exchange between the warps of a
// lane quarter: 2 buffers x warps per quarter x (2 classes x 2 values) x 128 rows.
template <int EPI>
constexpr int sm_exchange_floats() {
    return EPI == CONVT3D_EPI_SOFTMAX_SIGMOID && EpiCfg<EPI>::warps > 4 ? 2 * (EpiCfg<EPI>::warps / 4) * 4 * kTcTileM
                                                                      : 1;
}
constexpr int kMaxStages = 8;  // the MMA issue dispatches stage indices 0..7
// Longest accumulation chain of one tensor-memory accumulator, in K steps (32 fp32 /
// 64 bf16 channels x 12 MMAs each): about 770 roundings of the fp32 accumulator.
constexpr int kSegSteps = 64;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait
// Input channels per K step: 32 (128-byte rows, 128-byte swizzle) or 16
// (64-byte rows, 64-byte swizzle: half-size stages, twice as many of them).
#ifndef CONVT3D_TC_KCHUNK
#define CONVT3D_TC_KCHUNK 32
#endif
constexpr int kChunk = CONVT3D_TC_KCHUNK;
static_assert(kChunk == 16 || kChunk == 32, "K step must be 16 or 32 channels");
static_assert(kTcChunk % kChunk == 0, "channel padding must be a multiple of the K step");
constexpr uint32_t kRowBytes = kChunk * 4;
constexpr uint32_t kABytes = kTcTileM * kRowBytes;  // one 128 x kChunk fp32 activation plane

// One K step of a merged w-parity walk: which class's activation slice (0 or 1
// within the pair) at offsets (od, oh, ow) from the class's low corner, the
// weight slices of taps tb0 and (both classes) tb1, and the classes it feeds.
struct StepDesc {
    int16_t tb0, tb1;  // tb1 < 0: one class
    uint8_t cls, mask, ow, oh;
    uint8_t od, pad_[3];
};
// The pairs' walks hold sum over (rd, rh) of nt_d(rd) * nt_h(rh) * nm steps; every
// tap lies in exactly one parity class per dimension, so that is kd * kh * nm with
// nm (distinct w offsets) <= kw: at most 7 * 7 * 7 for the largest kernel.
constexpr int kMaxSteps = 512;
static_assert(kMaxSteps >= 7 * 7 * 7, "step table smaller than the largest merged walk");

struct TcParams {
    CUtensorMap a_hi[kMaxClasses];
    CUtensorMap a_lo[kMaxClasses];
    CUtensorMap b_hi;
    CUtensorMap b_lo;
    const float *bias;
    float *y;
    double *partials;
    uint32_t *status;
    int N, Cout, cout_pad, Do, Ho, Wo, sd, sh, sw, kc;
    int Din, Hin, Win;
    int epilogue, groups;
    float scale;
    int ngroups, tiles_per_sample, total_tiles;
    int tile_begin, tile_end;  // this launch's tiles (a range of whole samples; all of them by default)
    FastDiv div_tps;  // division by tiles_per_sample
    int stages;
    uint32_t stage_bytes, b_bytes;
    int planes;  // 2: split TF32 (A and B hi/lo), 1: single TF32 or BF16
    int cl;      // channels-last output
    int io16;    // y is a 16-bit array: kBF16 or kF16 (0: fp32)
    int bf16;    // operands are 16-bit (kind::f16 MMA)
    int half;    // the 16-bit operands are fp16 (else bf16)
    int chunk;   // input channels per K step (one 128-byte row)
    int nslices, slice_n;  // N slices per tile (Cout_pad > 256: each slice's K walk fills its own columns)
    int nbuf;              // accumulators in tensor memory: 2 (double-buffered) or 1
    int seg_steps;         // long K walks: steps per accumulation segment (SEG kernels)
    uint32_t sum_col;      // tensor-memory column of the segments' running sums (SEG kernels)
    uint32_t tmem_cols, acc_stride;
    GroupDesc grp[kMaxGroups];
    ClassDesc cls[kMaxClasses];
    TapDesc taps[kMaxTaps];
    StepDesc steps[kMaxSteps];  // merged walks (MERGED kernels)
};

struct Tile {
    int gi, n, t, slot;
};

// Tile index -> (group, sample, tile within the sample's q-grid).  Tiles are
// ordered sample by sample, then group by group (heaviest first), then tile:
// the parity groups of a stride-2 problem all read the same input planes, and
// finishing one sample's groups together keeps those planes in L2 between
// them (group-major order re-read the whole input once per group).  `grp` is
// the shared-memory copy of the group table.
__device__ __forceinline__ Tile decode(const TcParams &P, const GroupDesc *grp, int tile) {
    Tile r;
    r.n = (int)fastdiv((uint32_t)tile, P.div_tps);
    const int rem = tile - r.n * P.tiles_per_sample;
    int gi = 0;
    while (gi + 1 < P.ngroups && rem >= grp[gi + 1].tile_prefix) ++gi;
    r.gi = gi;
    r.t = rem - grp[gi].tile_prefix;
    r.slot = tile;
    return r;
}

__device__ __forceinline__ void record_error(uint32_t *status, uint32_t code, uint32_t site) {
    if (atomicCAS(status, 0u, code) == 0u) {
        status[1] = site;
        status[2] = blockIdx.x;
    }
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Statistics partial of values spread over the warp's lanes, written as
// (count n, sum S, M2 = sum of squared deviations from S / n) in fp64.  The
// lanes hold fp32 sums about a common shift c close to the values' mean --
// s1 = sum (v - c), s2 = sum (v - c)^2 over cnt values -- so no large common
// offset enters any fp32 sum, and the butterfly reductions stay in fp32 (this
// GPU's fp64 rate is a small fraction of its fp32 rate): M2 = sum s2 - (sum s1)^2 / n
// needs no more, and only S = n c + sum s1, whose terms differ in magnitude, is
// formed in fp64 (one fused multiply-add on one lane).
__device__ __forceinline__ void warp_moments(float s1, float s2, int n, float c, double *out) {
    // n: the warp's value count (the same in every lane)
    const float t1 = warp_sum_f(s1);
    const float t2 = warp_sum_f(s2);
    if ((threadIdx.x & 31) == 0) {
        out[0] = (double)n;
        out[1] = fma((double)n, (double)c, (double)t1);
        out[2] = n > 0 ? (double)fmaxf(t2 - t1 * t1 * __frcp_rn((float)n), 0.f) : 0.0;
    }
}

// Per-channel sums over the 32 lanes for 16 channels held by every lane:
// five butterfly stages that halve the channel count held per lane; lane l
// ends with the full sum of channel (l >> 1).
__device__ __forceinline__ float transpose_reduce16(const float (&v)[16], int lane) {
    float a[8];
    {
        const bool hi = lane & 16;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float send = hi ? v[i] : v[i + 8];
            const float keep = hi ? v[i + 8] : v[i];
            a[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
    }
    float b[4];
    {
        const bool hi = lane & 8;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float send = hi ? a[i] : a[i + 4];
            const float keep = hi ? a[i + 4] : a[i];
            b[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
    }
    float c[2];
    {
        const bool hi = lane & 4;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float send = hi ? b[i] : b[i + 2];
            const float keep = hi ? b[i + 2] : b[i];
            c[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
    }
    float d;
    {
        const bool hi = lane & 2;
        const float send = hi ? c[0] : c[1];
        const float keep = hi ? c[1] : c[0];
        d = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    return d + __shfl_xor_sync(0xffffffffu, d, 1);
}

// Pairwise maximum of 16 values (4 dependent levels instead of 15).
__device__ __forceinline__ float tree_max16(const float (&v)[16]) {
    float a[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = fmaxf(v[i], v[i + 8]);
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = fmaxf(a[i], a[i + 4]);
    return fmaxf(fmaxf(a[0], a[2]), fmaxf(a[1], a[3]));
}

// Classes (0, 1 or 2) whose row is inside the output, from the two row offsets.
__device__ __forceinline__ int valid_rows(const int (&off)[2], int ncls) {
    return (off[0] >= 0 ? 1 : 0) + (ncls > 1 && off[1] >= 0 ? 1 : 0);
}

// Position of epilogue row m of a tile for one class: output offset within a
// channel plane, or -1 when the row lies past the q-grid or the output.
__device__ __forceinline__ int row_offset(const TcParams &P, const GroupDesc &G, const ClassDesc &C, int t, int m) {
    const int q = t * kTcTileM + m;
    if (q >= G.vol) return -1;
    const int qd = (int)fastdiv((uint32_t)q, G.div_qhw);
    const int r = q - qd * (G.Qh * G.Qw);
    const int qh = (int)fastdiv((uint32_t)r, G.div_qw);
    const int od = P.sd * qd + C.rd;
    const int oh = P.sh * qh + C.rh;
    const int ow = P.sw * (r - qh * G.Qw) + C.rw;
    if (od >= P.Do || oh >= P.Ho || ow >= P.Wo) return -1;
    return (od * P.Ho + oh) * P.Wo + ow;
}

// Long reductions (SEG kernels, non-merged tiles).  The tensor cores round the
// fp32 accumulator once per MMA, and the error of a chain of such roundings grows
// with its length relative to the accumulated value; so a tile whose K walk
// (class 0's steps, then class 1's) exceeds seg_steps is split into nseg
// near-equal segments, each accumulated from zero in an accumulator buffer of its
// own, and the epilogue adds the segments' partial sums in fp32 into a running sum
// in tensor memory (sum_col).  The MMA thread and the epilogue derive the same plan.
struct SegPlan {
    int n[2];  // K steps of class 0 and class 1
    int total, nseg, len;
};

__device__ __forceinline__ SegPlan seg_plan(const TcParams &P, const GroupDesc &G, const ClassDesc *cls, int t) {
    SegPlan sp;
    sp.total = 0;
#pragma unroll
    for (int ci = 0; ci < 2; ++ci) {
        sp.n[ci] = 0;
        if (ci < G.ncls) {
            const TapRange tr = tile_taps(G, cls[G.cls[ci]], t, kTcTileM, P.Din);
            sp.n[ci] = (tr.end - tr.begin) * P.kc;
        }
        sp.total += sp.n[ci];
    }
    sp.nseg = sp.total > P.seg_steps ? (sp.total + P.seg_steps - 1) / P.seg_steps : 1;
    sp.len = (sp.total + sp.nseg - 1) / sp.nseg;
    return sp;
}

// Does class ci have K steps in [a, b) of the tile's walk?
__device__ __forceinline__ bool seg_touches(const SegPlan &sp, int ci, int a, int b) {
    const int b0 = ci == 0 ? 0 : sp.n[0];
    return sp.n[ci] > 0 && b0 < b && b0 + sp.n[ci] > a;
}

// KEEP (softmax only): 1 = each epilogue warp keeps its exponentials in
// registers (Cout <= 16 * kSoftmaxKeepChunks * warps per lane quarter); 2 = as
// 1, for w-parity pairs with each warp owning one class's channels (8 warps);
// 0 = the exponentials are recomputed from tensor memory.
// OPS: operand format, fixed at compile time so that the producer and MMA
// loops stay branch-free: 0 = split TF32 (hi and lo planes), 1 = TF32, 2 = BF16,
// 3 = split BF16 (hi and lo bf16 planes).
// MERGED: every group is a w-parity pair walked by merged w-taps (GroupDesc::nm):
// a K step whose w offset both classes have loads the activation slice once,
// the two classes' weight slices side by side, and issues one MMA of
// N = 2 * Cout_pad into both accumulators (they are adjacent in tensor memory).
// SEG: long K walks are accumulated in segments (see SegPlan); split formats only.
template <int EPI, int KEEP, int OPS, bool MERGED, bool SEG = false>
__global__ void __launch_bounds__(EpiCfg<EPI>::threads, 1) convt3d_tc_gemm(const __grid_constant__ TcParams P) {
    constexpr int kPlanes = (OPS == 0 || OPS == 3) ? 2 : 1;
    constexpr int kBSlots = MERGED ? 2 : 1;  // weight slices per plane in a stage
    constexpr int kEpiWarps = EpiCfg<EPI>::warps;
    constexpr int kHalves = kEpiWarps / 4;  // warps per tensor-memory lane quarter
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[2 * kMaxStages + 5];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    __shared__ float s_bias[kMaxCout];                     // bias, zero-padded to kMaxCout channels
    __shared__ __align__(16) float s_bias_l2e[kMaxCout];   // bias * log2(e) (softmax)
    __shared__ float s_xchg[sm_exchange_floats<EPI>()];   // softmax (max, sum) exchange, double-buffered
    // The group and class tables (and, for merged walks, the step table) in shared
    // memory: the producer and MMA threads index them per tile and per K step, and
    // an indexed read of the kernel parameters would go through the constant cache.
    __shared__ GroupDesc s_grp[kMaxGroups];
    __shared__ ClassDesc s_cls[kMaxClasses];
    __shared__ StepDesc s_steps[MERGED ? kMaxSteps : 1];

    // 1024-byte aligned ring of pipeline stages
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t full0 = ptx::smem_u32(&bars[0]);
    const uint32_t empty0 = ptx::smem_u32(&bars[kMaxStages]);
    const uint32_t tfull0 = ptx::smem_u32(&bars[2 * kMaxStages]);
    const uint32_t tempty0 = ptx::smem_u32(&bars[2 * kMaxStages + 2]);
    const uint32_t drain = ptx::smem_u32(&bars[2 * kMaxStages + 4]);
    const uint32_t smem_base = ptx::smem_u32(smem);

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < P.stages; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(tfull0 + 8 * a, 1);
            ptx::mbar_init(tempty0 + 8 * a, kEpiWarps * 32);
        }
        ptx::mbar_init(drain, 1);
        ptx::fence_mbar_init();
    }
    for (int c = threadIdx.x; c < kMaxCout; c += blockDim.x) {
        s_bias[c] = (P.bias && c < P.Cout) ? P.bias[c] : 0.f;
        s_bias_l2e[c] = s_bias[c] * kLog2e;
    }
    if (threadIdx.x < kMaxGroups) s_grp[threadIdx.x] = P.grp[threadIdx.x];
    if (threadIdx.x < kMaxClasses) s_cls[threadIdx.x] = P.cls[threadIdx.x];
    if constexpr (MERGED)
        for (int i = threadIdx.x; i < kMaxSteps; i += blockDim.x) s_steps[i] = P.steps[i];
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), P.tmem_cols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = tmem_slot;

    // ------------------------------------------------------------ producer
    // The producer and MMA loops read only the kernel parameters and loop
    // counters, so their control flow stays uniform; the MMA issue rate depends
    // on it.
    if (warp == 0) {
        if (lane == 0) {
            for (int gi = 0; gi < P.ngroups; ++gi)
                for (int ci = 0; ci < P.grp[gi].ncls; ++ci) {
                    ptx::prefetch_tmap(&P.a_hi[P.grp[gi].cls[ci]]);
                    if (kPlanes == 2) ptx::prefetch_tmap(&P.a_lo[P.grp[gi].cls[ci]]);
                }
            ptx::prefetch_tmap(&P.b_hi);
            if (kPlanes == 2) ptx::prefetch_tmap(&P.b_lo);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_phase = 0;  // per-stage bits: armed at least once, last armed parity
            bool ok = true;
            // One K step per input-channel chunk of one tap: the activation slice of
            // class `cls` at tap `td`, the weight slice of tap tb0 and, merged, of tap tb1.
            auto issue_tap = [&](const Tile &T, int cls, const ClassDesc &C, int qd0, int qh0, int qw0,
                                 const TapDesc td, int tb0, int tb1, int row0) {
                const int w0 = qw0 + C.lo_w, h0 = qh0 + C.lo_h, d0 = qd0 + C.lo_d;
                const uint16_t ow = (uint16_t)(td.dw - C.lo_w);
                const uint16_t oh = (uint16_t)(td.dh - C.lo_h);
                const uint16_t od = (uint16_t)(td.dd - C.lo_d);
                const uint32_t nb = tb1 >= 0 ? 2u : 1u;
                for (int kc = 0; kc < P.kc; ++kc) {
                    if (!ptx::mbar_wait_bounded(empty0 + 8 * stage, phase ^ 1u, &abort_flag, kWaitNs)) {
                        ok = false;
                        return;
                    }
                    const uint32_t fb = full0 + 8 * stage;
                    const uint32_t sb = smem_base + (uint32_t)stage * P.stage_bytes;
                    // stage layout: A_hi [A_lo] B_hi(slot 0 [, slot 1]) [B_lo(slot 0 [, slot 1])]
                    ptx::mbar_arrive_expect_tx(fb, (uint32_t)kPlanes * (kABytes + nb * P.b_bytes));
                    const int c0 = kc * P.chunk;
                    const uint32_t sbb = sb + (uint32_t)kPlanes * kABytes;
#if CONVT3D_OFFSETS_DHW
                    ptx::tma_load_im2col_5d(sb, &P.a_hi[cls], fb, c0, w0, h0, d0, T.n, od, oh, ow);
                    if (kPlanes == 2)
                        ptx::tma_load_im2col_5d(sb + kABytes, &P.a_lo[cls], fb, c0, w0, h0, d0, T.n, od, oh, ow);
#else
                    ptx::tma_load_im2col_5d(sb, &P.a_hi[cls], fb, c0, w0, h0, d0, T.n, ow, oh, od);
                    if (kPlanes == 2)
                        ptx::tma_load_im2col_5d(sb + kABytes, &P.a_lo[cls], fb, c0, w0, h0, d0, T.n, ow, oh, od);
#endif
                    ptx::tma_load_3d(sbb, &P.b_hi, fb, c0, row0, tb0);
                    if (MERGED && tb1 >= 0) ptx::tma_load_3d(sbb + P.b_bytes, &P.b_hi, fb, c0, row0, tb1);
                    if (kPlanes == 2) {
                        const uint32_t lo = sbb + (uint32_t)kBSlots * P.b_bytes;
                        ptx::tma_load_3d(lo, &P.b_lo, fb, c0, row0, tb0);
                        if (MERGED && tb1 >= 0) ptx::tma_load_3d(lo + P.b_bytes, &P.b_lo, fb, c0, row0, tb1);
                    }
                    armed |= 1u << stage;
                    armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
                    if (++stage == P.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            };
            for (int tile = P.tile_begin + blockIdx.x; ok && tile < P.tile_end; tile += gridDim.x) {
                const Tile T = decode(P, s_grp, tile);
                const GroupDesc &G = s_grp[T.gi];
                const int q0 = T.t * kTcTileM;
                const int qd0 = (int)fastdiv((uint32_t)q0, G.div_qhw);
                const int qhw = (int)fastdiv((uint32_t)q0, G.div_qw);  // q0 / Qw
                const int qh0 = qhw - qd0 * G.Qh, qw0 = q0 - qhw * G.Qw;
                if constexpr (MERGED) {
                    // the tile's run of the flattened walk (d-slices: the same for both classes)
                    const ClassDesc &C0 = s_cls[G.cls[0]], &C1 = s_cls[G.cls[1]];
                    const TapRange tr = tile_taps(G, C0, T.t, kTcTileM, P.Din);
                    const int a_begin = tr.a0, a_end = tr.a1 + 1;
                    const int s_end = G.step0 + a_end * G.steps_per_a;
                    // each class's base pixel of the tile
                    const int w00 = qw0 + C0.lo_w, h00 = qh0 + C0.lo_h, d00 = qd0 + C0.lo_d;
                    const int w01 = qw0 + C1.lo_w, h01 = qh0 + C1.lo_h, d01 = qd0 + C1.lo_d;
                    for (int st = G.step0 + a_begin * G.steps_per_a; ok && st < s_end; ++st) {
                        const StepDesc e = s_steps[st];
                        const bool one = e.cls != 0;
                        const int cls = one ? G.cls[1] : G.cls[0];
                        const int w0 = one ? w01 : w00, h0 = one ? h01 : h00, d0 = one ? d01 : d00;
                        const uint32_t nb = e.tb1 >= 0 ? 2u : 1u;
                        for (int kc = 0; kc < P.kc; ++kc) {
                            if (!ptx::mbar_wait_bounded(empty0 + 8 * stage, phase ^ 1u, &abort_flag, kWaitNs)) {
                                ok = false;
                                break;
                            }
                            const uint32_t fb = full0 + 8 * stage;
                            const uint32_t sb = smem_base + (uint32_t)stage * P.stage_bytes;
                            ptx::mbar_arrive_expect_tx(fb, (uint32_t)kPlanes * (kABytes + nb * P.b_bytes));
                            const int c0 = kc * P.chunk;
                            const uint32_t sbb = sb + (uint32_t)kPlanes * kABytes;
#if CONVT3D_OFFSETS_DHW
                            ptx::tma_load_im2col_5d(sb, &P.a_hi[cls], fb, c0, w0, h0, d0, T.n, e.od, e.oh, e.ow);
                            if (kPlanes == 2)
                                ptx::tma_load_im2col_5d(sb + kABytes, &P.a_lo[cls], fb, c0, w0, h0, d0, T.n, e.od, e.oh,
                                                        e.ow);
#else
                            ptx::tma_load_im2col_5d(sb, &P.a_hi[cls], fb, c0, w0, h0, d0, T.n, e.ow, e.oh, e.od);
                            if (kPlanes == 2)
                                ptx::tma_load_im2col_5d(sb + kABytes, &P.a_lo[cls], fb, c0, w0, h0, d0, T.n, e.ow, e.oh,
                                                        e.od);
#endif
                            ptx::tma_load_3d(sbb, &P.b_hi, fb, c0, 0, e.tb0);
                            if (e.tb1 >= 0) ptx::tma_load_3d(sbb + P.b_bytes, &P.b_hi, fb, c0, 0, e.tb1);
                            if (kPlanes == 2) {
                                const uint32_t lo = sbb + (uint32_t)kBSlots * P.b_bytes;
                                ptx::tma_load_3d(lo, &P.b_lo, fb, c0, 0, e.tb0);
                                if (e.tb1 >= 0) ptx::tma_load_3d(lo + P.b_bytes, &P.b_lo, fb, c0, 0, e.tb1);
                            }
                            armed |= 1u << stage;
                            armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
                            if (++stage == P.stages) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                    }
                } else {
                    for (int ci = 0; ok && ci < G.ncls; ++ci) {
                        const int cls = G.cls[ci];
                        const ClassDesc &C = s_cls[cls];
                        const TapRange tr = tile_taps(G, C, T.t, kTcTileM, P.Din);
                        for (int sl = 0; ok && sl < P.nslices; ++sl)  // the same activation walk per N slice
                            for (int j = tr.begin; ok && j < tr.end; ++j)
                                issue_tap(T, cls, C, qd0, qh0, qw0, P.taps[C.tap_begin + j], C.tap_begin + j, -1,
                                          sl * P.slice_n);
                    }
                }
            }
            if (!ok) {
                record_error(P.status, kErrTimeout, 1);
                abort_flag = 1;
            }
            // Drain: every load this thread issued has landed before the CTA may exit.
            for (int s = 0; s < P.stages; ++s)
                if (armed & (1u << s)) {
                    const volatile int never = 0;
                    ptx::mbar_wait_bounded(full0 + 8 * s, (armed_phase >> s) & 1u, &never, 200000000ull);
                }
        }
    }
    // ---------------------------------------------------------- MMA issuer
    else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = OPS >= 2 ? (P.half ? ptx::idesc_f16((uint32_t)P.slice_n)
                                                      : ptx::idesc_bf16((uint32_t)P.slice_n))
                                            : ptx::idesc_tf32((uint32_t)P.slice_n);
            // merged steps of both classes: N = 2 * Cout_pad
            const uint32_t idesc2 =
                OPS >= 2 ? (P.half ? ptx::idesc_f16(2u * (uint32_t)P.cout_pad) : ptx::idesc_bf16(2u * (uint32_t)P.cout_pad))
                         : ptx::idesc_tf32(2u * (uint32_t)P.cout_pad);
            constexpr uint64_t kA16 = kABytes >> 4;                  // one activation plane, 16-byte units
            const uint64_t b16 = (uint64_t)(P.b_bytes >> 4);         // one weight slice
            const uint64_t blo16 = (uint64_t)kBSlots * b16;          // B_lo after the B_hi slots
            int stage = 0;
            uint32_t phase = 0;
            int iter = 0;
            bool ok = true;
            // The K steps of one tap; `init`: the first product overwrites the accumulator(s).
            auto mma_tap = [&](uint32_t d_tmem, uint32_t id, bool init) {
                for (int kc = 0; kc < P.kc; ++kc) {
                    if (!ptx::mbar_wait_bounded(full0 + 8 * stage, phase, &abort_flag, kWaitNs)) {
                        ok = false;
                        return;
                    }
                    ptx::tc_fence_after();
                    // One descriptor per stage; the others differ only in the start-address
                    // field (16-byte units), which never carries out of its 14 bits here.
                    const uint64_t d0 = ptx::sdesc_k_swizzled(smem_base + (uint32_t)stage * P.stage_bytes, kRowBytes);
                    const uint32_t first = (init && kc == 0) ? 0u : 1u;
                    if constexpr (OPS == 0) {
#pragma unroll
                        for (int kk = 0; kk < kChunk / 8; ++kk) {  // 8 TF32 (32 bytes) per MMA
                            const uint64_t a_hi = d0 + 2 * kk;
                            const uint64_t a_lo = a_hi + kA16;
                            const uint64_t b_hi = a_hi + 2 * kA16;
                            const uint64_t b_lo = b_hi + blo16;
                            ptx::mma_tf32(d_tmem, a_hi, b_hi, id, kk ? 1u : first);
                            ptx::mma_tf32(d_tmem, a_hi, b_lo, id, 1u);
                            ptx::mma_tf32(d_tmem, a_lo, b_hi, id, 1u);
                        }
                    } else if constexpr (OPS == 2) {
#pragma unroll
                        for (int kk = 0; kk < kChunk / 8; ++kk) {  // 16 bf16 (32 bytes) per MMA
                            const uint64_t a = d0 + 2 * kk;
                            ptx::mma_bf16(d_tmem, a, a + kA16, id, kk ? 1u : first);
                        }
                    } else if constexpr (OPS == 3) {
#pragma unroll
                        for (int kk = 0; kk < kChunk / 8; ++kk) {  // split bf16: three products
                            const uint64_t a_hi = d0 + 2 * kk;
                            const uint64_t a_lo = a_hi + kA16;
                            const uint64_t b_hi = a_hi + 2 * kA16;
                            const uint64_t b_lo = b_hi + blo16;
                            ptx::mma_bf16(d_tmem, a_hi, b_hi, id, kk ? 1u : first);
                            ptx::mma_bf16(d_tmem, a_hi, b_lo, id, 1u);
                            ptx::mma_bf16(d_tmem, a_lo, b_hi, id, 1u);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < kChunk / 8; ++kk) {
                            const uint64_t a = d0 + 2 * kk;
                            ptx::mma_tf32(d_tmem, a, a + kA16, id, kk ? 1u : first);
                        }
                    }
                    ptx::mma_commit(empty0 + 8 * stage);
                    if (++stage == P.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            };
            for (int tile = P.tile_begin + blockIdx.x; ok && tile < P.tile_end; tile += gridDim.x, ++iter) {
                const Tile T = decode(P, s_grp, tile);
                const GroupDesc &G = s_grp[T.gi];
                int acc = P.nbuf == 2 ? (iter & 1) : 0;
                const uint32_t aph = (uint32_t)(P.nbuf == 2 ? iter >> 1 : iter) & 1u;
                if (!ptx::mbar_wait_bounded(tempty0 + 8 * acc, aph ^ 1u, &abort_flag, kWaitNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                uint32_t acc_base = tmem_base + (uint32_t)acc * P.acc_stride;
                if constexpr (MERGED) {
                    // same walk as the producer; shared offsets come first, so a merged step
                    // never meets one accumulator initialised and the other not
                    const ClassDesc &C0 = s_cls[G.cls[0]];
                    const TapRange tr = tile_taps(G, C0, T.t, kTcTileM, P.Din);
                    const int a_begin = tr.a0, a_end = tr.a1 + 1;
                    const int s_end = G.step0 + a_end * G.steps_per_a;
                    uint32_t ini = 0;  // bit c: class c's accumulator holds a product
                    for (int st = G.step0 + a_begin * G.steps_per_a; ok && st < s_end; ++st) {
                        const uint32_t mask = s_steps[st].mask;
                        const uint32_t d_tmem = acc_base + (mask == 2u ? (uint32_t)P.cout_pad : 0u);
                        mma_tap(d_tmem, mask == 3u ? idesc2 : idesc, (ini & mask) == 0u);
                        ini |= mask;
                    }
                } else if constexpr (SEG) {
                    // the tile's walk in segments: at each segment boundary the finished
                    // accumulator goes to the epilogue and the next segment starts from zero
                    // in the other buffer; within a segment, each class's steps run as one
                    // flat loop like the unsegmented walk's
                    const SegPlan sp = seg_plan(P, G, s_cls, T.t);
                    for (int sg = 0; ok && sg < sp.nseg; ++sg) {
                        if (sg > 0) {
                            ptx::mma_commit(tfull0 + 8 * acc);
                            ++iter;
                            acc = P.nbuf == 2 ? (iter & 1) : 0;
                            const uint32_t ph = (uint32_t)(P.nbuf == 2 ? iter >> 1 : iter) & 1u;
                            if (!ptx::mbar_wait_bounded(tempty0 + 8 * acc, ph ^ 1u, &abort_flag, kWaitNs)) {
                                ok = false;
                                break;
                            }
                            ptx::tc_fence_after();
                            acc_base = tmem_base + (uint32_t)acc * P.acc_stride;
                        }
                        const int k0 = sg * sp.len, k1 = min(k0 + sp.len, sp.total);
                        for (int ci = 0; ok && ci < G.ncls; ++ci) {
                            const int b0 = ci == 0 ? 0 : sp.n[0];
                            const int s0 = max(k0, b0) - b0, s1 = min(k1, b0 + sp.n[ci]) - b0;
                            const uint32_t d_tmem = acc_base + (uint32_t)ci * P.cout_pad;
                            for (int s = s0; s < s1; ++s) {
                                if (!ptx::mbar_wait_bounded(full0 + 8 * stage, phase, &abort_flag, kWaitNs)) {
                                    ok = false;
                                    break;
                                }
                                ptx::tc_fence_after();
                                const uint64_t d0 =
                                    ptx::sdesc_k_swizzled(smem_base + (uint32_t)stage * P.stage_bytes, kRowBytes);
#pragma unroll
                                for (int kk = 0; kk < kChunk / 8; ++kk) {  // split formats: three products
                                    const uint64_t a_hi = d0 + 2 * kk;
                                    const uint64_t a_lo = a_hi + kA16;
                                    const uint64_t b_hi = a_hi + 2 * kA16;
                                    const uint64_t b_lo = b_hi + b16;
                                    // the segment's first product of the class overwrites
                                    const uint32_t first = ((s - s0) | kk) ? 1u : 0u;
                                    if constexpr (OPS == 3) {
                                        ptx::mma_bf16(d_tmem, a_hi, b_hi, idesc, first);
                                        ptx::mma_bf16(d_tmem, a_hi, b_lo, idesc, 1u);
                                        ptx::mma_bf16(d_tmem, a_lo, b_hi, idesc, 1u);
                                    } else {
                                        ptx::mma_tf32(d_tmem, a_hi, b_hi, idesc, first);
                                        ptx::mma_tf32(d_tmem, a_hi, b_lo, idesc, 1u);
                                        ptx::mma_tf32(d_tmem, a_lo, b_hi, idesc, 1u);
                                    }
                                }
                                ptx::mma_commit(empty0 + 8 * stage);
                                if (++stage == P.stages) {
                                    stage = 0;
                                    phase ^= 1u;
                                }
                            }
                        }
                    }
                } else {
                    // flat step loop per class (the issue rate of the MMA-bound shapes depends on it)
                    for (int cs = 0; ok && cs < G.ncls * P.nslices; ++cs) {
                        const int ci = cs / P.nslices, sl = cs - ci * P.nslices;
                        const ClassDesc &C = s_cls[G.cls[ci]];
                        const uint32_t d_tmem = acc_base + (uint32_t)ci * P.cout_pad + (uint32_t)(sl * P.slice_n);
                        const TapRange tr = tile_taps(G, C, T.t, kTcTileM, P.Din);  // same taps as the producer
                        const int nsteps = (tr.end - tr.begin) * P.kc;
                        for (int s = 0; s < nsteps; ++s) {
                            if (!ptx::mbar_wait_bounded(full0 + 8 * stage, phase, &abort_flag, kWaitNs)) {
                                ok = false;
                                break;
                            }
                            ptx::tc_fence_after();
                            const uint64_t d0 =
                                ptx::sdesc_k_swizzled(smem_base + (uint32_t)stage * P.stage_bytes, kRowBytes);
                            if constexpr (OPS == 0) {
#pragma unroll
                                for (int kk = 0; kk < kChunk / 8; ++kk) {
                                    const uint64_t a_hi = d0 + 2 * kk;
                                    const uint64_t a_lo = a_hi + kA16;
                                    const uint64_t b_hi = a_hi + 2 * kA16;
                                    const uint64_t b_lo = b_hi + b16;
                                    // the class's first product overwrites the accumulator
                                    ptx::mma_tf32(d_tmem, a_hi, b_hi, idesc, (s | kk) ? 1u : 0u);
                                    ptx::mma_tf32(d_tmem, a_hi, b_lo, idesc, 1u);
                                    ptx::mma_tf32(d_tmem, a_lo, b_hi, idesc, 1u);
                                }
                            } else if constexpr (OPS == 2) {
#pragma unroll
                                for (int kk = 0; kk < kChunk / 8; ++kk) {
                                    const uint64_t a = d0 + 2 * kk;
                                    ptx::mma_bf16(d_tmem, a, a + kA16, idesc, (s | kk) ? 1u : 0u);
                                }
                            } else if constexpr (OPS == 3) {
#pragma unroll
                                for (int kk = 0; kk < kChunk / 8; ++kk) {
                                    const uint64_t a_hi = d0 + 2 * kk;
                                    const uint64_t a_lo = a_hi + kA16;
                                    const uint64_t b_hi = a_hi + 2 * kA16;
                                    const uint64_t b_lo = b_hi + b16;
                                    ptx::mma_bf16(d_tmem, a_hi, b_hi, idesc, (s | kk) ? 1u : 0u);
                                    ptx::mma_bf16(d_tmem, a_hi, b_lo, idesc, 1u);
                                    ptx::mma_bf16(d_tmem, a_lo, b_hi, idesc, 1u);
                                }
                            } else {
#pragma unroll
                                for (int kk = 0; kk < kChunk / 8; ++kk) {
                                    const uint64_t a = d0 + 2 * kk;
                                    ptx::mma_tf32(d_tmem, a, a + kA16, idesc, (s | kk) ? 1u : 0u);
                                }
                            }
                            ptx::mma_commit(empty0 + 8 * stage);
                            if (++stage == P.stages) {
                                stage = 0;
                                phase ^= 1u;
                            }
                        }
                    }
                }
                if (ok) ptx::mma_commit(tfull0 + 8 * acc);
            }
            if (!ok) {
                record_error(P.status, kErrTimeout, 2);
                abort_flag = 1;
            }
            // Drain: all issued MMAs complete before tensor memory is released.
            ptx::mma_commit(drain);
            const volatile int never = 0;
            ptx::mbar_wait_bounded(drain, 0, &never, 200000000ull);
        }
    }
    // ------------------------------------------------------------ epilogue
    else {
        // Two warps per tensor-memory lane quarter; warp `half` of a quarter takes
        // the 16-channel chunks j with j % 2 == half (groups g % 2 == half when
        // a group is made of whole chunks).
        const int ew = warp - 2;          // 0..kEpiWarps-1
        const int quarter = warp & 3;     // lane quarter this warp may access
        const int half = ew >> 2;         // which share of the channels (0 when kHalves == 1)
        const int m = quarter * 32 + lane;
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
        const int C = P.Cout;
        const int nchunks = (C + 15) / 16;
        const int64_t V = (int64_t)P.Do * P.Ho * P.Wo;
        constexpr bool gn = EPI == CONVT3D_EPI_RELU_GROUPNORM;
        constexpr bool bn = EPI == CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL;
        constexpr bool sm = EPI == CONVT3D_EPI_SOFTMAX_SIGMOID;
        const int nstat = gn ? 3 * P.groups : (bn ? 3 * C : 0);  // (n, S, M2) per group / channel
        const int cpg = gn ? C / P.groups : 16;
        const bool gn_inline = gn && (cpg % 16 == 0);  // groups made of whole 16-channel chunks
        const bool has_bias = P.bias != nullptr;
        auto mine = [&](int j) -> bool {                // does this warp own chunk j?
            return gn_inline ? ((16 * j) / cpg) % kHalves == half : j % kHalves == half;
        };
        int iter = 0;
        int tile = P.tile_begin + blockIdx.x;
        for (; tile < P.tile_end; tile += gridDim.x, ++iter) {
            const Tile T = decode(P, s_grp, tile);
            const GroupDesc &G = s_grp[T.gi];
            // SEG: the tile's earlier segments are added into the running sum here; a
            // class's columns in the last segment's buffer hold its last partial sum
            // if it has steps there (in_final), and the running sum holds the rest (has_sum)
            bool has_sum[2] = {false, false}, in_final[2] = {true, true};
            if constexpr (SEG) {
                const SegPlan sp = seg_plan(P, G, s_cls, T.t);
                bool failed = false;
                for (int sg = 0; sg + 1 < sp.nseg; ++sg, ++iter) {
                    const int a = P.nbuf == 2 ? (iter & 1) : 0;
                    const uint32_t ph = (uint32_t)(P.nbuf == 2 ? iter >> 1 : iter) & 1u;
                    if (!ptx::mbar_wait_bounded(tfull0 + 8 * a, ph, &abort_flag, kWaitNs)) {
                        failed = true;
                        break;
                    }
                    ptx::tc_fence_after();
                    __syncwarp();
                    const int k0 = sg * sp.len;
#pragma unroll
                    for (int ci = 0; ci < 2; ++ci) {
                        if (!seg_touches(sp, ci, k0, k0 + sp.len)) continue;
                        for (int j = 0; j < nchunks; ++j) {
                            if (!mine(j)) continue;
                            const uint32_t col = (uint32_t)(ci * P.cout_pad + 16 * j);
                            float v[16], t[16];
                            ptx::tmem_ld16(lane_base + (uint32_t)a * P.acc_stride + col, v);
                            if (has_sum[ci]) ptx::tmem_ld16(lane_base + P.sum_col + col, t);
                            ptx::tmem_wait_ld();
                            if (has_sum[ci]) {
#pragma unroll
                                for (int i = 0; i < 16; ++i) v[i] += t[i];
                            }
                            ptx::tmem_st16(lane_base + P.sum_col + col, v);
                        }
                        has_sum[ci] = true;
                    }
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(tempty0 + 8 * a);
                }
                if (failed) {
                    if (lane == 0) record_error(P.status, kErrTimeout, 3);
                    abort_flag = 1;
                    break;
                }
                const int kf = (sp.nseg - 1) * sp.len;
#pragma unroll
                for (int ci = 0; ci < 2; ++ci) in_final[ci] = seg_touches(sp, ci, kf, sp.total);
            }
            // a loaded accumulator chunk of class ci at channel c0, completed with the
            // running sum of the earlier segments (SEG kernels; nothing otherwise)
            auto seg_fix = [&](int ci, int c0, float (&v)[16]) {
                if constexpr (SEG) {
                    if (has_sum[ci]) {
                        float t[16];
                        ptx::tmem_ld16(lane_base + P.sum_col + (uint32_t)(ci * P.cout_pad + c0), t);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = (in_final[ci] ? v[i] : 0.f) + t[i];
                    }
                }
            };
            const int acc = P.nbuf == 2 ? (iter & 1) : 0;
            const uint32_t aph = (uint32_t)(P.nbuf == 2 ? iter >> 1 : iter) & 1u;
            if (!ptx::mbar_wait_bounded(tfull0 + 8 * acc, aph, &abort_flag, kWaitNs)) {
                if (lane == 0) record_error(P.status, kErrTimeout, 3);
                abort_flag = 1;
                break;
            }
            ptx::tc_fence_after();
            __syncwarp();

            int off[2];
            off[0] = row_offset(P, G, s_cls[G.cls[0]], T.t, m);
            off[1] = G.ncls > 1 ? row_offset(P, G, s_cls[G.cls[1]], T.t, m) : -1;
            // Stride-2 pairs write (even, odd) columns of one output row together.
            const bool pair_store = G.ncls == 2 && (P.Wo % 2 == 0);
            float *yn = P.y + (int64_t)T.n * C * V;
            // 16 channels c0.. of output position `off` of this sample: NCDHW (one
            // store per channel plane) or channels-last (contiguous, 16-byte stores
            // when every row starts 16-byte aligned)
            const bool plain_out = !P.io16 && !P.cl;  // NCDHW fp32, the common case, tested first
            auto store_row16 = [&](float *yb, int off, int c0, const float (&o)[16]) {
                if (plain_out) {
                    float *dst = yb + (int64_t)c0 * V + off;
                    if (c0 + 16 <= C) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) dst[(int64_t)i * V] = o[i];
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (c0 + i < C) dst[(int64_t)i * V] = o[i];
                    }
                    return;
                }
                if (P.io16) {  // bf16 / fp16 output: same element positions, 2-byte values
                    uint16_t *yh = reinterpret_cast<uint16_t *>(P.y) + (int64_t)T.n * C * V;
                    if (P.cl) {
                        uint16_t *dst = yh + (int64_t)off * C + c0;
                        if (c0 + 16 <= C && (C & 7) == 0) {  // two 16-byte stores of 8 values
                            uint32_t w[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) w[i] = cvt16x2(o[2 * i], o[2 * i + 1], P.io16);
                            reinterpret_cast<uint4 *>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                            reinterpret_cast<uint4 *>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (c0 + i < C) dst[i] = cvt16(o[i], P.io16);
                        }
                    } else {
                        uint16_t *dst = yh + (int64_t)c0 * V + off;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (c0 + i < C) dst[(int64_t)i * V] = cvt16(o[i], P.io16);
                    }
                    return;
                }
                if (P.cl) {
                    float *dst = yb + (int64_t)off * C + c0;
                    if (c0 + 16 <= C && (C & 3) == 0) {
#pragma unroll
                        for (int i = 0; i < 16; i += 4)
                            *reinterpret_cast<float4 *>(dst + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (c0 + i < C) dst[i] = o[i];
                    }
                } else {
                    float *dst = yb + (int64_t)c0 * V + off;
                    if (c0 + 16 <= C) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) dst[(int64_t)i * V] = o[i];
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (c0 + i < C) dst[(int64_t)i * V] = o[i];
                    }
                }
            };
            const uint32_t acc_col = (uint32_t)acc * P.acc_stride;
            // statistics: one partial row per (tile, lane quarter); the two warps of a
            // quarter fill disjoint slots of it
            double *part = P.partials + ((int64_t)T.slot * kTcStatRows + quarter) * nstat;

            if (sm) {
                // softmax over channels then sigmoid, per output position, in the base-2
                // domain: u = (conv + bias) * log2(e), softmax weight = 2^(u - M) / S.
                // Channel pairs (c, c+1) of one class travel together through packed
                // f32x2 arithmetic; the max and the exponentials are per element.
                const uint64_t l2e2 = pack2(kLog2e, kLog2e);
                // base-2 logits of one chunk of one class as 8 channel pairs (channels
                // past Cout get -inf, whose exponential is 0)
                auto logits = [&](int c0, const float (&raw)[16], uint64_t (&u)[8]) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        u[k] = ffma2(pack2(raw[2 * k], raw[2 * k + 1]), l2e2,
                                     *reinterpret_cast<const uint64_t *>(&s_bias_l2e[c0 + 2 * k]));
                    if (c0 + 16 > C) {  // ragged last chunk (warp-uniform branch)
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            float a, b;
                            unpack2(u[k], a, b);
                            u[k] = pack2(c0 + 2 * k < C ? a : -INFINITY, c0 + 2 * k + 1 < C ? b : -INFINITY);
                        }
                    }
                };
                auto max8 = [](const uint64_t (&u)[8]) {
                    float a[16];
#pragma unroll
                    for (int k = 0; k < 8; ++k) unpack2(u[k], a[2 * k], a[2 * k + 1]);
                    return tree_max16(a);
                };
                // u <- 2^(u - mx) in place; returns the sum of the 16 exponentials
                auto exp8 = [](uint64_t (&u)[8], float mx) {
                    const uint64_t neg = pack2(-mx, -mx);
                    uint64_t acc[4];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        float a, b;
                        unpack2(fadd2(u[k], neg), a, b);
                        u[k] = pack2(ex2_approx(a), ex2_approx(b));
                    }
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc[k] = fadd2(u[k], u[k + 4]);
                    acc[0] = fadd2(fadd2(acc[0], acc[2]), fadd2(acc[1], acc[3]));
                    float a, b;
                    unpack2(acc[0], a, b);
                    return a + b;
                };
                // sigmoid(f * e) for 8 pairs, with the polynomial's coefficients
                // pre-multiplied by powers of f (see sigmoid_coefficients), then the stores
                auto sigmoid16 = [](const uint64_t (&e)[8], const uint64_t (&A)[4], float (&o)[16]) {
                    const uint64_t half2 = pack2(0.5f, 0.5f);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint64_t x2 = fmul2(e[k], e[k]);
                        uint64_t q = ffma2(A[3], x2, A[2]);
                        q = ffma2(q, x2, A[1]);
                        q = ffma2(q, x2, A[0]);
                        unpack2(ffma2(e[k], q, half2), o[2 * k], o[2 * k + 1]);
                    }
                };
                auto finish = [&](int c0, int row_off, uint64_t (&e)[8], const uint64_t (&A)[4]) {
                    float o[16];
                    sigmoid16(e, A, o);
                    if (row_off >= 0) store_row16(yn, row_off, c0, o);
                };
                if constexpr (KEEP == 2) {
                    // w-parity pair: warp `half` of the lane quarter owns class `half`
                    // with all its channels, so each row's softmax stays inside one
                    // thread (no exchange between the warps)
                    const int ci = half;
                    const int row_off = half ? off[1] : off[0];  // a select, not an indexed array
                    constexpr int kAll = 2 * kSoftmaxKeepChunks;  // 16-channel chunks per class
                    const uint32_t col0 = lane_base + acc_col + (uint32_t)ci * P.cout_pad;
                    uint64_t e[kAll][8];
                    float mx = -INFINITY;
#pragma unroll
                    for (int j0 = 0; j0 < kAll; j0 += 2) {
                        float raw[2][16];
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj)
                            if (j0 + jj < nchunks) ptx::tmem_ld16(col0 + 16 * (j0 + jj), raw[jj]);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj)
                            if (j0 + jj < nchunks) {
                                logits(16 * (j0 + jj), raw[jj], e[j0 + jj]);
                                mx = fmaxf(mx, max8(e[j0 + jj]));
                            }
                    }
                    float sum = 0.f;
#pragma unroll
                    for (int j = 0; j < kAll; ++j)
                        if (j < nchunks) sum += exp8(e[j], mx);
                    uint64_t A[4];
                    sigmoid_coefficients(__frcp_rn(sum), A);
#pragma unroll
                    for (int j = 0; j < kAll; ++j)
                        if (j < nchunks) finish(16 * j, row_off, e[j], A);
                } else {
                // 1) this warp's chunks: maximum and sum of exponentials per class
                constexpr int kKeep = kSoftmaxKeepChunks;
                uint64_t e[KEEP ? kKeep : 1][2][8];
                float mx[2] = {-INFINITY, -INFINITY}, sum[2] = {0.f, 0.f};
                if (KEEP) {
                    _Pragma("unroll") for (int ci = 0; ci < 2; ++ci) if (ci < G.ncls) {
                        float raw[kKeep][16];
#pragma unroll
                        for (int jj = 0; jj < kKeep; ++jj) {
                            const int j = half + jj * kHalves;
                            if (j < nchunks)
                                ptx::tmem_ld16(lane_base + acc_col + (uint32_t)ci * P.cout_pad + 16 * j, raw[jj]);
                        }
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int jj = 0; jj < kKeep; ++jj) {
                            const int j = half + jj * kHalves;
                            if (j < nchunks) {
                                seg_fix(ci, 16 * j, raw[jj]);
                                logits(16 * j, raw[jj], e[jj][ci]);
                                mx[ci] = fmaxf(mx[ci], max8(e[jj][ci]));
                            }
                        }
#pragma unroll
                        for (int jj = 0; jj < kKeep; ++jj) {
                            const int j = half + jj * kHalves;
                            if (j < nchunks) sum[ci] += exp8(e[jj][ci], mx[ci]);
                        }
                    }
                } else {
                    // online: rescale the running sum whenever the maximum grows
                    for (int j = half; j < nchunks; j += kHalves) {
                        float raw[2][16];
                        _Pragma("unroll") for (int ci = 0; ci < 2; ++ci) if (ci < G.ncls)
                            ptx::tmem_ld16(lane_base + acc_col + (uint32_t)ci * P.cout_pad + 16 * j, raw[ci]);
                        ptx::tmem_wait_ld();
                        _Pragma("unroll") for (int ci = 0; ci < 2; ++ci) if (ci < G.ncls) {
                            seg_fix(ci, 16 * j, raw[ci]);
                            logits(16 * j, raw[ci], e[0][ci]);
                            const float cm = fmaxf(mx[ci], max8(e[0][ci]));
                            const float old = mx[ci] == -INFINITY ? 0.f : sum[ci] * ex2_approx(mx[ci] - cm);
                            mx[ci] = cm;
                            sum[ci] = old + exp8(e[0][ci], cm);
                        }
                    }
                }
                // 2) combine with the partner warp of this lane quarter: global maximum M
                //    and sum S; this warp's exponentials (relative to mx) scale by f
                float f[2], M[2];
                if (kHalves > 1) {
                    float *xm = s_xchg + ((iter & 1) * kHalves + half) * 4 * kTcTileM;  // [class][max,sum][row]
                    xm[0 * kTcTileM + m] = mx[0];
                    xm[1 * kTcTileM + m] = sum[0];
                    xm[2 * kTcTileM + m] = mx[1];
                    xm[3 * kTcTileM + m] = sum[1];
                    asm volatile("bar.sync %0, %1;" ::"r"(1 + quarter), "r"(32 * kHalves) : "memory");
                    const float *xb = s_xchg + (iter & 1) * kHalves * 4 * kTcTileM;
#pragma unroll
                    for (int ci = 0; ci < 2; ++ci) {
                        M[ci] = mx[ci];
#pragma unroll
                        for (int h = 0; h < kHalves; ++h)
                            M[ci] = fmaxf(M[ci], xb[(h * 4 + 2 * ci) * kTcTileM + m]);
                        float S = 0.f;
#pragma unroll
                        for (int h = 0; h < kHalves; ++h) {
                            const float om = xb[(h * 4 + 2 * ci) * kTcTileM + m];
                            const float os = xb[(h * 4 + 2 * ci + 1) * kTcTileM + m];
                            S += om == -INFINITY ? 0.f : os * ex2_approx(om - M[ci]);
                        }
                        const float inv = __frcp_rn(S);
                        const float mine_scale = mx[ci] == -INFINITY ? 0.f : ex2_approx(mx[ci] - M[ci]);
                        f[ci] = KEEP ? mine_scale * inv : inv;
                    }
                } else {
#pragma unroll
                    for (int ci = 0; ci < 2; ++ci) {
                        M[ci] = mx[ci];
                        f[ci] = __frcp_rn(sum[ci]);
                    }
                }
                // 3) outputs: weight t = f * e in (0, 1], then sigmoid(t). A w-parity pair's
                //    two classes are the adjacent columns (2 qw, 2 qw + 1) of one output row:
                //    with both in this thread, each channel's two outputs go out as one
                //    8-byte (fp32) or 4-byte (bf16) store, whole sectors per warp.
                if (KEEP == 1 && G.ncls == 2 && pair_store && !P.cl && off[0] >= 0 && off[1] >= 0) {
                    uint64_t A0[4], A1[4];
                    sigmoid_coefficients(f[0], A0);
                    sigmoid_coefficients(f[1], A1);
#pragma unroll
                    for (int jj = 0; jj < kKeep; ++jj) {
                        const int j = half + jj * kHalves;
                        if (j >= nchunks) continue;
                        const int c0 = 16 * j;
                        float o0[16], o1[16];
                        sigmoid16(e[jj][0], A0, o0);
                        sigmoid16(e[jj][1], A1, o1);
                        if (P.io16) {
                            uint16_t *yh = reinterpret_cast<uint16_t *>(P.y) + (int64_t)T.n * C * V;
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (c0 + i < C)
                                    *reinterpret_cast<uint32_t *>(yh + (int64_t)(c0 + i) * V + off[0]) =
                                        cvt16x2(o0[i], o1[i], P.io16);
                        } else {
                            float *d = yn + (int64_t)c0 * V + off[0];
                            if (c0 + 16 <= C) {
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    *reinterpret_cast<float2 *>(d + (int64_t)i * V) = make_float2(o0[i], o1[i]);
                            } else {
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    if (c0 + i < C)
                                        *reinterpret_cast<float2 *>(d + (int64_t)i * V) = make_float2(o0[i], o1[i]);
                            }
                        }
                    }
                } else
                _Pragma("unroll") for (int ci = 0; ci < 2; ++ci) if (ci < G.ncls) {
                    uint64_t A[4];
                    sigmoid_coefficients(f[ci], A);
                    if (KEEP) {
#pragma unroll
                        for (int jj = 0; jj < kKeep; ++jj) {
                            const int j = half + jj * kHalves;
                            if (j < nchunks) finish(16 * j, off[ci], e[jj][ci], A);
                        }
                    } else {
                        for (int j = half; j < nchunks; j += kHalves) {
                            float raw[16];
                            ptx::tmem_ld16(lane_base + acc_col + (uint32_t)ci * P.cout_pad + 16 * j, raw);
                            ptx::tmem_wait_ld();
                            seg_fix(ci, 16 * j, raw);
                            logits(16 * j, raw, e[0][ci]);
                            exp8(e[0][ci], M[ci]);
                            finish(16 * j, off[ci], e[0][ci], A);
                        }
                    }
                }
                }
            } else {
                // identity / relu+groupnorm store / batchnorm partial sums, per owned chunk
                // running group sums about the shift gc (groups of whole chunks)
                float gs1 = 0.f, gs2 = 0.f, gc = 0.f;
                // the warp's (row, class) pairs inside the output, and the lane whose row
                // supplies a group's shift (the first valid row of class 0, else of class 1)
                const unsigned vb0 = __ballot_sync(0xffffffffu, off[0] >= 0);
                const unsigned vb1 = __ballot_sync(0xffffffffu, off[1] >= 0);
                const int rows_valid = __popc(vb0) + __popc(vb1);
                const bool rows_valid0 = vb0 != 0u;
                const int shift_lane = vb0 ? __ffs(vb0) - 1 : (vb1 ? __ffs(vb1) - 1 : 0);
                for (int j = 0; j < nchunks; ++j) {
                    if (!mine(j)) continue;
                    const int c0 = 16 * j;
                    float v[2][16];
                    _Pragma("unroll") for (int ci = 0; ci < 2; ++ci) if (ci < G.ncls)
                        ptx::tmem_ld16(lane_base + acc_col + (uint32_t)ci * P.cout_pad + c0, v[ci]);
                    ptx::tmem_wait_ld();
                    if constexpr (SEG) {
                        _Pragma("unroll") for (int ci = 0; ci < 2; ++ci) if (ci < G.ncls) seg_fix(ci, c0, v[ci]);
                    }
                    if (G.ncls == 1) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[1][i] = 0.f;
                    }
                    // GroupNorm: v = ReLU(conv + b) feeds the statistics; the stored value is
                    // r = v - b (the accumulator itself where the ReLU passes, else -b), so no
                    // rounding at the bias's magnitude enters y before the normalise pass
                    float r[2][16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float b = s_bias[c0 + i];
                        if (gn && has_bias) {
                            const float t0 = v[0][i] + b, t1 = v[1][i] + b;
                            r[0][i] = t0 > 0.f ? v[0][i] : -b;
                            r[1][i] = t1 > 0.f ? v[1][i] : -b;
                            v[0][i] = fmaxf(t0, 0.f);
                            v[1][i] = fmaxf(t1, 0.f);
                        } else if (gn) {  // no bias: r = v
                            v[0][i] = fmaxf(v[0][i], 0.f);
                            v[1][i] = fmaxf(v[1][i], 0.f);
                        } else {
                            v[0][i] += b;
                            v[1][i] += b;
                        }
                    }
                    if (bn) {
                        // per channel of z = scale*(conv + bias) over this warp's rows (both
                        // classes of a pair): count, sum, and the squared deviations from the
                        // warp's own channel mean (no common offset enters the squares)
                        const bool val0 = off[0] >= 0, val1 = G.ncls > 1 && off[1] >= 0;
                        float z[2][16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            z[0][i] = val0 ? P.scale * v[0][i] : 0.f;
                            z[1][i] = val1 ? P.scale * v[1][i] : 0.f;
                        }
                        float sz = transpose_reduce16(z[0], lane);
                        if (G.ncls > 1) sz += transpose_reduce16(z[1], lane);
                        const int nrow = __popc(__ballot_sync(0xffffffffu, val0)) +
                                         __popc(__ballot_sync(0xffffffffu, val1));
                        const float mean = nrow > 0 ? sz / (float)nrow : 0.f;  // lanes 2i, 2i+1: channel c0 + i
                        // deviations from the warp's mean: their sum (the sum of z without the
                        // offset's rounding) and their squares
                        float q[2][16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float mi = __shfl_sync(0xffffffffu, mean, 2 * i);
                            z[0][i] = val0 ? z[0][i] - mi : 0.f;
                            z[1][i] = val1 ? z[1][i] - mi : 0.f;
                            q[0][i] = z[0][i] * z[0][i];
                            q[1][i] = z[1][i] * z[1][i];
                        }
                        float sd = transpose_reduce16(z[0], lane), m2 = transpose_reduce16(q[0], lane);
                        if (G.ncls > 1) {
                            sd += transpose_reduce16(z[1], lane);
                            m2 += transpose_reduce16(q[1], lane);
                        }
                        const int c = c0 + (lane >> 1);
                        if ((lane & 1) == 0 && c < C) {
                            part[3 * c] = (double)nrow;
                            part[3 * c + 1] = fma((double)nrow, (double)mean, (double)sd);
                            part[3 * c + 2] =
                                nrow > 0 ? (double)fmaxf(m2 - sd * sd * __frcp_rn((float)nrow), 0.f) : 0.0;
                        }
                        continue;
                    }
                    if (gn_inline) {
                        const float m0 = off[0] >= 0 ? 1.f : 0.f, m1 = off[1] >= 0 ? 1.f : 0.f;
                        if (c0 % cpg == 0) {
                            // first chunk of a group: one of its values (the first valid row's
                            // first channel) is the group's shift, |v - shift| ~ the group's spread
                            const float mine_v = rows_valid0 ? v[0][0] : v[1][0];
                            gc = rows_valid ? __shfl_sync(0xffffffffu, mine_v, shift_lane) : 0.f;
                            gs1 = gs2 = 0.f;
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float a = m0 * (v[0][i] - gc), b = m1 * (v[1][i] - gc);
                            gs1 += a + b;
                            gs2 += a * a + b * b;
                        }
                        if ((c0 + 16) % cpg == 0)  // this chunk closes group g (same for all lanes)
                            warp_moments(gs1, gs2, rows_valid * cpg, gc, part + 3 * (c0 / cpg));
                    }
                    if (gn && has_bias) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            v[0][i] = r[0][i];
                            v[1][i] = r[1][i];
                        }
                    }
                    if (P.io16 && !P.cl && pair_store) {  // 16-bit NCDHW: (even, odd) outputs as one pair
                        if (off[0] >= 0 && off[1] >= 0) {
                            uint16_t *yh = reinterpret_cast<uint16_t *>(P.y) + (int64_t)T.n * C * V;
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (c0 + i < C)
                                    *reinterpret_cast<uint32_t *>(yh + (int64_t)(c0 + i) * V + off[0]) =
                                        cvt16x2(v[0][i], v[1][i], P.io16);
                        }
                    } else if (P.cl || P.io16) {
                        _Pragma("unroll") for (int ci = 0; ci < 2; ++ci) if (ci < G.ncls)
                            if (off[ci] >= 0) store_row16(yn, off[ci], c0, v[ci]);
                    } else if (pair_store) {
                        if (off[0] >= 0 && off[1] >= 0) {
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                if (c0 + i < C)
                                    *reinterpret_cast<float2 *>(yn + (int64_t)(c0 + i) * V + off[0]) =
                                        make_float2(v[0][i], v[1][i]);
                        }
                    } else {
                        _Pragma("unroll") for (int ci = 0; ci < 2; ++ci) if (ci < G.ncls)
                            if (off[ci] >= 0) {
#pragma unroll
                                for (int i = 0; i < 16; ++i)
                                    if (c0 + i < C) yn[(int64_t)(c0 + i) * V + off[ci]] = v[ci][i];
                            }
                    }
                }
                if (gn && !gn_inline) {
                    // group statistics of the ReLU output: passes over tensor memory per group,
                    // groups g % 2 == half (all lanes in step; invalid rows contribute nothing):
                    // the warp's mean of the group first, then sums about it
                    for (int g = half; g < P.groups; g += kHalves) {
                        float c = 0.f, s1 = 0.f, s2 = 0.f;
                        int cnt = 0;
                        for (int pass = 0; pass < 2; ++pass) {
                            _Pragma("unroll") for (int ci = 0; ci < 2; ++ci) if (ci < G.ncls) {
                                const bool valid = off[ci] >= 0;
                                const uint32_t col = acc_col + (uint32_t)ci * P.cout_pad;
                                for (int c0 = (g * cpg) & ~15; c0 < (g + 1) * cpg; c0 += 16) {
                                    float v[16];
                                    ptx::tmem_ld16(lane_base + col + c0, v);
                                    ptx::tmem_wait_ld();
                                    seg_fix(ci, c0, v);
#pragma unroll
                                    for (int i = 0; i < 16; ++i) {
                                        const int ch = c0 + i;
                                        if (!valid || ch < g * cpg || ch >= (g + 1) * cpg) continue;
                                        const float d = fmaxf(v[i] + s_bias[ch], 0.f) - c;
                                        s1 += d;
                                        s2 += d * d;
                                        cnt += pass;
                                    }
                                }
                            }
                            if (pass == 0) {
                                const int n = warp_sum_i(valid_rows(off, G.ncls) * cpg);
                                c = n > 0 ? warp_sum_f(s1) / (float)n : 0.f;
                                s1 = s2 = 0.f;
                            }
                        }
                        warp_moments(s1, s2, warp_sum_i(cnt), c, part + 3 * g);
                    }
                }
            }
            // tensor memory of this accumulator may be overwritten from here on
            ptx::tc_fence_before();
            ptx::mbar_arrive(tempty0 + 8 * acc);
        }
        // Softmax with the channels of a lane quarter split between warps meets its
        // partner at a named barrier once per tile. A warp whose wait ran out left the
        // loop early: it still meets that barrier once for every tile it did not
        // finish, so the partner never waits on a warp that has gone.
        if constexpr (sm && KEEP != 2 && kHalves > 1)
            for (; tile < P.tile_end; tile += gridDim.x)
                asm volatile("bar.sync %0, %1;" ::"r"(1 + quarter), "r"(32 * kHalves) : "memory");
    }

    // ------------------------------------------------------------ teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, P.tmem_cols);
    }
}

// ------------------------------------------------------------------- host

typedef CUresult (*EncodeIm2colFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const int *, const int *, cuuint32_t, cuuint32_t,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr CUtensorMapSwizzle kSwizzle = kChunk == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;

struct DriverFns {
    EncodeIm2colFn im2col = nullptr;
    EncodeTiledFn tiled = nullptr;
    cudaError_t err = cudaSuccess;
};

const DriverFns &driver_fns() {
    static DriverFns fns = [] {
        DriverFns f;
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        f.err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p, 12000, cudaEnableDefault, &q);
        if (f.err == cudaSuccess && q == cudaDriverEntryPointSuccess) f.im2col = (EncodeIm2colFn)p;
        p = nullptr;
        cudaError_t e2 = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        if (e2 == cudaSuccess && q == cudaDriverEntryPointSuccess) f.tiled = (EncodeTiledFn)p;
        if (f.err == cudaSuccess) f.err = e2;
        return f;
    }();
    return fns;
}

int round_pow2(int v) {
    int p = 32;
    while (p < v) p *= 2;
    return p;
}

}  // namespace

// Per-plan state of the tensor-core launch: encoded tensor maps (re-encoded
// only when the workspace or the staged-input pointers change), tables and
// launch shape.
struct TcCache {
    TcParams P;
    const void *key[4];
    void (*kern)(const TcParams);
    int threads;
    size_t smem;
    int grid;
    bool ready;
};

void tc_cache_free(void *c) { delete static_cast<TcCache *>(c); }

// The kernel instance for the plan's epilogue, operand format OPS and (for
// softmax) register-kept exponentials; threads receives its block size.
template <int OPS, bool MERGED, bool SEG = false>
static void (*select_kernel(const convt3d_plan_s &p, int &threads))(const TcParams) {
    switch (p.d.epilogue) {
        case CONVT3D_EPI_IDENTITY:
            threads = EpiCfg<CONVT3D_EPI_IDENTITY>::threads;
            return convt3d_tc_gemm<CONVT3D_EPI_IDENTITY, 1, OPS, MERGED, SEG>;
        case CONVT3D_EPI_RELU_GROUPNORM:
            threads = EpiCfg<CONVT3D_EPI_RELU_GROUPNORM>::threads;
            return convt3d_tc_gemm<CONVT3D_EPI_RELU_GROUPNORM, 1, OPS, MERGED, SEG>;
        case CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL:
            threads = EpiCfg<CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL>::threads;
            return convt3d_tc_gemm<CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL, 1, OPS, MERGED, SEG>;
        case CONVT3D_EPI_SOFTMAX_SIGMOID:
            threads = EpiCfg<CONVT3D_EPI_SOFTMAX_SIGMOID>::threads;
            // registers hold the exponentials when each warp owns at most
            // kSoftmaxKeepChunks 16-channel chunks
            // Stride 2 along w with Cout <= 64, single-product formats: each warp of a
            // lane quarter owns one class's channels (no exchange; measured faster
            // there). The split formats, whose longer K steps leave the epilogue more
            // room, take the channel split below: one (max, sum) exchange per tile
            // buys each channel's (even, odd) columns stored as one pair.
            if constexpr ((OPS == 1 || OPS == 2) && !SEG)
                if (EpiCfg<CONVT3D_EPI_SOFTMAX_SIGMOID>::warps == 8 && p.g.ss[2] == 2 &&
                    p.cout_pad <= 16 * 2 * kSoftmaxKeepChunks)
                    return convt3d_tc_gemm<CONVT3D_EPI_SOFTMAX_SIGMOID, 2, OPS, MERGED, SEG>;
            return p.cout_pad <= 16 * kSoftmaxKeepChunks * (EpiCfg<CONVT3D_EPI_SOFTMAX_SIGMOID>::warps / 4)
                       ? convt3d_tc_gemm<CONVT3D_EPI_SOFTMAX_SIGMOID, 1, OPS, MERGED, SEG>
                       : convt3d_tc_gemm<CONVT3D_EPI_SOFTMAX_SIGMOID, 0, OPS, MERGED, SEG>;
    }
    return nullptr;
}

static cudaError_t tc_setup(convt3d_plan_s &p, TcCache &tc, const float *xs_hi, const float *xs_lo,
                            const float *w_hi, const float *w_lo) {
    const DriverFns &fn = driver_fns();
    if (!fn.im2col || !fn.tiled) return fn.err != cudaSuccess ? fn.err : cudaErrorNotSupported;
    TcParams *P = &tc.P;
    const Geometry &g = p.g;
    if (!tc.ready) {
        memset(P, 0, sizeof(*P));
        P->N = g.N;
        P->Cout = g.Cout;
        P->cout_pad = p.cout_pad;
        P->Do = g.Do;
        P->Ho = g.Ho;
        P->Wo = g.Wo;
        P->sd = g.ss[0];
        P->sh = g.ss[1];
        P->sw = g.ss[2];
        P->Din = g.Din;
        P->Hin = g.Hin;
        P->Win = g.Win;
        P->chunk = kRowBytes / p.elem_bytes;
        P->kc = p.cin_pad / P->chunk;
        P->bf16 = p.bf16;
        P->half = p.half;
        P->epilogue = p.d.epilogue;
        P->groups = p.d.groups;
        P->scale = p.d.scale;
        P->ngroups = p.ngroups;
        P->tiles_per_sample = p.tiles_per_sample;
        P->div_tps = make_fastdiv((uint32_t)p.tiles_per_sample);
        P->total_tiles = (int)p.tiles;
        int ncls_max = 1;
        for (int i = 0; i < p.ngroups; ++i) {
            P->grp[i] = p.grp[i];
            if (p.grp[i].ncls > ncls_max) ncls_max = p.grp[i].ncls;
        }
        if (p.merged) {
            // flatten each pair's merged walk: (d-slice a, h-tap b, merged w-tap m)
            int ns = 0;
            for (int gi = 0; gi < p.ngroups; ++gi) {
                GroupDesc &G = P->grp[gi];
                const ClassDesc &C0 = g.cls[G.cls[0]], &C1 = g.cls[G.cls[1]];
                G.step0 = ns;
                G.steps_per_a = C0.nt_h * G.nm;
                if (ns + C0.nt_d * G.steps_per_a > kMaxSteps) return cudaErrorInvalidConfiguration;
                for (int a = 0; a < C0.nt_d; ++a)
                    for (int b = 0; b < C0.nt_h; ++b)
                        for (int m = 0; m < G.nm; ++m) {
                            const int mask = G.mmask[m];
                            StepDesc e{};
                            const int t0 = (mask & 1) ? C0.tap_begin + (a * C0.nt_h + b) * C0.nt_w + G.me[m][0] : -1;
                            const int t1 = (mask & 2) ? C1.tap_begin + (a * C1.nt_h + b) * C1.nt_w + G.me[m][1] : -1;
                            const ClassDesc &C = (mask & 1) ? C0 : C1;
                            const TapDesc &td = g.taps[(mask & 1) ? t0 : t1];
                            e.cls = (mask & 1) ? 0 : 1;
                            e.mask = (uint8_t)mask;
                            e.tb0 = (int16_t)((mask & 1) ? t0 : t1);
                            e.tb1 = (int16_t)(mask == 3 ? t1 : -1);
                            e.ow = (uint8_t)(td.dw - C.lo_w);
                            e.oh = (uint8_t)(td.dh - C.lo_h);
                            e.od = (uint8_t)(td.dd - C.lo_d);
                            P->steps[ns++] = e;
                        }
            }
        }
        for (int i = 0; i < kMaxClasses; ++i) P->cls[i] = g.cls[i];
        for (int i = 0; i < kMaxTaps; ++i) P->taps[i] = g.taps[i];
        P->nslices = p.nslices;
        P->slice_n = p.cout_pad / p.nslices;
        // double-buffered accumulators where two fit the 512 tensor-memory columns
        const int acc_cols = ncls_max * p.cout_pad;
        P->nbuf = 2 * acc_cols <= 512 ? 2 : 1;
        P->acc_stride = (uint32_t)acc_cols;
        P->tmem_cols = (uint32_t)round_pow2(P->nbuf * acc_cols);
        // Long reductions (split formats, non-merged walks, one N slice): tiles whose walk
        // exceeds kSegSteps K steps accumulate in segments, with a running-sum region
        // beside the accumulators (three regions where they fit, else one buffer and the sum).
        const bool split = p.planes == 2;
        // BatchNorm+pool is left whole: the accumulation error is close to a common
        // relative factor, which the batch statistics' (z - mean) / sd cancels, and the
        // pooled mean averages the rest (it meets the bar at K = 8,000 unsegmented)
        int max_steps = 0;
        if (split && !p.merged && p.nslices == 1 && p.d.epilogue != CONVT3D_EPI_SCALE_BATCHNORM_AVGPOOL)
            for (int gi = 0; gi < p.ngroups; ++gi)
                for (int t = 0; t < p.grp[gi].tiles; ++t) {
                    int n = 0;
                    for (int ci = 0; ci < p.grp[gi].ncls; ++ci) {
                        const TapRange tr = tile_taps(p.grp[gi], g.cls[p.grp[gi].cls[ci]], t, kTcTileM, g.Din);
                        n += (tr.end - tr.begin) * P->kc;
                    }
                    max_steps = n > max_steps ? n : max_steps;
                }
        P->seg_steps = 0;
        P->sum_col = 0;
        if (max_steps > kSegSteps) {
            if (3 * acc_cols <= 512) {
                P->nbuf = 2;
                P->sum_col = (uint32_t)(2 * acc_cols);
                P->tmem_cols = (uint32_t)round_pow2(3 * acc_cols);
                P->seg_steps = kSegSteps;
            } else if (2 * acc_cols <= 512) {
                P->nbuf = 1;
                P->sum_col = (uint32_t)acc_cols;
                P->tmem_cols = (uint32_t)round_pow2(2 * acc_cols);
                P->seg_steps = kSegSteps;
            }
        }
        P->b_bytes = (uint32_t)P->slice_n * kRowBytes;
        P->planes = p.planes;
        P->cl = p.cl;
        P->io16 = p.io16;
        P->stage_bytes = (uint32_t)p.planes * (kABytes + (p.merged ? 2u : 1u) * P->b_bytes);
        const int ops = p.planes == 2 ? (p.bf16 ? 3 : 0) : (p.bf16 ? 2 : 1);
        if (P->seg_steps > 0)  // split formats only (ops 0 or 3), never merged
            tc.kern = ops == 3 ? select_kernel<3, false, true>(p, tc.threads) : select_kernel<0, false, true>(p, tc.threads);
        else switch (ops * 2 + (p.merged ? 1 : 0)) {
            case 0: tc.kern = select_kernel<0, false>(p, tc.threads); break;
            case 1: tc.kern = select_kernel<0, true>(p, tc.threads); break;
            case 2: tc.kern = select_kernel<1, false>(p, tc.threads); break;
            case 3: tc.kern = select_kernel<1, true>(p, tc.threads); break;
            case 4: tc.kern = select_kernel<2, false>(p, tc.threads); break;
            case 5: tc.kern = select_kernel<2, true>(p, tc.threads); break;
            case 6: tc.kern = select_kernel<3, false>(p, tc.threads); break;
            default: tc.kern = select_kernel<3, true>(p, tc.threads); break;
        }
        if (!tc.kern) return cudaErrorInvalidValue;
        // stage ring: as many stages as fit beside the kernel's static shared memory
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, tc.kern);
        if (e != cudaSuccess) return e;
        const size_t max_dyn = 232448 - fa.sharedSizeBytes;  // 227 KB opt-in limit per block
        int stages = (int)((max_dyn - 1024) / P->stage_bytes);
        if (stages > kMaxStages) stages = kMaxStages;
        if (stages < 2 || P->tmem_cols > 512) return cudaErrorInvalidConfiguration;
        P->stages = stages;
        tc.smem = 1024 + (size_t)stages * P->stage_bytes;
        e = cudaFuncSetAttribute(tc.kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc.smem);
        if (e != cudaSuccess) return e;
        int dev = 0, sms = 148;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        tc.grid = sms;
        tc.key[0] = tc.key[1] = tc.key[2] = tc.key[3] = nullptr;
        tc.ready = true;
    }
    if (tc.key[0] == xs_hi && tc.key[1] == xs_lo && tc.key[2] == w_hi && tc.key[3] == w_lo) return cudaSuccess;

    // activation maps: one im2col map per class and plane
    const cuuint64_t eb = (cuuint64_t)p.elem_bytes;
    const CUtensorMapDataType dt = !p.bf16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : (p.half ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    const cuuint64_t gdim[5] = {(cuuint64_t)p.cin_pad, (cuuint64_t)g.Win, (cuuint64_t)g.Hin, (cuuint64_t)g.Din,
                                (cuuint64_t)g.N};
    const cuuint64_t gstr[4] = {(cuuint64_t)p.cin_pad * eb, (cuuint64_t)p.cin_pad * eb * g.Win,
                                (cuuint64_t)p.cin_pad * eb * g.Win * g.Hin,
                                (cuuint64_t)p.cin_pad * eb * g.Win * g.Hin * g.Din};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    for (int gi = 0; gi < p.ngroups; ++gi) {
        const GroupDesc &G = p.grp[gi];
        for (int ci = 0; ci < G.ncls; ++ci) {
            const int c = G.cls[ci];
            const ClassDesc &C = g.cls[c];
            const int lo_w = C.lo_w, lo_h = C.lo_h, lo_d = C.lo_d;
            const int up_w = G.Qw - g.Win + lo_w, up_h = G.Qh - g.Hin + lo_h, up_d = G.Qd - g.Din + lo_d;
#if CONVT3D_CORNERS_DHW
            const int lower[3] = {lo_d, lo_h, lo_w}, upper[3] = {up_d, up_h, up_w};
#else
            const int lower[3] = {lo_w, lo_h, lo_d}, upper[3] = {up_w, up_h, up_d};
#endif
            for (int plane = 0; plane < p.planes; ++plane) {
                CUresult r = fn.im2col(plane ? &P->a_lo[c] : &P->a_hi[c], dt, 5,
                                       (void *)(plane ? xs_lo : xs_hi), gdim, gstr, lower, upper, P->chunk,
                                       kTcTileM, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, kSwizzle,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
                if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
            }
        }
    }
    // weight maps: [tap][cout_pad][cin_pad], box chunk x slice_n x 1
    const cuuint64_t wdim[3] = {(cuuint64_t)p.cin_pad, (cuuint64_t)p.cout_pad, (cuuint64_t)g.ntaps};
    const cuuint64_t wstr[2] = {(cuuint64_t)p.cin_pad * eb, (cuuint64_t)p.cin_pad * eb * p.cout_pad};
    const cuuint32_t box[3] = {(cuuint32_t)P->chunk, (cuuint32_t)P->slice_n, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    for (int plane = 0; plane < p.planes; ++plane) {
        CUresult r = fn.tiled(plane ? &P->b_lo : &P->b_hi, dt, 3,
                              (void *)(plane ? w_lo : w_hi), wdim, wstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              kSwizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    tc.key[0] = xs_hi;
    tc.key[1] = xs_lo;
    tc.key[2] = w_hi;
    tc.key[3] = w_lo;
    return cudaSuccess;
}

cudaError_t launch_tc(convt3d_plan_s &p, const float *xs_hi, const float *xs_lo, const float *w_hi,
                      const float *w_lo, const float *bias, float *y, double *partials, uint32_t *status,
                      int n0, int n1, cudaStream_t s) {
    static_assert(sizeof(TcParams) < 32000, "kernel parameter block too large");
    if (!p.tc_cache) {
        p.tc_cache = new (std::nothrow) TcCache();
        if (!p.tc_cache) return cudaErrorMemoryAllocation;
        static_cast<TcCache *>(p.tc_cache)->ready = false;
    }
    TcCache &tc = *static_cast<TcCache *>(p.tc_cache);
    cudaError_t e = tc_setup(p, tc, xs_hi, xs_lo, w_hi, w_lo);
    if (e != cudaSuccess) return e;
    tc.P.bias = bias;
    tc.P.y = y;
    tc.P.partials = partials;
    tc.P.status = status;
    // the tiles of samples [n0, n1): tiles are ordered sample by sample
    tc.P.tile_begin = n0 * tc.P.tiles_per_sample;
    tc.P.tile_end = n1 * tc.P.tiles_per_sample;
    const int count = tc.P.tile_end - tc.P.tile_begin;
    if (count <= 0) return cudaSuccess;
    tc.kern<<<count < tc.grid ? count : tc.grid, tc.threads, tc.smem, s>>>(tc.P);
    return cudaGetLastError();
}

}  // namespace convt3d
