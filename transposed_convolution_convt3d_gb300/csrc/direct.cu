// Tensor-core implicit GEMM reading the caller's NCDHW fp32 input directly,
// for stride-2-along-w problems with at most 32 input channels and rows of a
// multiple of 8 positions (the shape of the softmax workload: few channels,
// short K walks, HBM-bound output).
//
// The w-parity pair of each (d, h) output-parity class shares a tile (two
// accumulators side by side in tensor memory, merged w-taps as in the general
// kernel); a tile is TH rows of the pair's q-grid by its full width Qw
// (TH * Qw = 128).  What differs from the general kernel:
//  - no staged copy of x: for every input d-slice a tile reads, one TMA tiled
//    load brings the slab of x the tile needs (all channels, the tile's h rows
//    plus the taps' halo, the whole w extent plus halo; out-of-range elements
//    arrive as zeros) into shared memory;
//  - converter warps split the slab on chip into bf16 hi and lo (hi = bf16(v),
//    lo = bf16(v - hi), both rounded to nearest even), one K-major buffer with
//    the 64-byte swizzle per merged w offset dw: buffer row (h', w) holds x at
//    (h0 + h', w + dw) for the tile's TH rows plus the h halo.  An h tap dh is then
//    the same buffer read from row (dh - lo_h) * Qw on: a whole number of 8-row
//    swizzle atoms, so the MMA descriptors address it directly and the tile's
//    h taps share one conversion;
//  - one pipeline stage per d-slice: its activation buffers and the weight
//    slices of all its K steps, so the single-thread producer and MMA roles
//    hand over once per slice, not once per K step.
//
// CTA roles (persistent, one CTA per SM):
//   warp 0        TMA producer (one thread): x slabs and weight slices
//   warp 1        MMA issuer (one thread) + tensor-memory allocation
//   warps 2..7    converters: slab -> bf16 hi/lo activation buffers
//   warps 8..19   epilogue, three groups of four warps; group g takes every third
//                 tile of the CTA, one output row (both classes) per thread; the
//                 tiles rotate through four accumulator buffers, so the MMAs can
//                 run ahead of the epilogue
// Every wait is bounded; a wait that runs out records CONVT3D_ERR_TIMEOUT in the
// workspace status word, all roles drain and the kernel returns.
#include <stdio.h>
#include <string.h>

#include <new>

#include "convt3d_internal.h"
#include "epimath.cuh"
#include "ptx.cuh"

namespace convt3d {
namespace {

constexpr int kDirGroups = 4;          // (d, h) parity pairs of a stride-2 problem
constexpr int kDirMaxSteps = 128;      // merged K steps of all pairs
constexpr int kDirMaxStages = 4;
constexpr int kDirMaxSlabs = 4;
constexpr int kDirAccBufs = 4;         // accumulator buffers (all 512 tensor-memory columns)
constexpr int kDirAccCols = 128;       // tensor-memory columns per buffer (2 x cout_pad <= 128)
constexpr int kDirEpiGroups = 3;       // epilogue groups of four warps
constexpr int kDirEpiWarps = 4 * kDirEpiGroups;
constexpr int kDirConvWarps = 6;       // converter warps (the register budget per thread is the same for 18 and 20 warps)
constexpr int kDirConvThreads = 32 * kDirConvWarps;
constexpr int kDirThreads = 32 * (2 + kDirConvWarps + kDirEpiWarps);
constexpr int kDirK = 32;              // input channels per K step (one 64-byte bf16 row)
constexpr uint32_t kDirRowBytes = 64;
constexpr uint64_t kDirWaitNs = 2000000000ull;

// One merged K step: input offsets (dh, dw), which classes it feeds (bit c),
// the activation buffer of its w offset (mi), and its weight slices at boff in
// its stage's weight area: tb0 = the tap of class 0 (or of class 1 when only it
// has the offset), tb1 = class 1's tap when both have it (else -1); layout
// hi(tb0) [hi(tb1)] lo(tb0) [lo(tb1)].
struct DStep {
    int8_t dh, dw;
    uint8_t mask, mi;
    int16_t tb0, tb1;
    uint32_t boff;
    // the MMA's operand offsets within a stage, in 16-byte units (the descriptors'
    // start-address unit): activation rows, weight hi slices, and weight lo after hi
    uint16_t a16, b16, blo16, pad_;
};

// One w-parity pair: classes (rd, rh, 0) and (rd, rh, 1).
struct DGroup {
    int Qd, Qh;         // q-grid of the pair along d and h (the classes share rd, rh)
    int Qw0, Qw1;       // q-grid width of each class
    int rd, rh;         // output parities along d and h
    int nt_d;           // d-slices (taps along d)
    int spa;            // K steps per d-slice (h taps x merged w offsets)
    int step0;          // first step in the step table
    int lo_h;           // smallest h offset: the slab's first row is hb * TH + lo_h
    int nm;             // merged w offsets = activation buffers per slice
    int brows;          // rows of each activation buffer: (TH + h span) * Qw
    int nhb;            // h-blocks: ceil(Qh / TH)
    int tiles;          // tiles per sample: Qd x nhb
    int tile_prefix;    // tiles of earlier pairs within one sample
    uint32_t sb_bytes;  // weight slices of one d-slice's K steps
    uint32_t woff;      // its d-slice 0's weight slices in the packed weight (bytes)
    FastDiv div_nhb;
    int8_t dd[8];       // input d offset of each d-slice
    int8_t mdw[8];      // w offset of each activation buffer
};

struct DirectParams {
    CUtensorMap x_map;  // fp32 [N][Cin][Din][Hin][Win], box (wfp, hfp, 1, 32, 1)
    // The weight packed for this kernel: per pair and d-slice, the stage image of the
    // slice's weight slices (bf16 hi [lo] planes, rows of 32 channels, 64-byte swizzled
    // as the MMA descriptors read them), copied into a stage by one bulk load.
    const uint8_t *wdir;
    const float *bias;
    float *y;
    uint32_t *status;
    int N, Cout, cout_pad, Din, Do, Ho, Wo, sd, sh, sw;
    int Qw, TH;         // q-grid width, q rows per tile (TH * Qw = 128)
    int qw_shift;       // log2(Qw)
    int w_lo, wfp, hfp; // slab: first w and width (16-byte multiples), height
    int io16;           // y's 16-bit kind (kBF16 / kF16) when x and y are 16-bit arrays, else 0
    int ngroups, tiles_per_sample, total_tiles;
    FastDiv div_tps;
    int stages, slabs;
    uint32_t slab_bytes;   // one slab (wfp * hfp * 32 fp32), also its TMA byte count
    uint32_t slab_stride;  // slab bytes rounded up to 128 (the TMA destination alignment)
    uint32_t b_bytes;      // one weight slice: cout_pad rows x 64 bytes
    uint32_t buf_bytes;    // one plane of one activation buffer: max brows x 64 bytes
    uint32_t a_bytes;      // a stage's activation buffers: nm_max x planes x buf_bytes
    uint32_t stage_bytes;  // activation buffers + the largest slice's weight slices
    uint32_t wdir_bytes;   // the packed weight
    DGroup grp[kDirGroups];
    DStep steps[kDirMaxSteps];
};

struct DTile {
    int gi, n, qd, hb;
};

// Tile order: sample by sample (the pairs of a sample read the same input
// planes, which then stay in L2 between them), then pair, d position, h-block.
__device__ __forceinline__ DTile ddecode(const DirectParams &P, const DGroup *grp, int tile) {
    DTile r;
    r.n = (int)fastdiv((uint32_t)tile, P.div_tps);
    const int rem = tile - r.n * P.tiles_per_sample;
    int gi = 0;
    while (gi + 1 < P.ngroups && rem >= grp[gi + 1].tile_prefix) ++gi;
    r.gi = gi;
    const int t = rem - grp[gi].tile_prefix;
    r.qd = (int)fastdiv((uint32_t)t, grp[gi].div_nhb);
    r.hb = t - r.qd * grp[gi].nhb;
    return r;
}

__device__ __forceinline__ bool slice_live(const DirectParams &P, const DGroup &G, const DTile &T, int a) {
    return (unsigned)(T.qd + G.dd[a]) < (unsigned)P.Din;
}

__device__ __forceinline__ void drecord_error(uint32_t *status, uint32_t code, uint32_t site) {
    if (atomicCAS(status, 0u, code) == 0u) {
        status[1] = site;
        status[2] = blockIdx.x;
    }
}

// A wait by all 32 lanes of a warp with one outcome for all of them (a lane that
// saw the abort flag fails the wait for the whole warp), so that the warp's
// control flow stays uniform around its __syncwarp and collective instructions.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int *abort) {
    const bool w = ptx::mbar_wait_bounded(bar, parity, abort, kDirWaitNs);
    return __all_sync(0xffffffffu, w);
}

// Largest of 16 values in four dependent levels.
// max(a, b, c) in one instruction (the three-input form of max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// max(m, v[0..15]): eight three-input maxima.
__device__ __forceinline__ float max17(float m, const float (&v)[16]) {
    const float a0 = fmax3(v[0], v[1], v[2]), a1 = fmax3(v[3], v[4], v[5]), a2 = fmax3(v[6], v[7], v[8]);
    const float a3 = fmax3(v[9], v[10], v[11]), a4 = fmax3(v[12], v[13], v[14]);
    return fmax3(m, fmax3(a0, a1, a2), fmax3(a3, a4, v[15]));
}

// sigmoid(t) for t in [0, 1] as 1/2 + t * (s0 + s1 t^2 + s2 t^4): the odd part of sigmoid
// about 0 fitted by a linear program minimising the largest error over 20,001 points of
// [0, 1] (max error 2.6e-6, 2.7e-6 with the fp32 Horner evaluation below; the outputs lie
// in (1/2, 0.74), so this is under 2 % of a 1e-4 relative bound).
constexpr float kSig3t0 = 0.24998110691084421f;
constexpr float kSig3t1 = -0.020678075988383896f;
constexpr float kSig3t2 = 0.0017581814282046223f;

// Coefficients that evaluate sigmoid(f * e) from e directly:
// 1/2 + e * (s0 f + s1 f^3 e^2 + s2 f^5 e^4), packed as pairs.
__device__ __forceinline__ void sigmoid3_coefficients(float f, uint64_t (&A)[3]) {
    const float f2 = f * f;
    const float a0 = kSig3t0 * f, a1 = kSig3t1 * f * f2, a2 = kSig3t2 * f * f2 * f2;
    A[0] = pack2(a0, a0);
    A[1] = pack2(a1, a1);
    A[2] = pack2(a2, a2);
}

// Programmatic dependent launch: let the next grid in the stream (launched with
// programmatic stream serialization) start before this one completes ...
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ... and, in that grid, wait until the grids it depends on have completed and
// their memory operations are visible (returns at once without such a launch).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// (lo_elem, hi_elem) rounded to nearest-even bf16 and packed, lo_elem in the low half.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo_elem, float hi_elem) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi_elem), "f"(lo_elem));
    return r;
}

// The same in fp16.
__device__ __forceinline__ uint32_t f16x2_rn(float lo_elem, float hi_elem) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi_elem), "f"(lo_elem));
    return r;
}

// EPI: CONVT3D_EPI_SOFTMAX_SIGMOID or CONVT3D_EPI_IDENTITY.  OPS: 2 = BF16 (one product
// of bf16-rounded operands), 3 = split BF16 (three products), 4 = FP16 (one product of
// fp16-rounded operands).  X16: x and y are 16-bit arrays of the operands' own format (BF16
// or FP16 only): the slab already holds the operands, so the converter only re-lays it.
template <int EPI, int OPS, bool X16>
__global__ void __launch_bounds__(kDirThreads, 1) convt3d_direct_gemm(const __grid_constant__ DirectParams P) {
    constexpr int kPlanes = OPS == 3 ? 2 : 1;
    extern __shared__ __align__(1024) uint8_t dsmem_raw[];
    __shared__ __align__(8) uint64_t bars[3 * kDirMaxStages + 2 * kDirMaxSlabs + 2 * kDirAccBufs + 1];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    __shared__ __align__(16) float s_bias[kDirAccCols];      // bias (IDENTITY), zero-padded
    __shared__ __align__(16) float s_bias_l2e[kDirAccCols];  // bias * log2(e), -inf past Cout (softmax)
    __shared__ DGroup s_grp[kDirGroups];
    __shared__ DStep s_steps[kDirMaxSteps];

    // the 1024-byte aligned start, derived from the shared array by an offset (not an
    // integer round trip) so that ordinary loads and stores through it stay shared-memory ones
    uint8_t *smem = dsmem_raw + ((1024u - (ptx::smem_u32(dsmem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t fulla0 = ptx::smem_u32(&bars[0]);                       // stage's buffers built (converter warps)
    const uint32_t fullb0 = ptx::smem_u32(&bars[kDirMaxStages]);           // stage's weights landed (TMA bytes)
    const uint32_t empty0 = ptx::smem_u32(&bars[2 * kDirMaxStages]);       // stage consumed (MMA commit)
    const uint32_t slabf0 = ptx::smem_u32(&bars[3 * kDirMaxStages]);       // slab landed (TMA bytes)
    const uint32_t slabe0 = slabf0 + 8 * kDirMaxSlabs;                     // slab used (converter warps)
    const uint32_t accf0 = slabe0 + 8 * kDirMaxSlabs;                      // accumulator ready (MMA commit)
    const uint32_t acce0 = accf0 + 8 * kDirAccBufs;                        // accumulator read (128 threads)
    const uint32_t drain = acce0 + 8 * kDirAccBufs;
    const uint32_t stage_base = ptx::smem_u32(smem);
    const uint32_t slab_base = stage_base + (uint32_t)P.stages * P.stage_bytes;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < P.stages; ++s) {
            ptx::mbar_init(fulla0 + 8 * s, kDirConvWarps);
            ptx::mbar_init(fullb0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, 1);
        }
        for (int s = 0; s < P.slabs; ++s) {
            ptx::mbar_init(slabf0 + 8 * s, 1);
            ptx::mbar_init(slabe0 + 8 * s, kDirConvWarps);
        }
        for (int b = 0; b < kDirAccBufs; ++b) {
            ptx::mbar_init(accf0 + 8 * b, 1);
            ptx::mbar_init(acce0 + 8 * b, 128);
        }
        ptx::mbar_init(drain, 1);
        ptx::fence_mbar_init();
    }
    // The launch may overlap the end of the work before it in the stream (programmatic
    // dependent launch: the weight packing kernel lets it start early); no global memory is
    // read before that work has completed.
    grid_dependency_wait();
    for (int c = threadIdx.x; c < kDirAccCols; c += blockDim.x) {
        const float b = (P.bias && c < P.Cout) ? P.bias[c] : 0.f;
        s_bias[c] = b;
        s_bias_l2e[c] = c < P.Cout ? b * kLog2e : -__int_as_float(0x7f800000);
    }
    if (threadIdx.x < kDirGroups) s_grp[threadIdx.x] = P.grp[threadIdx.x];
    for (int i = threadIdx.x; i < kDirMaxSteps; i += blockDim.x) s_steps[i] = P.steps[i];
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&tmem_slot), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = tmem_slot;

    // ------------------------------------------------------------ producer
    if (warp == 0) {
        if (lane == 0) {
            ptx::prefetch_tmap(&P.x_map);
            int st = 0, sl = 0;
            uint32_t sph = 0, lph = 0;
            // per-slot bits: loaded at least once, and the parity of the last load
            uint32_t armed_st = 0, armed_st_ph = 0, armed_sl = 0, armed_sl_ph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x) {
                const DTile T = ddecode(P, s_grp, tile);
                const DGroup &G = s_grp[T.gi];
                for (int a = 0; ok && a < G.nt_d; ++a) {
                    if (!slice_live(P, G, T, a)) continue;
                    // the slice's slab of x
                    if (!ptx::mbar_wait_bounded(slabe0 + 8 * sl, lph ^ 1u, &abort_flag, kDirWaitNs)) {
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(slabf0 + 8 * sl, P.slab_bytes);
                    ptx::tma_load_5d(slab_base + (uint32_t)sl * P.slab_stride, &P.x_map, slabf0 + 8 * sl, P.w_lo,
                                     T.hb * P.TH + G.lo_h, T.qd + G.dd[a], 0, T.n);
                    armed_sl |= 1u << sl;
                    armed_sl_ph = (armed_sl_ph & ~(1u << sl)) | (lph << sl);
                    if (++sl == P.slabs) {
                        sl = 0;
                        lph ^= 1u;
                    }
                    // the weight slices of its K steps, one bulk copy into the stage's weight area
                    if (!ptx::mbar_wait_bounded(empty0 + 8 * st, sph ^ 1u, &abort_flag, kDirWaitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = fullb0 + 8 * st;
                    ptx::mbar_arrive_expect_tx(fb, G.sb_bytes);
                    ptx::bulk_load(stage_base + (uint32_t)st * P.stage_bytes + P.a_bytes,
                                   P.wdir + G.woff + (size_t)a * G.sb_bytes, G.sb_bytes, fb);
                    armed_st |= 1u << st;
                    armed_st_ph = (armed_st_ph & ~(1u << st)) | (sph << st);
                    if (++st == P.stages) {
                        st = 0;
                        sph ^= 1u;
                    }
                }
            }
            if (!ok) {
                drecord_error(P.status, kErrTimeout, 11);
                abort_flag = 1;
            }
            // Drain: every load this thread issued has landed before the CTA may exit.
            const volatile int never = 0;
            for (int s = 0; s < P.stages; ++s)
                if (armed_st & (1u << s)) ptx::mbar_wait_bounded(fullb0 + 8 * s, (armed_st_ph >> s) & 1u, &never, 200000000ull);
            for (int s = 0; s < P.slabs; ++s)
                if (armed_sl & (1u << s)) ptx::mbar_wait_bounded(slabf0 + 8 * s, (armed_sl_ph >> s) & 1u, &never, 200000000ull);
        }
    }
    // ---------------------------------------------------------- MMA issuer
    else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc1 =
                OPS == 4 ? ptx::idesc_f16((uint32_t)P.cout_pad) : ptx::idesc_bf16((uint32_t)P.cout_pad);
            const uint32_t idesc2 =
                OPS == 4 ? ptx::idesc_f16(2u * (uint32_t)P.cout_pad) : ptx::idesc_bf16(2u * (uint32_t)P.cout_pad);
            const uint64_t buf16 = (uint64_t)(P.buf_bytes >> 4);  // one buffer plane, 16-byte units
            int st = 0, it = 0;
            uint32_t sph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x, ++it) {
                const DTile T = ddecode(P, s_grp, tile);
                const DGroup &G = s_grp[T.gi];
                const int buf = it % kDirAccBufs;
                const uint32_t aph = (uint32_t)(it / kDirAccBufs) & 1u;
                if (!ptx::mbar_wait_bounded(acce0 + 8 * buf, aph ^ 1u, &abort_flag, kDirWaitNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t acc = tmem_base + (uint32_t)(buf * kDirAccCols);
                uint32_t ini = 0;  // bit c: class c's accumulator holds a product
                for (int a = 0; ok && a < G.nt_d; ++a) {
                    if (!slice_live(P, G, T, a)) continue;
                    if (!ptx::mbar_wait_bounded(fulla0 + 8 * st, sph, &abort_flag, kDirWaitNs) ||
                        !ptx::mbar_wait_bounded(fullb0 + 8 * st, sph, &abort_flag, kDirWaitNs)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    // the stage's descriptor; a step's operands are offsets from it (their start
                    // addresses stay below 2^18 bytes, so the additions never leave the field)
                    const uint64_t d0 = ptx::sdesc_k_swizzled(stage_base + (uint32_t)st * P.stage_bytes, kDirRowBytes);
                    const DStep *sp = s_steps + G.step0 + a * G.spa;
                    for (int j = 0; j < G.spa; ++j) {
                        const DStep e = sp[j];
                        const uint32_t mask = e.mask;
                        const uint32_t d_tmem = acc + (mask == 2u ? (uint32_t)P.cout_pad : 0u);
                        const uint32_t id = mask == 3u ? idesc2 : idesc1;
                        // shared offsets come first in every (d-slice, h-tap) run, so a step
                        // feeding both classes never finds one initialised and the other not
                        const uint32_t first = (ini & mask) ? 1u : 0u;
                        // buffer mi from row (dh - lo_h) * Qw on: a multiple of 8 rows (512 bytes)
                        const uint64_t a_hi = d0 + e.a16;
                        const uint64_t b_hi = d0 + e.b16;
                        const uint64_t b_lo = b_hi + e.blo16;
#pragma unroll
                        for (int kk = 0; kk < kDirK / 16; ++kk) {  // 16 bf16 (32 bytes) per MMA
                            const uint32_t acc_flag = kk ? 1u : first;
                            if constexpr (OPS == 3) {
                                ptx::mma_bf16(d_tmem, a_hi + 2 * kk, b_hi + 2 * kk, id, acc_flag);
                                ptx::mma_bf16(d_tmem, a_hi + 2 * kk, b_lo + 2 * kk, id, 1u);
                                ptx::mma_bf16(d_tmem, a_hi + buf16 + 2 * kk, b_hi + 2 * kk, id, 1u);
                            } else {
                                ptx::mma_bf16(d_tmem, a_hi + 2 * kk, b_hi + 2 * kk, id, acc_flag);
                            }
                        }
                        ini |= mask;
                    }
                    ptx::mma_commit(empty0 + 8 * st);
                    if (++st == P.stages) {
                        st = 0;
                        sph ^= 1u;
                    }
                }
                if (ok) ptx::mma_commit(accf0 + 8 * buf);
            }
            if (!ok) {
                drecord_error(P.status, kErrTimeout, 12);
                abort_flag = 1;
            }
            // Drain: all issued MMAs complete before tensor memory is released.
            ptx::mma_commit(drain);
            const volatile int never = 0;
            ptx::mbar_wait_bounded(drain, 0, &never, 200000000ull);
        }
    }
    // ---------------------------------------------------------- converters
    else if (warp < 2 + kDirConvWarps) {
        const int tid = (warp - 2) * 32 + lane;             // 0..kDirConvThreads-1
        const uint32_t plane = (uint32_t)(P.hfp * P.wfp);  // elements between channels in a slab
        int st = 0, sl = 0;
        uint32_t sph = 0, lph = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < P.total_tiles; tile += gridDim.x) {
            const DTile T = ddecode(P, s_grp, tile);
            const DGroup &G = s_grp[T.gi];
            for (int a = 0; ok && a < G.nt_d; ++a) {
                if (!slice_live(P, G, T, a)) continue;
                if (!warp_wait(slabf0 + 8 * sl, lph, &abort_flag) || !warp_wait(empty0 + 8 * st, sph ^ 1u, &abort_flag)) {
                    ok = false;
                    break;
                }
                const float *slab = reinterpret_cast<const float *>(smem + (size_t)(slab_base - stage_base) +
                                                                    (size_t)sl * P.slab_stride);
                uint8_t *stage = smem + (size_t)st * P.stage_bytes;
                // buffer mi, row r = (h', w): the 32 channels of x at slab row h', column
                // w + mdw[mi] - w_lo, in range by the slab's construction.  The rows of all
                // the slice's buffers are dealt to the converter threads in turn (no thread has more
                // than one row above another's); Qw is a power of two.
                int mi = 0, r = tid;
                while (mi < G.nm && r >= G.brows) {
                    r -= G.brows;
                    ++mi;
                }
                for (; mi < G.nm;) {
                    const int hp = r >> P.qw_shift, wq = r & (P.Qw - 1);
                    const int at = hp * P.wfp + (wq + G.mdw[mi] - P.w_lo);
                    uint32_t hi[16], lo[16];
                    if constexpr (X16) {
                        // the slab holds the operands: 16-bit channel pairs packed as they are
                        const uint16_t *src = reinterpret_cast<const uint16_t *>(slab) + at;
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            hi[k] = (uint32_t)src[(2 * k) * plane] | ((uint32_t)src[(2 * k + 1) * plane] << 16);
                    } else {
                    const float *src = slab + at;
                    float v[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) v[c] = src[c * plane];
                    const uint64_t neg1 = pack2(-1.f, -1.f);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        hi[k] = OPS == 4 ? f16x2_rn(v[2 * k], v[2 * k + 1]) : bf16x2_rn(v[2 * k], v[2 * k + 1]);
                        if constexpr (kPlanes == 2) {
                            // residuals v - hi of the pair in one packed fused multiply-add
                            const uint64_t h2 = pack2(__uint_as_float(hi[k] << 16), __uint_as_float(hi[k] & 0xFFFF0000u));
                            float r0, r1;
                            unpack2(ffma2(h2, neg1, pack2(v[2 * k], v[2 * k + 1])), r0, r1);
                            lo[k] = bf16x2_rn(r0, r1);
                        }
                    }
                    }
                    // 64-byte swizzle: 16-byte chunk j of row r lands at j ^ ((r >> 1) & 3)
                    uint8_t *row = stage + (size_t)mi * kPlanes * P.buf_bytes + (size_t)r * kDirRowBytes;
                    const uint32_t swz = (uint32_t)((r >> 1) & 3);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t o = ((uint32_t)c ^ swz) << 4;
                        *reinterpret_cast<uint4 *>(row + o) = make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
                        if constexpr (kPlanes == 2)
                            *reinterpret_cast<uint4 *>(row + P.buf_bytes + o) =
                                make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
                    }
                    r += kDirConvThreads;
                    while (mi < G.nm && r >= G.brows) {
                        r -= G.brows;
                        ++mi;
                    }
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::mbar_arrive(fulla0 + 8 * st);
                    ptx::mbar_arrive(slabe0 + 8 * sl);
                }
                if (++st == P.stages) {
                    st = 0;
                    sph ^= 1u;
                }
                if (++sl == P.slabs) {
                    sl = 0;
                    lph ^= 1u;
                }
            }
        }
        if (!ok) {
            if (lane == 0) drecord_error(P.status, kErrTimeout, 13);
            abort_flag = 1;
        }
    }
    // ------------------------------------------------------------ epilogue
    else {
        const int ew = warp - 2 - kDirConvWarps;
        const int eg = ew >> 2;        // epilogue group
        const int quarter = warp & 3;  // tensor-memory lane quarter this warp may access
        const int m = quarter * 32 + lane;
        const int hq_l = m / P.Qw, wq = m - hq_l * P.Qw;  // every row is used: TH * Qw = 128
        const uint32_t lane_base = tmem_base + ((uint32_t)(quarter * 32) << 16);
        const int C = P.Cout;
        const int nch = P.cout_pad / 16;
        const int V = P.Do * P.Ho * P.Wo;
        int it = 0;
        for (int tile = blockIdx.x; tile < P.total_tiles; tile += gridDim.x, ++it) {
            if (it % kDirEpiGroups != eg) continue;
            const DTile T = ddecode(P, s_grp, tile);
            const DGroup &G = s_grp[T.gi];
            const int buf = it % kDirAccBufs;
            const uint32_t aph = (uint32_t)(it / kDirAccBufs) & 1u;
            const uint32_t acc = lane_base + (uint32_t)(buf * kDirAccCols);
            if (!warp_wait(accf0 + 8 * buf, aph, &abort_flag)) {
                if (lane == 0) drecord_error(P.status, kErrTimeout, 14);
                abort_flag = 1;
                break;
            }
            ptx::tc_fence_after();
            // a tile none of whose d-slices reaches the input has no products: zeros
            bool live = false;
            for (int a = 0; a < G.nt_d; ++a) live |= slice_live(P, G, T, a);
            const int hq = T.hb * P.TH + hq_l;
            const int od = P.sd * T.qd + G.rd, oh = P.sh * hq + G.rh;
            float *yn = P.y + (size_t)T.n * C * V;
            const bool row_ok = hq < G.Qh;
            const bool valid0 = row_ok && wq < G.Qw0, valid1 = row_ok && wq < G.Qw1;
            const int off0 = row_ok ? (od * P.Ho + oh) * P.Wo + P.sw * wq : 0;  // class 0's column; class 1 is next
            float *dst = yn + off0;
            // each channel's (even, odd) output columns as one 8-byte store where the
            // rows allow (even output width)
            const bool pairs = P.Wo % 2 == 0;
            const bool full = C == P.cout_pad;  // no ragged last chunk
            // 16 channels c0.. of the row: class 0 in a, class 1 in b
            auto store16 = [&](int c0, const float (&a)[16], const float (&b)[16]) {
                if constexpr (X16) {  // 16-bit y: the pair as one 4-byte store
                    uint16_t *d16 = reinterpret_cast<uint16_t *>(P.y) + (size_t)T.n * C * V + off0;
                    if (full && valid1 && pairs) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            *reinterpret_cast<uint32_t *>(d16 + (size_t)(c0 + i) * V) = cvt16x2(a[i], b[i], P.io16);
                        return;
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        if (c0 + i >= C) break;
                        if (valid0) d16[(size_t)(c0 + i) * V] = cvt16(a[i], P.io16);
                        if (valid1) d16[(size_t)(c0 + i) * V + 1] = cvt16(b[i], P.io16);
                    }
                    return;
                }
                if (full && valid1 && pairs) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        *reinterpret_cast<float2 *>(dst + (size_t)(c0 + i) * V) = make_float2(a[i], b[i]);
                    return;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (c0 + i >= C) break;
                    if (valid0) dst[(size_t)(c0 + i) * V] = a[i];
                    if (valid1) dst[(size_t)(c0 + i) * V + 1] = b[i];
                }
            };
            if constexpr (EPI == CONVT3D_EPI_IDENTITY) {
                // conv + bias, 16 channels at a time
#pragma unroll 1
                for (int j = 0; j < nch; ++j) {
                    float t0[16], t1[16];
                    ptx::tmem_ld16(acc + (uint32_t)(16 * j), t0);
                    ptx::tmem_ld16(acc + (uint32_t)(P.cout_pad + 16 * j), t1);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float b = s_bias[16 * j + i];
                        t0[i] = (live ? t0[i] : 0.f) + b;
                        t1[i] = (live ? t1[i] : 0.f) + b;
                    }
                    store16(16 * j, t0, t1);
                }
            } else {
                // softmax over channels then sigmoid, per class, in the base-2 domain:
                // u = (conv + bias) log2(e), weight 2^(u - M) / S (channels past Cout have
                // u = -inf, weight 0).  The row's values stay in tensor memory between the
                // passes, 16 channels at a time: logits (and their max), exponentials (and
                // their sum), then the sigmoid; class 0's results wait there until class 1's
                // are formed, so that each channel's two columns go out together.
                const uint64_t l2e2 = pack2(kLog2e, kLog2e);
                const uint64_t half2 = pack2(0.5f, 0.5f);
#pragma unroll 1
                for (int cls = 0; cls < 2; ++cls) {
                    const uint32_t col = acc + (uint32_t)(cls * P.cout_pad);
                    float mx = -__int_as_float(0x7f800000);
                    // a tile with no products (no live d-slice) has logits = bias alone: a
                    // separate loop, so that the live one carries no per-value select
                    if (live) {
#pragma unroll 1
                        for (int j = 0; j < nch; ++j) {
                            float v[16];
                            ptx::tmem_ld16(col + (uint32_t)(16 * j), v);
                            ptx::tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const uint64_t u =
                                    ffma2(pack2(v[2 * k], v[2 * k + 1]), l2e2,
                                          *reinterpret_cast<const uint64_t *>(&s_bias_l2e[16 * j + 2 * k]));
                                unpack2(u, v[2 * k], v[2 * k + 1]);
                            }
                            mx = max17(mx, v);
                            ptx::tmem_st16(col + (uint32_t)(16 * j), v);
                        }
                    } else {
#pragma unroll 1
                        for (int j = 0; j < nch; ++j) {
                            float v[16];
#pragma unroll
                            for (int k = 0; k < 16; ++k) v[k] = s_bias_l2e[16 * j + k];
                            mx = max17(mx, v);
                            ptx::tmem_st16(col + (uint32_t)(16 * j), v);
                        }
                    }
                    ptx::tmem_wait_st();
                    const uint64_t nm2 = pack2(-mx, -mx);
                    uint64_t s2 = pack2(0.f, 0.f);
#pragma unroll 1
                    for (int j = 0; j < nch; ++j) {
                        float v[16];
                        ptx::tmem_ld16(col + (uint32_t)(16 * j), v);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            float a, b;
                            unpack2(fadd2(pack2(v[2 * k], v[2 * k + 1]), nm2), a, b);
                            v[2 * k] = ex2_approx(a);
                            v[2 * k + 1] = ex2_approx(b);
                            s2 = fadd2(s2, pack2(v[2 * k], v[2 * k + 1]));
                        }
                        ptx::tmem_st16(col + (uint32_t)(16 * j), v);
                    }
                    ptx::tmem_wait_st();
                    float sa, sb;
                    unpack2(s2, sa, sb);
                    uint64_t A[3];
                    sigmoid3_coefficients(__frcp_rn(sa + sb), A);
#pragma unroll 1
                    for (int j = 0; j < nch; ++j) {
                        float v[16], w[16];
                        ptx::tmem_ld16(col + (uint32_t)(16 * j), v);
                        if (cls == 1) ptx::tmem_ld16(acc + (uint32_t)(16 * j), w);  // class 0's results
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint64_t e = pack2(v[2 * k], v[2 * k + 1]);
                            const uint64_t e2 = fmul2(e, e);
                            uint64_t t = ffma2(A[2], e2, A[1]);
                            t = ffma2(t, e2, A[0]);
                            unpack2(ffma2(t, e, half2), v[2 * k], v[2 * k + 1]);
                        }
                        if (cls == 0)
                            ptx::tmem_st16(col + (uint32_t)(16 * j), v);
                        else
                            store16(16 * j, w, v);
                    }
                    ptx::tmem_wait_st();
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(acce0 + 8 * buf);
        }
    }
    __syncthreads();
    if (warp == 1) ptx::tmem_dealloc(tmem_base, 512);
}

// ----------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled(cudaError_t &err) {
    static cudaError_t e0 = cudaSuccess;
    static EncodeTiledFn fn = [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        e0 = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
        return (e0 == cudaSuccess && q == cudaDriverEntryPointSuccess) ? (EncodeTiledFn)p : nullptr;
    }();
    err = e0;
    return fn;
}

// The kernel's tables and slab geometry for a plan, or false when the plan is
// outside what the kernel handles.
bool direct_geometry(const convt3d_plan_s &p, DirectParams &P) {
    const Geometry &g = p.g;
    const int epi = p.d.epilogue;
    // 16-bit x and y only with the single-product precision of their own format (the plan's
    // validation pairs io_bf16 with BF16 and io_fp16 with FP16)
    if (!p.tc || !p.merged || p.cl || !p.bf16 || p.nslices != 1 || (p.io16 != kF32 && p.planes != 1)) return false;
    if (epi != CONVT3D_EPI_SOFTMAX_SIGMOID && epi != CONVT3D_EPI_IDENTITY) return false;
    const int eb = p.io16 != kF32 ? 2 : 4;  // bytes per element of x
    const int al = 16 / eb;                  // elements per 16 bytes: TMA strides and x-coordinates
    if (g.Cin > kDirK || g.Win % al != 0 || p.cout_pad > 64 || p.ngroups > kDirGroups) return false;
    memset(&P, 0, sizeof(P));
    P.io16 = p.io16;
    P.N = g.N;
    P.Cout = g.Cout;
    P.cout_pad = p.cout_pad;
    P.Din = g.Din;
    P.Do = g.Do;
    P.Ho = g.Ho;
    P.Wo = g.Wo;
    P.sd = g.ss[0];
    P.sh = g.ss[1];
    P.sw = g.ss[2];
    P.Qw = p.grp[0].Qw;
    // rows of whole 8-row swizzle atoms, whole rows per tile: Qw a multiple of 8 dividing 128
    if (P.Qw < 8 || P.Qw > 128 || P.Qw % 8 != 0 || 128 % P.Qw != 0) return false;
    P.TH = 128 / P.Qw;
    while ((1 << P.qw_shift) < P.Qw) ++P.qw_shift;
    P.ngroups = p.ngroups;
    P.b_bytes = (uint32_t)p.cout_pad * kDirRowBytes;
    const uint32_t planes = (uint32_t)p.planes;
    int dw_min = 1 << 20, dw_max = -(1 << 20), span_h = 0, ns = 0, prefix = 0, nm_max = 1, brows_max = 0;
    uint32_t sb_max = 0, woff = 0;
    for (int gi = 0; gi < p.ngroups; ++gi) {
        const GroupDesc &S = p.grp[gi];
        if (S.ncls != 2 || S.Qw != P.Qw || S.nm > 8) return false;
        const ClassDesc &C0 = g.cls[S.cls[0]], &C1 = g.cls[S.cls[1]];
        if (C0.rw != 0 || C1.rw != 1 || C0.nt_d != C1.nt_d || C0.nt_h != C1.nt_h || C0.nt_d > 8) return false;
        DGroup &G = P.grp[gi];
        G.Qd = S.Qd;
        G.Qh = S.Qh;
        G.Qw0 = C0.Qw;
        G.Qw1 = C1.Qw;
        G.rd = C0.rd;
        G.rh = C0.rh;
        G.nt_d = C0.nt_d;
        G.nm = S.nm;
        G.spa = C0.nt_h * S.nm;
        G.step0 = ns;
        G.lo_h = C0.lo_h;
        for (int mi = 0; mi < S.nm; ++mi) G.mdw[mi] = S.mdw[mi];
        int hi_h = C0.lo_h;
        for (int a = 0; a < C0.nt_d; ++a) G.dd[a] = g.taps[C0.tap_begin + a * C0.nt_h * C0.nt_w].dd;
        if (ns + G.nt_d * G.spa > kDirMaxSteps) return false;
        uint32_t boff = 0;
        for (int a = 0; a < C0.nt_d; ++a, boff = 0)
            for (int b = 0; b < C0.nt_h; ++b)
                for (int mi = 0; mi < S.nm; ++mi) {
                    const int mask = S.mmask[mi];
                    const int t0 = (mask & 1) ? C0.tap_begin + (a * C0.nt_h + b) * C0.nt_w + S.me[mi][0] : -1;
                    const int t1 = (mask & 2) ? C1.tap_begin + (a * C1.nt_h + b) * C1.nt_w + S.me[mi][1] : -1;
                    const TapDesc &td = g.taps[(mask & 1) ? t0 : t1];
                    DStep &e = P.steps[ns++];
                    e.dh = td.dh;
                    e.dw = td.dw;
                    e.mask = (uint8_t)mask;
                    e.mi = (uint8_t)mi;
                    e.tb0 = (int16_t)((mask & 1) ? t0 : t1);
                    e.tb1 = (int16_t)(mask == 3 ? t1 : -1);
                    e.boff = boff;
                    boff += planes * (mask == 3 ? 2u : 1u) * P.b_bytes;
                    G.sb_bytes = boff;  // the same for every d-slice
                    dw_min = td.dw < dw_min ? td.dw : dw_min;
                    dw_max = td.dw > dw_max ? td.dw : dw_max;
                    hi_h = td.dh > hi_h ? td.dh : hi_h;
                }
        sb_max = G.sb_bytes > sb_max ? G.sb_bytes : sb_max;
        G.woff = woff;
        woff += (uint32_t)G.nt_d * G.sb_bytes;
        const int sph = hi_h - G.lo_h;
        span_h = sph > span_h ? sph : span_h;
        G.brows = (P.TH + sph) * P.Qw;
        brows_max = G.brows > brows_max ? G.brows : brows_max;
        nm_max = G.nm > nm_max ? G.nm : nm_max;
        G.nhb = (G.Qh + P.TH - 1) / P.TH;
        G.tiles = G.Qd * G.nhb;
        G.div_nhb = make_fastdiv((uint32_t)(G.nhb > 0 ? G.nhb : 1));
        G.tile_prefix = prefix;
        prefix += G.tiles;
    }
    P.w_lo = dw_min >= 0 ? dw_min / al * al : -((-dw_min + al - 1) / al * al);
    P.wfp = (P.Qw + dw_max - P.w_lo + al - 1) / al * al;
    P.hfp = P.TH + span_h;
    if (P.wfp > 256 || P.hfp > 256) return false;
    P.slab_bytes = (uint32_t)(P.wfp * P.hfp * kDirK * eb);
    P.slab_stride = (P.slab_bytes + 127u) / 128u * 128u;
    P.wdir_bytes = woff;
    P.tiles_per_sample = prefix;
    P.div_tps = make_fastdiv((uint32_t)(prefix > 0 ? prefix : 1));
    const int64_t total = (int64_t)prefix * g.N;
    if (prefix < 1 || total >= ((int64_t)1 << 31)) return false;
    P.total_tiles = (int)total;
    P.buf_bytes = (uint32_t)brows_max * kDirRowBytes;  // a multiple of 512: whole swizzle atoms
    P.a_bytes = ((uint32_t)nm_max * planes * P.buf_bytes + 1023u) / 1024u * 1024u;
    P.stage_bytes = P.a_bytes + (sb_max + 1023u) / 1024u * 1024u;
    for (int gi = 0; gi < P.ngroups; ++gi) {
        const DGroup &G = P.grp[gi];
        for (int j = 0; j < G.nt_d * G.spa; ++j) {
            DStep &e = P.steps[G.step0 + j];
            const uint32_t arow = (uint32_t)P.Qw * kDirRowBytes;
            e.a16 = (uint16_t)(((uint32_t)e.mi * planes * P.buf_bytes + (uint32_t)(e.dh - G.lo_h) * arow) >> 4);
            e.b16 = (uint16_t)((P.a_bytes + e.boff) >> 4);
            e.blo16 = (uint16_t)(((e.tb1 >= 0 ? 2u : 1u) * P.b_bytes) >> 4);
        }
    }
    // shared memory beside the static tables (under 4 KB) and the alignment slack (227 KB per
    // block): 1..3 slabs, 2..4 stages
    const size_t budget = 232448 - 4096 - 1024;
    P.slabs = 3;
    while (P.slabs > 1 && (size_t)P.slabs * P.slab_stride + 2 * (size_t)P.stage_bytes > budget) --P.slabs;
    const size_t used = (size_t)P.slabs * P.slab_stride;
    P.stages = used < budget ? (int)((budget - used) / P.stage_bytes) : 0;
    if (P.stages > kDirMaxStages) P.stages = kDirMaxStages;
    return P.stages >= 2;
}

// One weight slice of the packed weight: cout_pad rows of 32 bf16 channels (64
// bytes, 16-byte chunks stored at chunk ^ ((row >> 1) & 3)) of tap widx, hi or lo.
struct DPackEntry {
    uint32_t dst;
    int16_t widx;
    uint8_t lo, pad_;
};
constexpr int kDirMaxPack = 1024;
struct DPackParams {
    const float *w;
    uint8_t *dst;
    int Cin, Cout, k3, cout_pad, cin_g, cout_g, split, half, w16, n;
    DPackEntry e[kDirMaxPack];
};

// One block per weight slice, four threads per row: each writes one 16-byte chunk
// (8 input channels) of the row, split into bf16 hi and lo (rounded to nearest
// even, lo = bf16(v - hi)).  w is [Cin][Cout/G][taps]; channels of different
// convolution groups, and rows or channels past Cout or Cin, are zero.
__global__ void pack_direct_kernel(const __grid_constant__ DPackParams Q) {
    grid_launch_dependents();  // the GEMM may launch and set up meanwhile
    const DPackEntry E = Q.e[blockIdx.x];
    const int r = threadIdx.x >> 2, pch = threadIdx.x & 3;
    if (r >= Q.cout_pad) return;
    const int jc = pch ^ ((r >> 1) & 3);  // the logical chunk this physical chunk holds
    const int co = r;
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        float v[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int ci = 8 * jc + e + q;
            v[q] = 0.f;
            if (ci < Q.Cin && co < Q.Cout && ci / Q.cin_g == co / Q.cout_g)
            {
                const int64_t src = ((int64_t)ci * Q.cout_g + co % Q.cout_g) * Q.k3 + E.widx;
                v[q] = Q.w16 ? ld16(Q.w, src, Q.w16) : Q.w[src];
            }
        }
        uint32_t h = Q.half ? f16x2_rn(v[0], v[1]) : bf16x2_rn(v[0], v[1]);
        if (E.lo) {
            const float h0 = __uint_as_float(h << 16), h1 = __uint_as_float(h & 0xFFFF0000u);
            h = bf16x2_rn(v[0] - h0, v[1] - h1);
        }
        out[e / 2] = h;
    }
    *reinterpret_cast<uint4 *>(Q.dst + E.dst + (size_t)r * kDirRowBytes + (size_t)pch * 16) =
        make_uint4(out[0], out[1], out[2], out[3]);
}

// The weight slices in the packed weight's order (pair, d-slice, K step, plane,
// class slot), each placed where the stage image of its slice puts it.
bool direct_pack_table(const convt3d_plan_s &p, const DirectParams &P, DPackParams &Q) {
    Q.n = 0;
    for (int gi = 0; gi < P.ngroups; ++gi) {
        const DGroup &G = P.grp[gi];
        for (int a = 0; a < G.nt_d; ++a)
            for (int j = 0; j < G.spa; ++j) {
                const DStep &st = P.steps[G.step0 + a * G.spa + j];
                const uint32_t nb = st.tb1 >= 0 ? 2u : 1u;
                for (int plane = 0; plane < p.planes; ++plane)
                    for (uint32_t slot = 0; slot < nb; ++slot) {
                        if (Q.n >= kDirMaxPack) return false;
                        DPackEntry &en = Q.e[Q.n++];
                        en.dst = G.woff + (uint32_t)a * G.sb_bytes + st.boff + ((uint32_t)plane * nb + slot) * P.b_bytes;
                        en.widx = p.g.taps[slot ? st.tb1 : st.tb0].widx;
                        en.lo = (uint8_t)plane;
                    }
            }
    }
    Q.Cin = p.g.Cin;
    Q.Cout = p.g.Cout;
    Q.k3 = p.g.kvol;
    Q.cout_pad = p.cout_pad;
    Q.cin_g = p.g.Cin / p.g.G;
    Q.cout_g = p.g.Cout / p.g.G;
    Q.split = p.planes == 2;
    Q.half = p.half;
    Q.w16 = p.io16;
    return true;
}

struct DirectCache {
    DirectParams P;
    DPackParams Q;
    const void *key[2];
    void (*kern)(const DirectParams);
    size_t smem;
    int grid;
    bool ready;
};

// The plan's launch state: tables, kernel instance, shared memory and grid.
cudaError_t direct_prepare(convt3d_plan_s &p, DirectCache *&out) {
    if (!p.direct_cache) {
        DirectCache *c = new (std::nothrow) DirectCache();
        if (!c) return cudaErrorMemoryAllocation;
        c->ready = false;
        p.direct_cache = c;
    }
    DirectCache &dc = *static_cast<DirectCache *>(p.direct_cache);
    out = &dc;
    if (dc.ready) return cudaSuccess;
    DirectParams &P = dc.P;
    cudaError_t e;
    if (!direct_geometry(p, P)) return cudaErrorInvalidConfiguration;
    if (!direct_pack_table(p, P, dc.Q)) return cudaErrorInvalidConfiguration;
    const bool split = p.planes == 2;
    const bool sm = p.d.epilogue == CONVT3D_EPI_SOFTMAX_SIGMOID, x16 = p.io16 != kF32;
    constexpr int SM = CONVT3D_EPI_SOFTMAX_SIGMOID, ID = CONVT3D_EPI_IDENTITY;
    if (split)
        dc.kern = sm ? convt3d_direct_gemm<SM, 3, false> : convt3d_direct_gemm<ID, 3, false>;
    else if (p.half)
        dc.kern = x16 ? (sm ? convt3d_direct_gemm<SM, 4, true> : convt3d_direct_gemm<ID, 4, true>)
                      : (sm ? convt3d_direct_gemm<SM, 4, false> : convt3d_direct_gemm<ID, 4, false>);
    else
        dc.kern = x16 ? (sm ? convt3d_direct_gemm<SM, 2, true> : convt3d_direct_gemm<ID, 2, true>)
                      : (sm ? convt3d_direct_gemm<SM, 2, false> : convt3d_direct_gemm<ID, 2, false>);
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, dc.kern)) != cudaSuccess) return e;
    dc.smem = 1024 + (size_t)P.stages * P.stage_bytes + (size_t)P.slabs * P.slab_stride;
    if (dc.smem + fa.sharedSizeBytes > 232448) return cudaErrorInvalidConfiguration;
    if ((e = cudaFuncSetAttribute(dc.kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dc.smem)) != cudaSuccess)
        return e;
    int dev = 0, sms = 148;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    dc.grid = P.total_tiles < sms ? P.total_tiles : sms;
    dc.key[0] = dc.key[1] = nullptr;
    dc.ready = true;
    return cudaSuccess;
}

}  // namespace

bool direct_supported(const convt3d_plan_s &p) {
    DirectParams *P = new (std::nothrow) DirectParams();
    if (!P) return false;
    const bool ok = direct_geometry(p, *P);
    delete P;
    return ok;
}

size_t direct_weight_bytes(const convt3d_plan_s &p) {
    DirectParams *P = new (std::nothrow) DirectParams();
    if (!P) return 0;
    const size_t n = direct_geometry(p, *P) ? P->wdir_bytes : 0;
    delete P;
    return n;
}

void direct_cache_free(void *c) { delete static_cast<DirectCache *>(c); }

cudaError_t launch_direct_pack(convt3d_plan_s &p, const float *w, void *dst, cudaStream_t s) {
    static_assert(sizeof(DPackParams) < 32000, "kernel parameter block too large");
    DirectCache *dc = nullptr;
    cudaError_t e = direct_prepare(p, dc);
    if (e != cudaSuccess) return e;
    dc->Q.w = w;
    dc->Q.dst = static_cast<uint8_t *>(dst);
    pack_direct_kernel<<<dc->Q.n, 4 * p.cout_pad, 0, s>>>(dc->Q);
    return cudaGetLastError();
}

cudaError_t launch_direct(convt3d_plan_s &p, const float *x, const void *wdir, const float *bias, float *y,
                          uint32_t *status, cudaStream_t s) {
    static_assert(sizeof(DirectParams) < 32000, "kernel parameter block too large");
    DirectCache *dcp = nullptr;
    cudaError_t e = direct_prepare(p, dcp);
    if (e != cudaSuccess) return e;
    DirectCache &dc = *dcp;
    DirectParams &P = dc.P;
    if (dc.key[0] != x) {
        cudaError_t ferr;
        EncodeTiledFn enc = encode_tiled(ferr);
        if (!enc) return ferr != cudaSuccess ? ferr : cudaErrorNotSupported;
        const Geometry &g = p.g;
        // x: NCDHW (fp32, or the 16-bit operand format), box = one slab (all 32 channel planes of
        // the tile's rows and halo)
        const cuuint64_t xdim[5] = {(cuuint64_t)g.Win, (cuuint64_t)g.Hin, (cuuint64_t)g.Din, (cuuint64_t)g.Cin,
                                    (cuuint64_t)g.N};
        const cuuint64_t eb = p.io16 != kF32 ? 2 : 4;
        const cuuint64_t xstr[4] = {(cuuint64_t)g.Win * eb, (cuuint64_t)g.Win * g.Hin * eb,
                                    (cuuint64_t)g.Win * g.Hin * g.Din * eb, (cuuint64_t)g.Win * g.Hin * g.Din * g.Cin * eb};
        const cuuint32_t xbox[5] = {(cuuint32_t)P.wfp, (cuuint32_t)P.hfp, 1, (cuuint32_t)kDirK, 1};
        const cuuint32_t es[5] = {1, 1, 1, 1, 1};
        const CUtensorMapDataType xdt = p.io16 == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                        : p.io16 == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        if (enc(&P.x_map, xdt, 5, (void *)x, xdim, xstr, xbox, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        dc.key[0] = x;
    }
    P.wdir = static_cast<const uint8_t *>(wdir);
    P.bias = bias;
    P.y = y;
    P.status = status;
    // Launched as a programmatic dependent of the work before it in the stream: it may start
    // once that work lets it (the weight packing kernel does at its start; any other kernel at
    // its end) and sets up its barriers and tensor memory meanwhile; every thread waits for that
    // work to complete before its first global-memory read.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)dc.grid);
    cfg.blockDim = dim3(kDirThreads);
    cfg.dynamicSmemBytes = dc.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, dc.kern, P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace convt3d
