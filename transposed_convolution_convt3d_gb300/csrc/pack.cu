// Weight re-layout and input staging.
//
// The weight of a ConvTranspose3d is [Cin, Cout/G, kd, kh, kw] (PyTorch layout,
// as on all three transcript pages, where G = 1); page l2_p49 notes the Cin stride makes
// per-Cout access strided and re-lays it per output channel.  Here the
// weight is re-laid per parity class and tap:
//   tensor-core path: [tap][Cout_pad][Cin_pad] (K-major rows, Cin contiguous),
//                     split into TF32 (or bf16) hi and lo planes, or one TF32,
//                     bf16 or fp16 plane;
//   FFMA path:        [tap][Cin_pad][Cout_pad] fp32.
// The tensor-core path also stages x (NCDHW, or already channels-last) into channels-last
// [N][D][H][W][Cin_pad] hi/lo planes (one TF32-rounded, bf16 or fp16 plane for
// the single-product precisions), the layout its TMA im2col loads read.
// x and w may arrive as bf16 or fp16 arrays (kind w16 / x16).

#include "convt3d_internal.h"

namespace convt3d {
namespace {

// Split v into a TF32-exact head (low 13 mantissa bits cleared) and the
// exact fp32 remainder: v == hi + lo, |lo| < 2^-10 |v|.
__device__ __forceinline__ void split_tf32(float v, float &hi, float &lo) {
    hi = __uint_as_float(__float_as_uint(v) & 0xFFFFE000u);
    lo = v - hi;
}

// Round v to the nearest TF32 value (ties away from zero): the PTX
// conversion cvt.rna.tf32.f32, whose result keeps 10 explicit mantissa bits.
__device__ __forceinline__ float round_tf32(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

// Split v into a bf16 head and a bf16 tail, both rounded to nearest even:
// v - hi is exact in fp32 and |v - hi - lo| <= 2^-16 |v| (two 8-bit halves of
// a 16-bit significand).
__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(v);
    lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

struct TapIndex {
    int16_t widx[kMaxTaps];
};

// Grouped convolution (G > 1): w is [Cin, Cout/G, taps]; the packed copy is the
// dense [Cout][Cin] matrix per tap with zeros where ci and co lie in different
// groups, so the GEMM needs no knowledge of groups.
__global__ void pack_weights_kernel(const float *__restrict__ w, float *__restrict__ hi,
                                    float *__restrict__ lo, int Cin, int Cout, int k3, int ntaps,
                                    int cin_pad, int cout_pad, int kmajor, int mode, int cin_g, int cout_g,
                                    int w16, const __grid_constant__ TapIndex taps) {
    const int64_t total = (int64_t)ntaps * cin_pad * cout_pad;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        int j, ci, co;
        if (kmajor) {  // [tap][co][ci]
            ci = (int)(i % cin_pad);
            co = (int)((i / cin_pad) % cout_pad);
            j = (int)(i / ((int64_t)cin_pad * cout_pad));
        } else {       // [tap][ci][co]
            co = (int)(i % cout_pad);
            ci = (int)((i / cout_pad) % cin_pad);
            j = (int)(i / ((int64_t)cin_pad * cout_pad));
        }
        float v = 0.0f;
        if (ci < Cin && co < Cout && ci / cin_g == co / cout_g) {
            const int64_t src = ((int64_t)ci * cout_g + co % cout_g) * k3 + taps.widx[j];
            v = w16 ? ld16(w, src, w16) : w[src];
        }
        if (lo && mode == 3) {  // split bf16 planes (2-byte elements)
            split_bf16(v, reinterpret_cast<__nv_bfloat16 *>(hi)[i], reinterpret_cast<__nv_bfloat16 *>(lo)[i]);
        } else if (lo) {
            float h, l;
            split_tf32(v, h, l);
            hi[i] = h;
            lo[i] = l;
        } else if (mode == 2 || mode == 4) {  // bf16 / fp16 operands: the plane holds 2-byte elements
            reinterpret_cast<uint16_t *>(hi)[i] = cvt16(v, mode == 4 ? kF16 : kBF16);
        } else {
            hi[i] = mode == 1 ? round_tf32(v) : v;  // TF32-rounded, or fp32 for the FFMA path
        }
    }
}

// Tensor-core layout [tap][cout_pad][cin_pad] through a 32 x 32 shared-memory
// tile per (output channel, 32 taps, 32 input channels): the reads run along
// the weight's contiguous tap axis, the writes along cin, both coalesced.
// mode: 0 = split TF32 (fp32 hi/lo planes), 1 = TF32-rounded, 2 = bf16,
// 3 = split bf16 (bf16 hi/lo planes), 4 = fp16.
__global__ void pack_weights_kmajor_kernel(const float *__restrict__ w, float *__restrict__ hi,
                                           float *__restrict__ lo, int Cin, int Cout, int k3, int ntaps,
                                           int cin_pad, int cout_pad, int mode, int cin_g, int cout_g, int w16,
                                           const __grid_constant__ TapIndex taps) {
    __shared__ float tile[32][33];  // [ci][tap]
    __shared__ int s_widx[32];      // this block's taps: one parameter read each (lanes that index
                                    // the parameter table with different taps would serialise)
    const int ci0 = blockIdx.x * 32, j0 = blockIdx.y * 32, co = blockIdx.z;
    const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
    const bool co_ok = co < Cout;
    if (ty == 0) s_widx[tx] = j0 + tx < ntaps ? taps.widx[j0 + tx] : 0;
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 32; r += 8) {
        const int ci = ci0 + ty + r, j = j0 + tx;
        float v = 0.0f;
        if (co_ok && ci < Cin && j < ntaps && ci / cin_g == co / cout_g) {
            const int64_t src = ((int64_t)ci * cout_g + co % cout_g) * k3 + s_widx[tx];
            v = w16 ? ld16(w, src, w16) : w[src];
        }
        tile[ty + r][tx] = v;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 32; r += 8) {
        const int j = j0 + ty + r, ci = ci0 + tx;
        if (j >= ntaps || ci >= cin_pad) continue;
        const int64_t i = ((int64_t)j * cout_pad + co) * cin_pad + ci;
        const float v = tile[tx][ty + r];
        if (mode == 3) {
            split_bf16(v, reinterpret_cast<__nv_bfloat16 *>(hi)[i], reinterpret_cast<__nv_bfloat16 *>(lo)[i]);
        } else if (mode == 0) {
            float h, l;
            split_tf32(v, h, l);
            hi[i] = h;
            lo[i] = l;
        } else if (mode == 2 || mode == 4) {
            reinterpret_cast<uint16_t *>(hi)[i] = cvt16(v, mode == 4 ? kF16 : kBF16);
        } else {
            hi[i] = round_tf32(v);
        }
    }
}

// NCDHW -> NDHWC(+channel padding) transpose of one sample, 32 positions x
// 32 channels per block through shared memory; both the global read (along
// positions) and the write (along channels) are 128-byte rows.
__global__ void stage_input_kernel(const float *__restrict__ x, float *__restrict__ hi,
                                   float *__restrict__ lo, int Cin, int cin_pad, int64_t S, int bf16, int x16) {
    // bf16: the 16-bit operand kind (kBF16 / kF16), 0 for fp32 planes; x16: x's kind
    __shared__ float tile[32][33];
    const int n = blockIdx.z;
    const int c0 = blockIdx.y * 32;
    const int64_t s0 = (int64_t)blockIdx.x * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
    const int64_t xb = (int64_t)n * Cin * S;
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
        const int c = c0 + ty + j;
        const int64_t s = s0 + tx;
        const int64_t i = xb + (int64_t)c * S + s;
        tile[ty + j][tx] = (c < Cin && s < S) ? (x16 ? ld16(x, i, x16) : x[i]) : 0.0f;
    }
    __syncthreads();
    float *hn = hi + (int64_t)n * S * cin_pad;
    float *ln = lo ? lo + (int64_t)n * S * cin_pad : nullptr;
#pragma unroll
    for (int j = 0; j < 32; j += 8) {
        const int64_t s = s0 + ty + j;
        const int c = c0 + tx;
        if (s < S) {
            if (ln && bf16) {  // split bf16 planes (2-byte elements)
                const int64_t o = ((int64_t)n * S + s) * cin_pad + c;
                split_bf16(tile[tx][ty + j], reinterpret_cast<__nv_bfloat16 *>(hi)[o],
                           reinterpret_cast<__nv_bfloat16 *>(lo)[o]);
            } else if (ln) {
                float h, l;
                split_tf32(tile[tx][ty + j], h, l);
                hn[s * cin_pad + c] = h;
                ln[s * cin_pad + c] = l;
            } else if (bf16) {  // single bf16 or fp16 plane (2-byte elements)
                reinterpret_cast<uint16_t *>(hi)[((int64_t)n * S + s) * cin_pad + c] = cvt16(tile[tx][ty + j], bf16);
            } else {  // single TF32 plane
                hn[s * cin_pad + c] = round_tf32(tile[tx][ty + j]);
            }
        }
    }
}

// Channels-last input [N][D][H][W][Cin] -> the same rows padded to cin_pad
// channels (hi/lo planes, or one TF32 / bf16 plane): no transpose, 8 rows x
// 32 channels per block, coalesced on both sides.
__global__ void stage_input_cl_kernel(const float *__restrict__ x, float *__restrict__ hi, float *__restrict__ lo,
                                      int Cin, int cin_pad, int64_t rows, int bf16, int x16) {
    const int64_t r = (int64_t)blockIdx.x * 8 + threadIdx.y;
    const int c = blockIdx.y * 32 + threadIdx.x;
    if (r >= rows) return;
    const float v = c >= Cin ? 0.0f : (x16 ? ld16(x, r * Cin + c, x16) : __ldg(x + r * Cin + c));
    const int64_t o = r * cin_pad + c;
    if (lo && bf16) {
        split_bf16(v, reinterpret_cast<__nv_bfloat16 *>(hi)[o], reinterpret_cast<__nv_bfloat16 *>(lo)[o]);
    } else if (lo) {
        float h, l;
        split_tf32(v, h, l);
        hi[o] = h;
        lo[o] = l;
    } else if (bf16) {
        reinterpret_cast<uint16_t *>(hi)[o] = cvt16(v, bf16);
    } else {
        hi[o] = round_tf32(v);
    }
}

}  // namespace

cudaError_t launch_pack_weights(const convt3d_plan_s &p, const float *w, float *hi, float *lo, int kmajor,
                                cudaStream_t s) {
    TapIndex t;
    for (int j = 0; j < kMaxTaps; ++j) t.widx[j] = j < p.g.ntaps ? p.g.taps[j].widx : 0;
    const int mode = p.bf16 ? (p.planes == 2 ? 3 : (p.half ? 4 : 2)) : (p.planes == 1 ? 1 : 0);
    if (kmajor) {  // tensor-core layout (cout_pad rows of every tap; cin_pad is a multiple of 32)
        dim3 grid((unsigned)(p.cin_pad / 32), (unsigned)((p.g.ntaps + 31) / 32), (unsigned)p.cout_pad);
        pack_weights_kmajor_kernel<<<grid, dim3(32, 8), 0, s>>>(w, hi, lo, p.g.Cin, p.g.Cout, p.g.kvol, p.g.ntaps,
                                                                p.cin_pad, p.cout_pad, mode, p.g.Cin / p.g.G,
                                                                p.g.Cout / p.g.G, p.io16, t);
        return cudaGetLastError();
    }
    const int64_t total = (int64_t)p.g.ntaps * p.cin_pad * p.cout_pad;
    const int threads = 256;
    const int blocks = (int)((total + threads - 1) / threads < 4096 ? (total + threads - 1) / threads : 4096);
    pack_weights_kernel<<<blocks, threads, 0, s>>>(w, hi, lo, p.g.Cin, p.g.Cout, p.g.kvol, p.g.ntaps, p.cin_pad,
                                                   p.cout_pad, kmajor, mode, p.g.Cin / p.g.G, p.g.Cout / p.g.G,
                                                   p.io16, t);
    return cudaGetLastError();
}

// The staged operand's 16-bit kind (0: fp32 planes).
static int op16(const convt3d_plan_s &p) { return p.bf16 ? (p.half ? kF16 : kBF16) : kF32; }

cudaError_t launch_stage_input(const convt3d_plan_s &p, const float *x, float *hi, float *lo, int n0, int n1,
                               cudaStream_t s) {
    // samples [n0, n1): the kernels see the batch from sample n0 on (x and the planes offset by
    // whole samples; element offsets in units of each array's element)
    const int64_t S = (int64_t)p.g.Din * p.g.Hin * p.g.Win;
    const int nn = n1 - n0;
    if (nn <= 0) return cudaSuccess;
    const int64_t xoff = (int64_t)n0 * p.g.Cin * S * (p.io16 ? 2 : 4);                 // bytes
    const int64_t poff = (int64_t)n0 * S * p.cin_pad * (op16(p) ? 2 : 4);              // bytes
    const float *xn = reinterpret_cast<const float *>(reinterpret_cast<const char *>(x) + xoff);
    float *hn = reinterpret_cast<float *>(reinterpret_cast<char *>(hi) + poff);
    float *ln = lo ? reinterpret_cast<float *>(reinterpret_cast<char *>(lo) + poff) : nullptr;
    if (p.cl) {
        const int64_t rows = S * nn;
        dim3 grid((unsigned)((rows + 7) / 8), (unsigned)(p.cin_pad / 32));
        stage_input_cl_kernel<<<grid, dim3(32, 8), 0, s>>>(xn, hn, ln, p.g.Cin, p.cin_pad, rows, op16(p), p.io16);
        return cudaGetLastError();
    }
    dim3 grid((unsigned)((S + 31) / 32), (unsigned)(p.cin_pad / 32), (unsigned)nn);
    dim3 block(32, 8);
    stage_input_kernel<<<grid, block, 0, s>>>(xn, hn, ln, p.g.Cin, p.cin_pad, S, op16(p), p.io16);
    return cudaGetLastError();
}

}  // namespace convt3d
