// Epilogue arithmetic shared by the tensor-core kernels: the base-2
// exponential, packed two-lane fp32 operations and the sigmoid polynomial.
#pragma once

#include <stdint.h>

namespace convt3d {

constexpr float kLog2e = 1.4426950408889634f;

// 2^x with the PTX approximate base-2 exponential (ex2.approx.ftz.f32).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed two-lane fp32 arithmetic (add/mul/fma.rn.f32x2): one instruction on a
// pair of values held as one 64-bit register pair.
__device__ __forceinline__ uint64_t pack2(float a, float b) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ void unpack2(uint64_t v, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}

__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// sigmoid(t) for t in [0, 1] as 1/2 + t * (s0 + s1 t^2 + s2 t^4 + s3 t^6): the
// odd part of sigmoid about 0 fitted by a linear program minimising the largest
// error over 20,001 points of [0, 1] (max error 5.6e-8; 1.2e-7 with the fp32
// Horner evaluation below).
constexpr float kSig0 = 0.24999944865703583f;
constexpr float kSig1 = -0.020825687795877457f;
constexpr float kSig2 = 0.0020543981809169054f;
constexpr float kSig3 = -0.0001696429681032896f;

// Coefficients that evaluate sigmoid(f * e) from e directly:
// 1/2 + e * (s0 f + s1 f^3 e^2 + s2 f^5 e^4 + s3 f^7 e^6), packed as pairs.
__device__ __forceinline__ void sigmoid_coefficients(float f, uint64_t (&A)[4]) {
    const float f2 = f * f;
    const float a0 = kSig0 * f, a1 = kSig1 * f * f2, a2 = kSig2 * f * f2 * f2, a3 = kSig3 * f * f2 * f2 * f2;
    A[0] = pack2(a0, a0);
    A[1] = pack2(a1, a1);
    A[2] = pack2(a2, a2);
    A[3] = pack2(a3, a3);
}

}  // namespace convt3d
