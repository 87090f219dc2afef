// Shared device helpers of the denoise-step library (CUDA sources only).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/tt_denoise.h"

namespace tt {

// First device-side error wins; later ones are dropped.
__device__ __forceinline__ void report_error(uint32_t *dev_err, uint32_t code) {
    if (dev_err != nullptr) atomicCAS(dev_err, 0u, code);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

// Low / high bfloat16 halves of a 32-bit word as fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// fp32 -> bf16 bits, round to nearest even (finite inputs; NaN stays NaN).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float x) {
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
    u += 0x7fffu + ((u >> 16) & 1u);
    return u >> 16;
}

// 2^x on the special-function unit (flushes denormal results to zero).  Callers pass
// exponents up to +8 as well: the attention's lazy rescale lets a tile's scores exceed
// the running maximum by up to 2^8 before it moves, so P <= 2^8 (exact enough in bf16,
// and far from overflow in the fp32 sums).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace tt
