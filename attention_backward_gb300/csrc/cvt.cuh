// Conversions between f32 and the 16-bit input types, and the hardware exp2.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <cstring>

namespace ab {

// Two f32 values rounded (nearest-even) to fp16/bf16 and packed low-first.
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  uint32_t r;
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    memcpy(&r, &h, 4);
  } else {
    __half2 h = __floats2half2_rn(a, b);
    memcpy(&r, &h, 4);
  }
  return r;
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    __nv_bfloat162 h;
    memcpy(&h, &w, 4);
    return __bfloat1622float2(h);
  } else {
    __half2 h;
    memcpy(&h, &w, 4);
    return __half22float2(h);
  }
}

// The rounding residuals of a pair packed by pack2 (``hi``), rounded and packed
// the same way: a + b's 16-bit hi pair plus this lo pair carries about 16
// significant bits of each value.
template <bool BF16>
__device__ __forceinline__ uint32_t lo_pair(float a, float b, uint32_t hi) {
  const float2 h = unpack2<BF16>(hi);
  return pack2<BF16>(a - h.x, b - h.y);
}

// 2^x on the multi-function unit (MUFU.EX2), flush-to-zero.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace ab
