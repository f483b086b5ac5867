// softmax.cuh — arithmetic of the tcgen05 attention kernel's softmax warps: packed fp32 pairs
// (one instruction does the FMA or ADD of two columns) and a three-input max, which halve the
// instructions a row of scores costs.
#pragma once

#include <stdint.h>

namespace pkv {
namespace sm {

// ---- packed fp32 pairs (.b64 = {lo, hi}) --------------------------------------------------------
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// bf16 pair {lo, hi} (round to nearest even) from an fp32 pair
__device__ __forceinline__ uint32_t bf16x2(uint64_t v) {
  float lo, hi;
  unf2(v, lo, hi);
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// fp16 pair {lo, hi} (round to nearest even) from an fp32 pair
__device__ __forceinline__ uint32_t f16x2(uint64_t v) {
  float lo, hi;
  unf2(v, lo, hi);
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace sm
}  // namespace pkv
