// ssd_tc.cuh -- small helpers shared by the tensor-core kernels.
#pragma once

#include "ssd_device.cuh"

namespace ssd {

constexpr int kTcN = 128;  // state size handled by the tensor-core kernels

// The scaled form of the head-pair chunk scan (chunk_scan_hb) and the chunk
// states it reads.  With a_j the in-chunk running log2 decay (a_j <= 0,
// falling to a_last) and a reference r <= 0 per (batch, chunk, head), the
// scan multiplies x_j by 2^(r - a_j), the chunk's entering state by 2^r, and
// row i of the result by 2^(a_i - r).  r = min(0, a_last + kScaledRange) keeps
// every factor within 2^-kScaledRange .. 2^kScaledRange, so no product
// overflows float32 or bfloat16 (sums of |S x| below 2^31) and no factor
// leaves the normal range, provided a_last >= -kScaledRangeMax; chunks that
// decay further are computed head by head.
constexpr float kScaledRange = 96.f;
constexpr float kScaledRangeMax = 2.f * kScaledRange;

__device__ __forceinline__ bool scaled_form_ok(float a_last) { return a_last >= -kScaledRangeMax; }
__device__ __forceinline__ float scaled_form_ref(float a_last) {
  return fminf(0.f, a_last + kScaledRange);
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Multiplies the 8 bf16 values of a 16-byte chunk by s (round to nearest even).
__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, float s) {
  float2 f;
  f = unpack_bf16x2(v.x); v.x = pack_bf16x2(f.x * s, f.y * s);
  f = unpack_bf16x2(v.y); v.y = pack_bf16x2(f.x * s, f.y * s);
  f = unpack_bf16x2(v.z); v.z = pack_bf16x2(f.x * s, f.y * s);
  f = unpack_bf16x2(v.w); v.w = pack_bf16x2(f.x * s, f.y * s);
  return v;
}

}  // namespace ssd
