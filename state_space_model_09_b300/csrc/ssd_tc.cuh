// ssd_tc.cuh -- small helpers shared by the tensor-core kernels.
#pragma once

#include "ssd_device.cuh"

namespace ssd {

constexpr int kTcN = 128;  // state size handled by the tensor-core kernels

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
