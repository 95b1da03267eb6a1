// ssd_state.cuh -- chunk states and state passing in one tensor-core kernel.
//
// One CTA walks the chunks of one (batch b, head h, 64-column slice of P) in
// order.  For chunk c, with cs the in-chunk inclusive running sum of
// softplus(dt) * A_h (computed here from dt):
//   S_c   = B_c^T diag(w) x_c,     w_j = exp(cs_last - cs_j)         (green step)
//   Hin_c = state entering chunk c                                   (stored, bf16)
//   state = exp(cs_last) * state + S_c                               (yellow step)
// (Mamba-2 page, section "SSD算法": the chunk-final states by batched matmul and
// the scan over chunks with the chunk decays; the pages note the scan is
// short -- here it runs in registers while the next chunk streams in.)  The
// running state starts at h0 (or zero) and its last value is h_final.
//
// S_c is one tcgen05 MMA chain: M = 128 state rows (TMEM lanes), N = 64
// columns, K = Q tokens, both operands MN-major in 128B-swizzled smem written
// by TMA.  256 threads: thread t owns state row t % 128 and columns
// 32 (t / 128) .. +31, kept in registers across chunks.  The next chunk's
// cumsum runs while the current chunk's MMA is in flight; two CTAs share an SM
// so one's tile loads overlap the other's work.
#pragma once

#include "ssd_device.cuh"
#include "ssd_tc.cuh"

namespace ssd {

template <int Q>
struct StatePass {
  static constexpr int N = kTcN;
  static constexpr int PS = 64;  // P columns per CTA
  static constexpr int kB = N * Q * 2;
  static constexpr int kX = PS * Q * 2;
  static constexpr int kThreads = 256;
  // tiles + double-buffered (cs, w) + decay[2] + warp sums + barriers
  static constexpr int kBytes = kB + kX + (4 * Q + 2 + 8) * 4 + 4 * 8 + 16 + 1024;
  static_assert(kBytes <= 113 * 1024, "two CTAs per SM");
};

template <int Q>
__global__ void __launch_bounds__(256, 2)
    chunk_state_pass_tc(const __grid_constant__ CUtensorMap mapB,
                        const __grid_constant__ CUtensorMap mapX, const float *__restrict__ dt,
                        const float *__restrict__ A, const float *__restrict__ h0,
                        __nv_bfloat16 *__restrict__ Hin, float *__restrict__ h_final, int64_t T,
                        int H, int GB, int nc, int P, int softplus) {
  using L = StatePass<Q>;
  constexpr int N = L::N, PS = L::PS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *Bt = smem;
  uint8_t *Xt = Bt + L::kB;
  float *csb = reinterpret_cast<float *>(Xt + L::kX);  // [2][Q] running sums
  float *wb = csb + 2 * Q;                              // [2][Q] exp(cs_last - cs_j)
  float *decay_s = wb + 2 * Q;                          // [2]
  float *wsum = decay_s + 2;                            // warp totals
  uint64_t *bars = reinterpret_cast<uint64_t *>(wsum + 8);  // [0] tma, [1] mma
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 4);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);

  const int p0 = blockIdx.x * PS, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gb = h / (H / GB);
  const float Ah = A[h];
  const int n = tid & 127, cbase = 32 * (tid >> 7);  // state row, first column

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&mapB);
    prefetch_tensormap(&mapX);
  }
  if (warp == 0) tmem_alloc(tslot, PS);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16) + cbase;

  auto issue_loads = [&](int c) {
    mbar_arrive_expect_tx(&bars[0], L::kB + L::kX);
#pragma unroll
    for (int s = 0; s < N / 64; ++s) tma_load_4d(Bt + s * Q * 128, &mapB, &bars[0], 64 * s, gb, c * Q, b);
    tma_load_4d(Xt, &mapX, &bars[0], p0, h, c * Q, b);
  };
  auto load_dt = [&](int c) {
    const int64_t t = static_cast<int64_t>(c) * Q + tid;
    return (tid < Q && t < T) ? dt[(static_cast<int64_t>(b) * T + t) * H + h] : 0.f;
  };
  // cumsum of softplus(dt) * A_h over chunk c into buffer c & 1 (one token per thread)
  auto cumsum = [&](int c, float z) {
    float *cs = csb + (c & 1) * Q, *w = wb + (c & 1) * Q;
    const int64_t t = static_cast<int64_t>(c) * Q + tid;
    float v = (tid < Q && t < T) ? (softplus ? softplus_f32(z) : z) * Ah : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    for (int ww = 0; ww < warp; ++ww) v += wsum[ww];
    if (tid < Q) cs[tid] = v;
    __syncthreads();
    const float cl = cs[Q - 1];
    if (tid < Q) w[tid] = __expf(cl - v);
    if (tid == 0) decay_s[c & 1] = __expf(cl);
    // readers of w / decay synchronise later in the loop
  };

  const int64_t srow = ((static_cast<int64_t>(b) * H + h) * N + n) * P + p0 + cbase;
  float st[32];
  if (h0) {
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 v = *reinterpret_cast<const float4 *>(h0 + srow + e);
      st[e] = v.x; st[e + 1] = v.y; st[e + 2] = v.z; st[e + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) st[e] = 0.f;
  }

  if (tid == 0) issue_loads(0);
  cumsum(0, load_dt(0));
  float z_next = nc > 1 ? load_dt(1) : 0.f;
  for (int c = 0; c < nc; ++c) {
    // ---- entering state of this chunk -> Hin (bf16)
    {
      __nv_bfloat16 *dst = Hin + (((static_cast<int64_t>(b) * nc + c) * H + h) * N + n) * P + p0 + cbase;
#pragma unroll
      for (int e = 0; e < 32; e += 8)
        *reinterpret_cast<uint4 *>(dst + e) =
            make_uint4(pack_bf16x2(st[e], st[e + 1]), pack_bf16x2(st[e + 2], st[e + 3]),
                       pack_bf16x2(st[e + 4], st[e + 5]), pack_bf16x2(st[e + 6], st[e + 7]));
    }
    __syncthreads();  // w / decay of chunk c complete
    const float *w = wb + (c & 1) * Q;
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[0], c & 1, abort_flag));
    if (ok) {
      // x row j *= w_j (a row keeps its 16-byte chunks under the swizzle)
      uint4 *xv = reinterpret_cast<uint4 *>(Xt);
#pragma unroll 4
      for (int idx = tid; idx < Q * 8; idx += 256) xv[idx] = scale_bf16x8(xv[idx], w[idx >> 3]);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0 && !*abort_flag) {
      tc_fence_after_sync();
      constexpr uint32_t idesc = idesc_bf16(128, PS, true, true);
      const uint32_t bt = smem_u32(Bt), xt = smem_u32(Xt);
#pragma unroll
      for (int k = 0; k < Q / 16; ++k)
        mma_bf16(tmem, sdesc_sw128(bt + k * 2048, Q * 128, 1024),
                 sdesc_sw128(xt + k * 2048, Q * 128, 1024), idesc, k > 0 ? 1u : 0u);
      mma_commit(&bars[1]);
    }
    // ---- next chunk's cumsum while the MMA runs
    if (c + 1 < nc) {
      cumsum(c + 1, z_next);
      if (c + 2 < nc) z_next = load_dt(c + 2);
    }
    ok = !*abort_flag && mbar_wait(&bars[1], c & 1, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after_sync();
    if (tid == 0 && ok && c + 1 < nc) issue_loads(c + 1);  // the tiles are free again
    if (ok) {
      const float decay = decay_s[c & 1];
      float sv[32];
      tmem_ld32(taddr, sv);
#pragma unroll
      for (int e = 0; e < 32; ++e) st[e] = fmaf(decay, st[e], sv[e]);
    }
    tc_fence_before_sync();
  }
  if (h_final) {
#pragma unroll
    for (int e = 0; e < 32; e += 4)
      *reinterpret_cast<float4 *>(h_final + srow + e) = make_float4(st[e], st[e + 1], st[e + 2], st[e + 3]);
  }
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, PS);
}

}  // namespace ssd
