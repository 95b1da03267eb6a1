// ssd_cp.cuh -- context parallelism over the sequence (Mamba-2 page, section
// "序列并行的两种形式", context parallelism: each GPU computes its segment's
// outputs and final state, and the states are passed from GPU to GPU).
//
// A rank holding tokens [t_r, t_r+1) of every sequence runs the layer on its
// segment from a zero state (rank 0 from h0): y_local and F_r, the segment's
// final state.  With Lambda_r the segment's total decay (the product of its
// tokens' exp(dt A)), the true state entering segment r is
//   H_in(0) = 0 (rank 0 already started from h0),
//   H_in(r + 1) = Lambda_r H_in(r) + F_r                   (the scan over ranks),
// and, with a_t the running log2 decay from the segment's start to token t
// (inclusive, the same convention as inside a chunk),
//   y_t = y_local_t + 2^(a_t) C_t^T H_in(r),   h_final = Lambda_r H_in(r) + F_r
// -- the chunk algorithm's state-passing and output-from-initial-state steps
// applied once more, one level up, with segments in place of chunks.
//
// Kernels: row_cumsum_kernel (a_t from the per-token decays dt_decay_kernel
// writes; Lambda = 2^(a_last)), cp_combine_kernel (H_in(r) and h_final,
// elementwise over the states), cp_correct_tc (the C H_in product on the
// tensor cores, bf16 C with N = 128 and P in {64, 128}) or cp_correct_simt
// (every other shape, float32 CUDA cores).
#pragma once

#include "ssd_tc.cuh"

namespace ssd {

// ----------------------------------------------------------------------------
// In place: a[row, t] = sum_{k <= t} a[row, k] over rows of length T (one block
// per row, 1024 tokens per pass); decay[row] = 2^(a[row, T - 1]) when given.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) row_cumsum_kernel(float *__restrict__ a, int64_t T,
                                                         float *__restrict__ decay) {
  __shared__ float wsum[8];
  float *r = a + static_cast<int64_t>(blockIdx.x) * T;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float carry = 0.f;
  for (int64_t base = 0; base < T; base += 1024) {
    const int64_t t0 = base + 4 * tid;
    float v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = t0 + k < T ? r[t0 + k] : 0.f;
#pragma unroll
    for (int k = 1; k < 4; ++k) v[k] += v[k - 1];
    const float tot = v[3];
    float incl = tot;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    float before = 0.f, block = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      before += w < warp ? wsum[w] : 0.f;
      block += wsum[w];
    }
    __syncthreads();  // wsum is rewritten by the next pass
    const float off = carry + before + incl - tot;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (t0 + k < T) r[t0 + k] = v[k] + off;
    carry += block;
  }
  if (decay && tid == 0) decay[blockIdx.x] = ex2_approx(carry);
}

// ----------------------------------------------------------------------------
// H_in(rank) from the gathered segment decays and final states, and this
// rank's true final state:
//   H = 0; for r' < rank: H = Lambda_r' H + F_r';   h_in = H;
//   h_final = Lambda_rank H + F_rank
// decays [nranks, BH], finals [nranks, BH, NP]; one float4 per thread.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cp_combine_kernel(const float *__restrict__ decays,
                                                         const float *__restrict__ finals,
                                                         int rank, int64_t BH, int NP,
                                                         float *__restrict__ h_in,
                                                         float *__restrict__ h_final) {
  const int64_t i4 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total4 = BH * NP / 4;
  if (i4 >= total4) return;
  const int64_t bh = i4 * 4 / NP;
  float4 H = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r = 0; r < rank; ++r) {
    const float L = decays[static_cast<int64_t>(r) * BH + bh];
    const float4 F = reinterpret_cast<const float4 *>(finals + static_cast<int64_t>(r) * BH * NP)[i4];
    H = make_float4(fmaf(L, H.x, F.x), fmaf(L, H.y, F.y), fmaf(L, H.z, F.z), fmaf(L, H.w, F.w));
  }
  if (h_in) reinterpret_cast<float4 *>(h_in)[i4] = H;
  if (h_final) {
    const float L = decays[static_cast<int64_t>(rank) * BH + bh];
    const float4 F =
        reinterpret_cast<const float4 *>(finals + static_cast<int64_t>(rank) * BH * NP)[i4];
    reinterpret_cast<float4 *>(h_final)[i4] =
        make_float4(fmaf(L, H.x, F.x), fmaf(L, H.y, F.y), fmaf(L, H.z, F.z), fmaf(L, H.w, F.w));
  }
}

// ----------------------------------------------------------------------------
// y[b, t, h, :] += 2^(a[b, h, t]) (C[b, t, g(h), :] H_in[b, h]) on the tensor
// cores: one CTA per (batch row, 128-token tile, run of heads sharing a C
// group).  The C tile (128 tokens x 128 state columns, bf16, TMA) is the
// K-major A operand of every head's MMA; each head's H_in (float32 in
// global memory) is rounded to bf16 into a 128-byte-swizzled tile, the
// MN-major B operand; D (128 x P, float32) sits in tensor memory; thread t of
// the four warps reads token t's row and updates y.  Rows past T are not
// written.  Every wait is bounded in time.
// ----------------------------------------------------------------------------
template <int P>
struct CpTc {
  static constexpr int N = kTcN, TQ = 128;
  static constexpr int kBytes = 1024 + 2 * TQ * 128 + (P / 64) * N * 128 + 64;
};

template <int P>
__global__ void __launch_bounds__(128, 1)
    cp_correct_tc(const __grid_constant__ CUtensorMap mapC, const float *__restrict__ h_in,
                  const float *__restrict__ a, __nv_bfloat16 *__restrict__ y, int64_t T, int H,
                  int GC, int hpc) {
  constexpr int N = CpTc<P>::N, TQ = CpTc<P>::TQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *Cs = smem;                  // two 64-column atoms, each [TQ rows][128 B]
  uint8_t *Hs = Cs + 2 * TQ * 128;     // P / 64 atoms, each [N rows][128 B]
  uint64_t *bars = reinterpret_cast<uint64_t *>(Hs + (P / 64) * N * 128);  // C in, MMA done
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
  const int tid = threadIdx.x, warp = tid >> 5;
  const int b = blockIdx.z;
  const int h_begin = blockIdx.y * hpc, h_end = min(H, h_begin + hpc);
  const int g = h_begin / (H / GC);  // hpc divides H / GC: one group per CTA
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * TQ;

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, P);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;
  if (tid == 0) {
    prefetch_tensormap(&mapC);
    mbar_arrive_expect_tx(&bars[0], 2 * TQ * 128);
    tma_load_4d(Cs, &mapC, &bars[0], 0, g, static_cast<int>(t0), b);
    tma_load_4d(Cs + TQ * 128, &mapC, &bars[0], 64, g, static_cast<int>(t0), b);
  }
  const uint32_t cs = smem_u32(Cs), hs = smem_u32(Hs);
  constexpr uint32_t idesc = idesc_bf16(128, P, false, true);
  const int64_t t = t0 + tid;
  const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
  bool ok = true;
  for (int h = h_begin; h < h_end && ok; ++h) {
    const int it = h - h_begin;
    // H_in of (b, h) -> bf16 operand tile: row n, column p in atom p / 64
    const float *src = h_in + (static_cast<int64_t>(b) * H + h) * N * P;
    for (int e = tid; e < N * P / 8; e += 128) {
      const int n = e / (P / 8), c8 = e % (P / 8);
      const float4 v0 = *reinterpret_cast<const float4 *>(src + n * P + 8 * c8);
      const float4 v1 = *reinterpret_cast<const float4 *>(src + n * P + 8 * c8 + 4);
      *reinterpret_cast<uint4 *>(Hs + (c8 >> 3) * N * 128 + sw128_offset(n, 8 * (c8 & 7))) =
          make_uint4(pack_bf16x2(v0.x, v0.y), pack_bf16x2(v0.z, v0.w), pack_bf16x2(v1.x, v1.y),
                     pack_bf16x2(v1.z, v1.w));
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      const bool in = it > 0 || mbar_wait(&bars[0], 0, abort_flag);
      if (in) {
        tc_fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks) {
          const uint32_t koff = (ks >> 2) * TQ * 128 + (ks & 3) * 32;
          mma_bf16(tmem, sdesc_sw128(cs + koff, 16, 1024), sdesc_sw128(hs + ks * 2048, N * 128, 1024),
                   idesc, ks > 0 ? 1u : 0u);
        }
        mma_commit(&bars[1]);
      }
    }
    const bool w = mbar_wait(&bars[1], it & 1, abort_flag);
    ok = __syncthreads_and(w && !*abort_flag) != 0;
    if (!ok) break;
    tc_fence_after_sync();
    float acc[P];
#pragma unroll
    for (int c = 0; c < P / 32; ++c) {
      float v[32];
      tmem_ld32(tmem + lane_base + 32 * c, v);
#pragma unroll
      for (int e = 0; e < 32; ++e) acc[32 * c + e] = v[e];
    }
    if (t < T) {
      const float f = ex2_approx(a[(static_cast<int64_t>(b) * H + h) * T + t]);
      uint4 *row = reinterpret_cast<uint4 *>(y + ((static_cast<int64_t>(b) * T + t) * H + h) * P);
#pragma unroll
      for (int q = 0; q < P / 8; ++q) {
        uint4 u = row[q];
        uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 yv = unpack_bf16x2(wv[k]);
          wv[k] = pack_bf16x2(fmaf(f, acc[8 * q + 2 * k], yv.x), fmaf(f, acc[8 * q + 2 * k + 1], yv.y));
        }
        row[q] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
    }
    tc_fence_before_sync();
    __syncthreads();  // the next head's MMA overwrites the accumulator and reads a new tile
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, P);
}

// ----------------------------------------------------------------------------
// The same update in float32 on the CUDA cores, for any shape and io dtype:
// block (32-token tile, 64-column slice of P, b H + h); shared memory holds
// the C tile [32][N] and the H_in slice [N][PS] as float32; thread (token
// ty, columns 8 tx .. 8 tx + 7 of the slice) sums over n.
// ----------------------------------------------------------------------------
template <typename IO>
__global__ void __launch_bounds__(256) cp_correct_simt(const IO *__restrict__ C,
                                                       const float *__restrict__ h_in,
                                                       const float *__restrict__ a,
                                                       IO *__restrict__ y, int64_t T, int H,
                                                       int GC, int N, int P, int PS) {
  extern __shared__ float fs[];
  float *Ct = fs;             // [32][N]
  float *Hsl = fs + 32 * N;   // [N][PS]
  const int64_t bh = blockIdx.z;
  const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
  const int g = h / (H / GC);
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * 32;
  const int p0 = blockIdx.y * PS;
  const int tid = threadIdx.x, ty = tid >> 3, tx = tid & 7;
  for (int e = tid; e < 32 * N; e += 256) {
    const int r = e / N, n = e % N;
    Ct[e] = t0 + r < T ? to_f32(C[((static_cast<int64_t>(b) * T + t0 + r) * GC + g) * N + n]) : 0.f;
  }
  const float *src = h_in + bh * N * P + p0;
  for (int e = tid; e < N * PS; e += 256) Hsl[e] = src[(e / PS) * P + e % PS];
  __syncthreads();
  const int64_t t = t0 + ty;
  const int ncol = PS / 8;  // columns per thread: PS / 8 (PS in {16, 32, 64})
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int n = 0; n < N; ++n) {
    const float cv = Ct[ty * N + n];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < ncol) acc[j] = fmaf(cv, Hsl[n * PS + tx * ncol + j], acc[j]);
  }
  if (t >= T) return;
  const float f = exp2f(a[bh * T + t]);
  IO *row = y + ((static_cast<int64_t>(b) * T + t) * H + h) * P + p0 + tx * ncol;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < ncol) row[j] = from_f32<IO>(fmaf(f, acc[j], to_f32(row[j])));
}

}  // namespace ssd
