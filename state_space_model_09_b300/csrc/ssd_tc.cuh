// ssd_tc.cuh -- the two contractions of the chunked SSD algorithm on the
// 5th-generation tensor cores (tcgen05), bf16 operands staged by TMA into
// 128-byte-swizzled shared memory, float32 accumulators in tensor memory.
//
//   chunk_state_tc : S_c = B_c^T diag(w) x_c          (Mamba-2 page, "SSD算法",
//                    w_j = exp(cs_last - cs_j)         the green step)
//   chunk_scan_tc  : y = (L o C B^T) x                 (orange: diagonal block)
//                      + diag(exp(cs)) C Hin           (blue: true initial state)
//                      + D x                           (skip term, in the epilogue)
//
// Both kernels are written for N (state size) = 128, i.e. one M = 128 tile of
// the state, and for the chunk lengths / head dims the launcher admits:
//   chunk_state_tc: Q in {128, 256}, P in {64, 128}
//   chunk_scan_tc : (Q, P) in {(256, 64), (128, 64), (128, 128)}
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

// ============================================================================
// chunk_state_tc
//   grid (H, nc, batch), 128 threads (4 warps).
//   smem: Bt = N/64 tiles [Q rows j][64 n]  -- A operand (B^T), MN-major
//         Xt = P/64 tiles [Q rows j][64 p]  -- B operand (x, scaled), MN-major
//   D (TMEM, 128 lanes = n, P columns) = Bt^T * Xt over K = Q tokens.
// ============================================================================
template <int Q, int P>
struct ChunkStateSmem {
  static constexpr int kB = kTcN * Q * 2;
  static constexpr int kX = P * Q * 2;
  static constexpr int kW = Q * 4;
  static constexpr int kBytes = kB + kX + kW + 64 + 1024;  // + barriers + alignment slack
};

template <int Q, int P>
__global__ void __launch_bounds__(128, 1)
    chunk_state_tc(const __grid_constant__ CUtensorMap mapB, const __grid_constant__ CUtensorMap mapX,
                   const float *__restrict__ cs, float *__restrict__ S, int H, int GB, int nc) {
  using L = ChunkStateSmem<Q, P>;
  constexpr int N = kTcN;
  constexpr uint32_t kCols = P;  // 64 or 128: a power of two >= 32
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *Bt = smem;
  uint8_t *Xt = Bt + L::kB;
  float *w = reinterpret_cast<float *>(Xt + L::kX);
  uint64_t *bars = reinterpret_cast<uint64_t *>(w + Q);  // [0] tma, [1] mma
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);

  const int h = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gb = h / (H / GB);

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&mapB);
    prefetch_tensormap(&mapX);
  }
  if (warp == 0) tmem_alloc(tslot, kCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;

  if (tid == 0) {
    mbar_arrive_expect_tx(&bars[0], L::kB + L::kX);
#pragma unroll
    for (int s = 0; s < N / 64; ++s) tma_load_4d(Bt + s * Q * 128, &mapB, &bars[0], 64 * s, gb, c * Q, b);
#pragma unroll
    for (int s = 0; s < P / 64; ++s) tma_load_4d(Xt + s * Q * 128, &mapX, &bars[0], 64 * s, h, c * Q, b);
  }
  const float *csc = cs + ((static_cast<int64_t>(b) * H + h) * nc + c) * Q;
  const float cl = csc[Q - 1];
  for (int j = tid; j < Q; j += 128) w[j] = __expf(cl - csc[j]);
  __syncthreads();

  bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[0], 0, abort_flag));
  if (ok) {
    // scale row j of x by w_j (a row keeps its 16-byte chunks under the swizzle)
    uint4 *xv = reinterpret_cast<uint4 *>(Xt);
    for (int idx = tid; idx < (P / 64) * Q * 8; idx += 128) xv[idx] = scale_bf16x8(xv[idx], w[(idx >> 3) % Q]);
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (tid == 0 && !*abort_flag) {
    tc_fence_after_sync();
    constexpr uint32_t idesc = idesc_bf16(128, P, true, true);
    const uint32_t bt = smem_u32(Bt), xt = smem_u32(Xt);
#pragma unroll
    for (int k = 0; k < Q / 16; ++k) {
      const uint64_t ad = sdesc_sw128(bt + k * 2048, Q * 128, 1024);
      const uint64_t bd = sdesc_sw128(xt + k * 2048, Q * 128, 1024);
      mma_bf16(tmem, ad, bd, idesc, k > 0 ? 1u : 0u);
    }
    mma_commit(&bars[1]);
  }
  __syncthreads();
  ok = !*abort_flag;
  if (ok) ok = mbar_wait(&bars[1], 0, abort_flag);
  ok = __all_sync(0xffffffffu, ok);
  tc_fence_after_sync();
  if (ok) {
    const int n = 32 * warp + lane;
    float *dst = S + (((static_cast<int64_t>(b) * nc + c) * H + h) * N + n) * P;
#pragma unroll
    for (int cc = 0; cc < P; cc += 16) {
      float v[16];
      tmem_ld16(tmem + (static_cast<uint32_t>(32 * warp) << 16) + cc, v);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 16; e += 4)
        *reinterpret_cast<float4 *>(dst + cc + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kCols);
}

// ============================================================================
// chunk_scan_tc
//   grid (H, nc, batch), 256 threads (8 warps; warps w and w + 4 share TMEM
//   lane quarter w % 4 and split the columns).
//   The chunk's Q rows form MT = Q/128 row tiles of M = 128.  Row tile mt
//   needs the causal columns j < 128 (mt + 1) of S = C B^T.
//   smem: Ct  = N/64 tiles [Q rows i][64 n]   (A of C B^T, then of C' Hin)
//         Bt  = N/64 tiles [Q rows j][64 n]   (B of C B^T)  -- reused as A2
//         A2  = per row tile, 2 (mt+1) k-blocks [128 rows][64 j] of bf16 L o S
//         Xt  = P/64 tiles [Q rows j][64 p]   (B of (L o S) x, MN-major)
//         Ht  = P/64 tiles [N rows n][64 p]   (B of C' Hin, MN-major)
//   TMEM: S tiles at columns 128 mt (mt+1) / 2 (width 128 (mt + 1)), then the
//         Y accumulators (P columns per row tile).
// ============================================================================
template <int Q, int P>
struct ChunkScanSmem {
  static constexpr int MT = Q / 128;
  static constexpr int kC = kTcN * Q * 2;
  static constexpr int kBt = kTcN * Q * 2;
  static constexpr int kA2 = 128 * 128 * 2 * (MT * (MT + 1) / 2);
  static constexpr int kU = kBt > kA2 ? kBt : kA2;  // Bt / A2 union
  static constexpr int kX = P * Q * 2;
  static constexpr int kH = P * kTcN * 2;
  static constexpr int kF = Q * 4 * 2;  // cs * log2(e), exp(cs)
  static constexpr int kBytes = kC + kU + kX + kH + kF + 64 + 1024;
  static constexpr int kSCols = 128 * MT * (MT + 1) / 2;
  static constexpr int kCols = kSCols + MT * P;
  static constexpr uint32_t kAlloc = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128
                                   : kCols <= 256 ? 256 : 512;
  static_assert(kCols <= 512, "TMEM columns exceeded");
};

template <int Q, int P>
__global__ void __launch_bounds__(256, 1)
    chunk_scan_tc(const __grid_constant__ CUtensorMap mapC, const __grid_constant__ CUtensorMap mapB,
                  const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapH,
                  const float *__restrict__ cs, const float *__restrict__ D,
                  __nv_bfloat16 *__restrict__ y, int64_t T, int H, int GB, int GC, int nc) {
  using L = ChunkScanSmem<Q, P>;
  constexpr int N = kTcN, MT = L::MT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *Ct = smem;
  uint8_t *Bt = Ct + L::kC;  // also A2
  uint8_t *Xt = Bt + L::kU;
  uint8_t *Ht = Xt + L::kX;
  float *csq = reinterpret_cast<float *>(Ht + L::kH);  // cs * log2(e)
  float *eq = csq + Q;                                 // exp(cs)
  uint64_t *bars = reinterpret_cast<uint64_t *>(eq + Q);  // [0] tma, [1] mma1, [2] mma2
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 3);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);

  const int h = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int gb = h / (H / GB), gc = h / (H / GC);

  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    mbar_init(&bars[2], 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&mapC);
    prefetch_tensormap(&mapB);
    prefetch_tensormap(&mapX);
    prefetch_tensormap(&mapH);
  }
  if (warp == 0) tmem_alloc(tslot, L::kAlloc);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;

  if (tid == 0) {
    mbar_arrive_expect_tx(&bars[0], L::kC + L::kBt + L::kX + L::kH);
#pragma unroll
    for (int s = 0; s < N / 64; ++s) {
      tma_load_4d(Ct + s * Q * 128, &mapC, &bars[0], 64 * s, gc, c * Q, b);
      tma_load_4d(Bt + s * Q * 128, &mapB, &bars[0], 64 * s, gb, c * Q, b);
    }
#pragma unroll
    for (int s = 0; s < P / 64; ++s) {
      tma_load_4d(Xt + s * Q * 128, &mapX, &bars[0], 64 * s, h, c * Q, b);
      tma_load_3d(Ht + s * N * 128, &mapH, &bars[0], 64 * s, 0, (b * nc + c) * H + h);
    }
  }
  {
    const float *csc = cs + ((static_cast<int64_t>(b) * H + h) * nc + c) * Q;
    for (int i = tid; i < Q; i += 256) {
      const float v = csc[i] * 1.4426950408889634f;
      csq[i] = v;
      eq[i] = ex2_approx(v);
    }
  }
  __syncthreads();

  // ---- MMA1: S_mt = C[rows of mt] * B[0 : 128 (mt+1)]^T, K = N --------------
  bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[0], 0, abort_flag));
  __syncthreads();
  if (tid == 0 && !*abort_flag) {
    tc_fence_after_sync();
    const uint32_t ct = smem_u32(Ct), bt = smem_u32(Bt);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const uint32_t idesc = idesc_bf16(128, 128 * (mt + 1), false, false);
      const uint32_t dcol = 128 * mt * (mt + 1) / 2;
#pragma unroll
      for (int ks = 0; ks < N / 16; ++ks) {
        const uint32_t koff = (ks >> 2) * Q * 128 + (ks & 3) * 32;
        const uint64_t ad = sdesc_sw128(ct + koff + mt * 128 * 128, 16, 1024);
        const uint64_t bd = sdesc_sw128(bt + koff, 16, 1024);
        mma_bf16(tmem + dcol, ad, bd, idesc, ks > 0 ? 1u : 0u);
      }
    }
    mma_commit(&bars[1]);
  }
  ok = !*abort_flag;
  if (ok) ok = mbar_wait(&bars[1], 0, abort_flag);
  ok = __all_sync(0xffffffffu, ok);
  tc_fence_after_sync();

  // ---- L o S -> bf16 A2 (into the B tile's space); C rows scaled by exp(cs) ----
  if (ok) {
    const int r = 32 * quarter + lane;  // row inside the row tile = TMEM lane
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int i = 128 * mt + r;
      const float ci = csq[i];
      const int ncol = 128 * (mt + 1);
      const int cbeg = half * (ncol / 2), cend = cbeg + ncol / 2;
      uint8_t *a2 = Bt + 128 * 128 * 2 * (mt * (mt + 1) / 2);
      const uint32_t scol = 128 * mt * (mt + 1) / 2;
      for (int cc = cbeg; cc < cend; cc += 16) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * quarter) << 16) + scol + cc, v);
        tmem_ld_wait();
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const int j = cc + e;
          const float l0 = j <= i ? ex2_approx(ci - csq[j]) : 0.f;
          const float l1 = j + 1 <= i ? ex2_approx(ci - csq[j + 1]) : 0.f;
          pk[e >> 1] = pack_bf16x2(v[e] * l0, v[e + 1] * l1);
        }
        uint8_t *blk = a2 + (cc >> 6) * (128 * 128);
        const int col = cc & 63;
        *reinterpret_cast<uint4 *>(blk + sw128_offset(r, col)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4 *>(blk + sw128_offset(r, col + 8)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
    }
    uint4 *cv = reinterpret_cast<uint4 *>(Ct);
    for (int idx = tid; idx < (N / 64) * Q * 8; idx += 256) cv[idx] = scale_bf16x8(cv[idx], eq[(idx >> 3) % Q]);
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();

  // ---- MMA2 + MMA3: Y_mt = A2_mt * x[0 : 128 (mt+1)] + C'_mt * Hin ------------
  if (tid == 0 && !*abort_flag) {
    tc_fence_after_sync();
    const uint32_t ct = smem_u32(Ct), a2b = smem_u32(Bt), xt = smem_u32(Xt), ht = smem_u32(Ht);
    constexpr uint32_t idesc = idesc_bf16(128, P, false, true);
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const uint32_t dcol = L::kSCols + mt * P;
      const uint32_t a2 = a2b + 128 * 128 * 2 * (mt * (mt + 1) / 2);
#pragma unroll
      for (int ks = 0; ks < 8 * (mt + 1); ++ks) {
        const uint64_t ad = sdesc_sw128(a2 + (ks >> 2) * (128 * 128) + (ks & 3) * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(xt + ks * 2048, Q * 128, 1024);
        mma_bf16(tmem + dcol, ad, bd, idesc, ks > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int ks = 0; ks < N / 16; ++ks) {
        const uint64_t ad =
            sdesc_sw128(ct + (ks >> 2) * Q * 128 + (ks & 3) * 32 + mt * 128 * 128, 16, 1024);
        const uint64_t bd = sdesc_sw128(ht + ks * 2048, N * 128, 1024);
        mma_bf16(tmem + dcol, ad, bd, idesc, 1u);
      }
    }
    mma_commit(&bars[2]);
  }
  ok = !*abort_flag;
  if (ok) ok = mbar_wait(&bars[2], 0, abort_flag);
  ok = __all_sync(0xffffffffu, ok);
  tc_fence_after_sync();

  // ---- epilogue: y = Y + D x, rounded to bf16 ---------------------------------
  if (ok) {
    const float Dh = D ? D[h] : 0.f;
    const int r = 32 * quarter + lane;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      const int i = 128 * mt + r;
      const int64_t t = static_cast<int64_t>(c) * Q + i;
      const bool store = t < T;
      const uint32_t dcol = L::kSCols + mt * P;
      __nv_bfloat16 *yrow = y + ((static_cast<int64_t>(b) * T + t) * H + h) * P;
#pragma unroll
      for (int cc = half * (P / 2); cc < (half + 1) * (P / 2); cc += 16) {
        float v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * quarter) << 16) + dcol + cc, v);
        tmem_ld_wait();
        const uint8_t *xs = Xt + (cc >> 6) * Q * 128;
        const uint4 x0 = *reinterpret_cast<const uint4 *>(xs + sw128_offset(i, cc & 63));
        const uint4 x1 = *reinterpret_cast<const uint4 *>(xs + sw128_offset(i, (cc & 63) + 8));
        const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 xf = unpack_bf16x2(xw[e]);
          pk[e] = pack_bf16x2(fmaf(Dh, xf.x, v[2 * e]), fmaf(Dh, xf.y, v[2 * e + 1]));
        }
        if (store) {
          *reinterpret_cast<uint4 *>(yrow + cc) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4 *>(yrow + cc + 8) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, L::kAlloc);
}

}  // namespace ssd
