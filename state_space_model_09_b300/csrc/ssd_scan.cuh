// ssd_scan.cuh -- chunk_scan on tcgen05 tensor cores, looping over the heads
// that share one (B, C) group inside a chunk.
//
// For one (batch b, chunk c) and each head h of a head range, with cs the
// in-chunk inclusive running sum of softplus(dt) * A_h (computed here from dt)
// and Hin the chunk's true initial state:
//   y = (L o C B^T + D_h I) x  +  diag(exp(cs)) C Hin,   L[i,j] = exp(cs_i - cs_j), j <= i
// (Mamba-2 page, section "SSD算法": the orange diagonal block in quadratic form
// and the blue term from the true initial state; the skip term D x rides on
// the diagonal of the masked score matrix).
//
// S = C B^T depends only on the (B, C) group, so it is computed once per group
// into tensor memory and reused by every head of the group.  Per head:
//   MMA3:  Y  = C Hin                       (TMEM accumulator, K = N)
//   mask:  A2 = bf16(L o S + D I)           (TMEM -> registers -> swizzled smem)
//   scale: Y *= exp(cs_i) row by row        (tcgen05.ld / tcgen05.st)
//   MMA2:  Y += A2 x                        (K = causal columns)
//   out:   y = bf16(Y), staged in smem, written by TMA tile stores
// L is never formed in memory.  It is factorised per 32-column band: for a row
// i below band k (reference column r_k = 32k + 31),
//   L[i,j] = exp(cs_i - cs_rk) * exp(cs_rk - cs_j),
// both factors <= 1 because cs does not increase, so only the 32 x 32 blocks on
// the diagonal need an exponential per element.
//
// Row order: a TMEM lane quarter is tied to a warp, and causal masking gives
// the lower rows more work.  With two 128-row tiles (Q = 256) the C tile's
// second half is loaded with its four 32-row blocks in reverse order, so lane
// quarter q holds rows 32q.. of the first tile and rows 224 - 32q.. of the
// second: every quarter then has nine non-zero 32-column bands.
//
// Warp roles: warps 0-15 (512 threads; four per TMEM lane quarter) do the
// cumsum, mask, scaling and output; warp 16 (one elected lane) issues every
// TMA load and MMA.  Every wait is bounded in time.
#pragma once

#include "ssd_device.cuh"
#include "ssd_tc.cuh"

namespace ssd {

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// waits until at most one committed bulk store group of this thread is still
// reading its shared-memory source
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

constexpr int kScanComputeWarps = 16;
constexpr int kScanThreads = 32 * (kScanComputeWarps + 1);
// barrier among the compute threads only (warps 0-15)
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

template <int Q, int P>
struct ScanHL {
  static constexpr int N = kTcN;
  static constexpr int MT = Q / 128;
  static constexpr int kC = N * Q * 2;
  static constexpr int kB = N * Q * 2;
  static constexpr int kA2 = 128 * 128 * 2 * (MT * (MT + 1) / 2);
  static constexpr int kU = kB > kA2 ? kB : kA2;
  static constexpr int kX = P * Q * 2;
  static constexpr int kH = P * N * 2;
  static constexpr int kStageTile = P * 128 * 2;  // y staging of one 128-row tile
  static constexpr int kMaxHeads = 12;            // most heads per CTA
  // cs*log2e, exp(cs), band factors, warp sums, D, softplus(dt)*A [Q][kMaxHeads]
  static constexpr int kFloats = 3 * Q + 32 + kMaxHeads + Q * kMaxHeads;
  static constexpr int kBars = 12;
  static constexpr int kBytes = kC + kU + kX + kH + kFloats * 4 + kBars * 8 + 16 + 1024;
  static constexpr int kSCols = 128 * MT * (MT + 1) / 2;
  static constexpr int kCols = kSCols + MT * P;
  static constexpr uint32_t kAlloc = kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  static_assert(kCols <= 512, "TMEM columns exceeded");
  static_assert(kBytes <= 227 * 1024, "shared memory exceeded");
  // tile 0 is staged in the first A2 block, tile 1 in the second
  static_assert(kStageTile <= 128 * 128 * 2, "y staging must fit an A2 block");
  static constexpr int kThreads = kScanThreads;
};

enum : int {
  kBarCB = 0, kBarX, kBarH, kBarS, kBarM3, kBarM2a, kBarM2b, kBarA2a, kBarA2b, kBarYFree, kBarStore
};

// Chunk row held by smem/TMEM row s of the C tile (see "Row order" above).
template <int MT>
__device__ __forceinline__ int scan_row(int s) {
  if (MT == 1 || s < 128) return s;
  return 128 + 32 * (3 - ((s - 128) >> 5)) + (s & 31);
}

// Masked scores of one 32-column band kb of row tile mt for the calling warp's
// 32 rows: A2 = bf16(L o S + D I) written into the swizzled A2 block.  Kept out
// of line: one copy serves every band, which keeps the kernel's code small.
template <int MT>
__device__ __noinline__ void scan_mask_band(uint8_t *Bt, uint32_t tlane, const float *cs2,
                                            const float *cf, int q, int lane, int mt, int kb,
                                            float Dh) {
  const int r = 32 * q + lane;               // TMEM lane / A2 row
  const int i = scan_row<MT>(128 * mt + r);  // chunk row
  const int diag_band = i >> 5;              // uniform over the warp
  uint8_t *blk = Bt + 128 * 128 * 2 * (mt * (mt + 1) / 2) + (kb >> 1) * (128 * 128);
  const int col0 = (kb & 1) * 32;
  uint32_t pk[16];
  if (kb > diag_band) {
#pragma unroll
    for (int e = 0; e < 16; ++e) pk[e] = 0u;
  } else {
    float v[32];
    tmem_ld32(tlane + 128 * mt * (mt + 1) / 2 + 32 * kb, v);
    const float ci = cs2[i];
    const float4 *c4 = reinterpret_cast<const float4 *>((kb < diag_band ? cf : cs2) + 32 * kb);
    if (kb < diag_band) {
      const float rf = ex2_approx(ci - cs2[32 * kb + 31]);
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 f = c4[e >> 2];
        pk[e >> 1] = pack_bf16x2(v[e] * rf * f.x, v[e + 1] * rf * f.y);
        pk[(e >> 1) + 1] = pack_bf16x2(v[e + 2] * rf * f.z, v[e + 3] * rf * f.w);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 f = c4[e >> 2];
        const int j = 32 * kb + e;
        float l0 = j <= i ? v[e] * ex2_approx(ci - f.x) : 0.f;
        float l1 = j + 1 <= i ? v[e + 1] * ex2_approx(ci - f.y) : 0.f;
        float l2 = j + 2 <= i ? v[e + 2] * ex2_approx(ci - f.z) : 0.f;
        float l3 = j + 3 <= i ? v[e + 3] * ex2_approx(ci - f.w) : 0.f;
        if (j == i) l0 += Dh;
        if (j + 1 == i) l1 += Dh;
        if (j + 2 == i) l2 += Dh;
        if (j + 3 == i) l3 += Dh;
        pk[e >> 1] = pack_bf16x2(l0, l1);
        pk[(e >> 1) + 1] = pack_bf16x2(l2, l3);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e)
    *reinterpret_cast<uint4 *>(blk + sw128_offset(r, col0 + 8 * e)) =
        make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
}

template <int Q, int P>
__global__ void __launch_bounds__(kScanThreads, 1)
    chunk_scan_hl(const __grid_constant__ CUtensorMap mapC32, const __grid_constant__ CUtensorMap mapB,
                  const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapH,
                  const __grid_constant__ CUtensorMap mapY128, const float *__restrict__ dt,
                  const float *__restrict__ A, const float *__restrict__ D, int64_t T, int H,
                  int GB, int GC, int nc, int heads_per_cta, int softplus) {
  using L = ScanHL<Q, P>;
  constexpr int N = L::N, MT = L::MT, KMAX = L::kMaxHeads;
  constexpr int CW = kScanComputeWarps;
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *Ct = smem;
  uint8_t *Bt = Ct + L::kC;  // B tile, then the A2 blocks (and the y staging)
  uint8_t *Xt = Bt + L::kU;
  uint8_t *Ht = Xt + L::kX;
  float *cs2 = reinterpret_cast<float *>(Ht + L::kH);  // cs * log2(e)
  float *ecs = cs2 + Q;                                // exp(cs)
  float *cf = ecs + Q;                                 // exp(cs_{j|31} - cs_j)
  float *wsum = cf + Q;                                // per-warp scan totals
  float *D_s = wsum + 32;                              // D of this CTA's heads
  float *dA_s = D_s + KMAX;                            // softplus(dt) * A  [Q][KMAX]
  uint64_t *bars = reinterpret_cast<uint64_t *>(dA_s + Q * KMAX);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + L::kBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);

  const int c = blockIdx.y, b = blockIdx.z;
  const int h_begin = blockIdx.x * heads_per_cta;
  const int nh = min(H, h_begin + heads_per_cta) - h_begin;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hpg_b = H / GB, hpg_c = H / GC;
  auto new_group_at = [&](int k) {
    const int h = h_begin + k;
    return k == 0 || h / hpg_b != (h - 1) / hpg_b || h / hpg_c != (h - 1) / hpg_c;
  };

  if (tid == 0) {
    for (int i = 0; i < L::kBars; ++i) {
      const bool per_warp = i == kBarA2a || i == kBarA2b || i == kBarYFree;
      mbar_init(&bars[i], per_warp ? CW : 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == CW) tmem_alloc(tslot, L::kAlloc);
  if (warp < CW) {
    // this CTA's D and softplus(dt) * A for its heads and chunk, staged once
    if (tid < nh) D_s[tid] = D ? D[h_begin + tid] : 0.f;
    const int64_t t_row0 = static_cast<int64_t>(c) * Q;
    for (int idx = tid; idx < Q * nh; idx += 32 * CW) {
      const int t = idx / nh, k = idx % nh;
      float v = 0.f;
      if (t_row0 + t < T) {
        const float z = dt[(static_cast<int64_t>(b) * T + t_row0 + t) * H + h_begin + k];
        v = (softplus ? softplus_f32(z) : z) * A[h_begin + k];
      }
      dA_s[t * KMAX + k] = v;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;

  if (warp == CW) {
    // ================================================================ control
    if (lane == 0) {
      prefetch_tensormap(&mapC32);
      prefetch_tensormap(&mapB);
      prefetch_tensormap(&mapX);
      prefetch_tensormap(&mapH);
      const uint32_t ct = smem_u32(Ct), bt = smem_u32(Bt), xt = smem_u32(Xt), ht = smem_u32(Ht);
      const int hrow = (b * nc + c) * H;
      auto load_x = [&](int hh) {
        mbar_arrive_expect_tx(&bars[kBarX], L::kX);
#pragma unroll
        for (int s = 0; s < P / 64; ++s)
          tma_load_4d(Xt + s * Q * 128, &mapX, &bars[kBarX], 64 * s, hh, c * Q, b);
      };
      auto load_h = [&](int hh) {
        mbar_arrive_expect_tx(&bars[kBarH], L::kH);
#pragma unroll
        for (int s = 0; s < P / 64; ++s)
          tma_load_3d(Ht + s * N * 128, &mapH, &bars[kBarH], 64 * s, 0, hrow + hh);
      };
      load_x(h_begin);
      load_h(h_begin);
      int group = -1;
      for (int k = 0; k < nh && !*abort_flag; ++k) {
        const int h = h_begin + k;
        const bool more = k + 1 < nh;
        if (more) {  // warm L2 with the next head's tiles
#pragma unroll
          for (int s = 0; s < P / 64; ++s) {
            tma_prefetch_4d(&mapX, 64 * s, h + 1, c * Q, b);
            tma_prefetch_3d(&mapH, 64 * s, 0, hrow + h + 1);
          }
        }
        if (new_group_at(k)) {
          ++group;
          // the previous head's y stores must have left the B/A2 region
          if (k > 0 && !mbar_wait(&bars[kBarStore], (k - 1) & 1, abort_flag)) break;
          mbar_arrive_expect_tx(&bars[kBarCB], L::kC + L::kB);
#pragma unroll
          for (int s = 0; s < N / 64; ++s) {
#pragma unroll
            for (int rb = 0; rb < Q / 32; ++rb)
              tma_load_4d(Ct + s * Q * 128 + rb * 32 * 128, &mapC32, &bars[kBarCB], 64 * s,
                          h / hpg_c, c * Q + scan_row<MT>(32 * rb), b);
            tma_load_4d(Bt + s * Q * 128, &mapB, &bars[kBarCB], 64 * s, h / hpg_b, c * Q, b);
          }
          if (!mbar_wait(&bars[kBarCB], group & 1, abort_flag)) break;
          tc_fence_after_sync();
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t idesc = idesc_bf16(128, 128 * (mt + 1), false, false);
            const uint32_t dcol = 128 * mt * (mt + 1) / 2;
#pragma unroll
            for (int ks = 0; ks < N / 16; ++ks) {
              const uint32_t koff = (ks >> 2) * Q * 128 + (ks & 3) * 32;
              mma_bf16(tmem + dcol, sdesc_sw128(ct + koff + mt * 128 * 128, 16, 1024),
                       sdesc_sw128(bt + koff, 16, 1024), idesc, ks > 0 ? 1u : 0u);
            }
          }
          mma_commit(&bars[kBarS]);
        }
        // MMA3: Y_mt = C_mt Hin   (needs Hin and the previous head's Y read out)
        if (!mbar_wait(&bars[kBarH], k & 1, abort_flag)) break;
        if (k > 0 && !mbar_wait(&bars[kBarYFree], (k - 1) & 1, abort_flag)) break;
        tc_fence_after_sync();
        constexpr uint32_t idesc_y = idesc_bf16(128, P, false, true);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int ks = 0; ks < N / 16; ++ks) {
            const uint64_t ad =
                sdesc_sw128(ct + (ks >> 2) * Q * 128 + (ks & 3) * 32 + mt * 128 * 128, 16, 1024);
            mma_bf16(tmem + L::kSCols + mt * P, ad, sdesc_sw128(ht + ks * 2048, N * 128, 1024),
                     idesc_y, ks > 0 ? 1u : 0u);
          }
        }
        mma_commit(&bars[kBarM3]);
        if (!mbar_wait(&bars[kBarM3], k & 1, abort_flag)) break;
        if (more) load_h(h + 1);
        // MMA2: Y_mt += A2_mt x, each row tile as soon as its A2 block is written
        if (!mbar_wait(&bars[kBarX], k & 1, abort_flag)) break;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const bool last = mt + 1 == MT;
          if (!mbar_wait(&bars[last ? kBarA2b : kBarA2a], k & 1, abort_flag)) break;
          tc_fence_after_sync();
          const uint32_t a2 = bt + 128 * 128 * 2 * (mt * (mt + 1) / 2);
#pragma unroll
          for (int ks = 0; ks < 8 * (mt + 1); ++ks) {
            const uint64_t ad = sdesc_sw128(a2 + (ks >> 2) * (128 * 128) + (ks & 3) * 32, 16, 1024);
            mma_bf16(tmem + L::kSCols + mt * P, ad, sdesc_sw128(xt + ks * 2048, Q * 128, 1024),
                     idesc_y, 1u);
          }
          mma_commit(&bars[last ? kBarM2b : kBarM2a]);
        }
        if (*abort_flag) break;
        if (!mbar_wait(&bars[kBarM2b], k & 1, abort_flag)) break;
        if (more) load_x(h + 1);
      }
    }
    __syncwarp();
  } else {
    // ================================================================ compute
    const int q = warp & 3, hs = warp >> 2;  // TMEM lane quarter, sub-warp of the quarter
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    // in-chunk inclusive cumsum of dA for head index k -> cs2, ecs, cf
    auto cumsum = [&](int k) {
      float v = tid < Q ? dA_s[tid * KMAX + k] : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += o;
      }
      if (lane == 31) wsum[warp] = v;
      compute_sync();
      if (tid < Q) {
        float base = 0.f;
        for (int w = 0; w < warp; ++w) base += wsum[w];
        v += base;
        cs2[tid] = v * kLog2e;
        ecs[tid] = ex2_approx(v * kLog2e);
      }
      compute_sync();
      if (tid < Q) cf[tid] = ex2_approx(cs2[tid | 31] - cs2[tid]);
      compute_sync();
    };
    auto mask_band = [&](int mt, int kb, float Dh) {
      scan_mask_band<MT>(Bt, tmem + lane_base, cs2, cf, q, lane, mt, kb, Dh);
    };
    constexpr int CPW = P / 4;  // Y columns per warp of a quarter
    // y staging of row tile mt: the first A2 block for tile 0, the second for tile 1
    auto stage_of = [&](int mt) { return Bt + 128 * 128 * 2 * (mt * (mt + 1) / 2); };

    cumsum(0);
    int group = -1;
    for (int k = 0; k < nh; ++k) {
      const int h = h_begin + k;
      const bool more = k + 1 < nh;
      const bool new_group = new_group_at(k);
      if (new_group) ++group;
      // The previous head's y stores must have read their staging before the
      // A2 blocks are rewritten.  kBarStore is arrived once per head k >= 1
      // when both have; a new group (whose B tile overwrites the whole region)
      // waits for that before its C B^T product.
      const bool full_wait = MT == 1 || new_group;
      if (k > 0) {
        if (tid == 0) {
          if (full_wait) {
            bulk_wait_read0();
            mbar_arrive(&bars[kBarStore]);
          } else {
            bulk_wait_read1();  // tile 0's staging only
          }
        }
        compute_sync();
      }
      const bool ok_s = !new_group || mbar_wait(&bars[kBarS], group & 1, abort_flag);
      const bool ok = __all_sync(0xffffffffu, ok_s) && !*abort_flag;
      tc_fence_after_sync();
      const float Dh = D_s[k];
      if (ok) mask_band(0, hs, Dh);
      // ---- Y *= exp(cs_i) once MMA3 (Y = C Hin) is done
      bool ok3 = ok && mbar_wait(&bars[kBarM3], k & 1, abort_flag);
      ok3 = __all_sync(0xffffffffu, ok3);
      tc_fence_after_sync();
      if (ok3) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const float e_i = ecs[scan_row<MT>(128 * mt + 32 * q + lane)];
          const uint32_t dcol = L::kSCols + mt * P + CPW * hs;
#pragma unroll
          for (int cc = 0; cc < CPW; cc += 16) {
            float v[16];
            tmem_ld16(tmem + lane_base + dcol + cc, v);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] *= e_i;
            tmem_st16(tmem + lane_base + dcol + cc, v);
          }
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[MT == 2 ? kBarA2a : kBarA2b]);
      if (MT == 2) {
        if (k > 0 && !full_wait) {  // the previous head's tile-1 store has read its staging
          if (tid == 0) {
            bulk_wait_read0();
            mbar_arrive(&bars[kBarStore]);
          }
          compute_sync();
        }
        if (ok3) {
          mask_band(1, hs, Dh);
          mask_band(1, hs + 4, Dh);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarA2b]);
      }
      // ---- next head's cumsum overlaps the last MMA2
      if (more) cumsum(k + 1);
      // ---- output: Y -> bf16 -> staging per row tile, then TMA stores
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        bool ok2 = ok3 && mbar_wait(mt + 1 < MT ? &bars[kBarM2a] : &bars[kBarM2b], k & 1, abort_flag);
        ok2 = __all_sync(0xffffffffu, ok2);
        tc_fence_after_sync();
        if (!ok2) continue;
        const int r = 32 * q + lane;
        const int row = scan_row<MT>(128 * mt + r) - 128 * mt;  // row within the tile
        uint8_t *stage = stage_of(mt);
#pragma unroll
        for (int cc = 0; cc < CPW; cc += 16) {
          float v[16];
          tmem_ld16(tmem + lane_base + L::kSCols + mt * P + CPW * hs + cc, v);
          const int col = CPW * hs + cc;
#pragma unroll
          for (int e = 0; e < 16; e += 8)
            *reinterpret_cast<uint4 *>(stage + ((col + e) >> 6) * (128 * 128) +
                                       sw128_offset(row, (col + e) & 63)) =
                make_uint4(pack_bf16x2(v[e], v[e + 1]), pack_bf16x2(v[e + 2], v[e + 3]),
                           pack_bf16x2(v[e + 4], v[e + 5]), pack_bf16x2(v[e + 6], v[e + 7]));
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarYFree]);
      fence_proxy_async_smem();
      compute_sync();
      if (tid == 0 && !*abort_flag) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
          for (int s = 0; s < P / 64; ++s)
            tma_store_4d(&mapY128, stage_of(mt) + s * (128 * 128), 64 * s, h, c * Q + 128 * mt, b);
          bulk_commit();
        }
      }
    }
    if (tid == 0) bulk_wait_all();
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == CW) tmem_dealloc(tmem, L::kAlloc);
}

}  // namespace ssd
