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
//   out:   y = bf16(Y), staged in the (then dead) x tile, written by TMA tile stores
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
// mask, scaling and output; warp 16 (one elected lane) issues every TMA load
// and MMA; warp 17 computes each head's in-chunk cumsum and decay tables one
// head ahead into a double buffer.  Every wait is bounded in time.
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

constexpr int kScanComputeWarps = 16;
constexpr int kScanControlWarp = kScanComputeWarps;      // TMA + MMA issue
constexpr int kScanAuxWarp = kScanComputeWarps + 1;      // per-head decay tables
constexpr int kScanThreads = 32 * (kScanComputeWarps + 2);
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
  static constexpr int kMaxHeads = 16;            // most heads per CTA
  static constexpr int kMaxFlaggedHeads = 128;    // ... when computing flagged heads only
  // per-head decay tables, double-buffered: cs*log2e, exp(cs), the factors
  // 2^(a_{j|31} - a_j) and 2^(a_{j&~31} - a_j); plus D of the CTA's heads
  static constexpr int kTables = 4;
  // + D of the CTA's heads
  static constexpr int kFloats = 2 * kTables * Q + kMaxFlaggedHeads;
  static constexpr int kBars = 16;
  static constexpr int kBytes =
      kC + kU + kX + kH + kFloats * 4 + kBars * 8 + 16 + 4 * (kMaxFlaggedHeads + 2) + 1024;
  static constexpr int kSCols = 128 * MT * (MT + 1) / 2;
  static constexpr int kCols = kSCols + MT * P;
  static constexpr uint32_t kAlloc = kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
  static_assert(kCols <= 512, "TMEM columns exceeded");
  static_assert(kBytes <= 227 * 1024, "shared memory exceeded");
  static constexpr int kThreads = kScanThreads;
};

// kBarM2: every MMA2 of the head done (x tile and A2 blocks free);
// kBarYStaged: the compute warps wrote the head's bf16 y into the x tile;
// kBarXFree: the head's y store has read the x tile (the next x may land).
enum : int {
  kBarCB = 0, kBarX, kBarH, kBarS, kBarM3, kBarM2a, kBarM2, kBarA2a, kBarA2b, kBarYFree, kBarXFree,
  kBarTabFull0, kBarTabFull1, kBarTabEmpty0, kBarTabEmpty1, kBarYStaged, kNumScanBars
};
static_assert(kNumScanBars <= ScanHL<128, 64>::kBars, "barrier slots");

// Chunk row held by smem/TMEM row s of the C tile (see "Row order" above).
template <int MT>
__device__ __forceinline__ int scan_row(int s) {
  if (MT == 1 || s < 128) return s;
  return 128 + 32 * (3 - ((s - 128) >> 5)) + (s & 31);
}

// Masked scores of one 32-column band kb of row tile mt for the calling warp's
// 32 rows: A2 = bf16(L o S + D I) written into the swizzled A2 block.  With
// a = cs * log2(e) (non-increasing):
//   band left of the row's band : L = 2^(a_i - a_ref) * 2^(a_ref - a_j), ref = band end
//                                 (both factors <= 1);
//   the row's own band          : L = 2^(a_i - a_r) * 2^(a_r - a_j), r = band start,
//                                 when the band's range a_r - a_{r+31} < 100 (so the
//                                 second factor cannot overflow); otherwise one
//                                 exponential per element.
// Kept out of line: one copy serves every band, which keeps the code small.
template <int MT>
__device__ __noinline__ void scan_mask_band(uint8_t *Bt, uint32_t tlane, const float *a,
                                            const float *cf, const float *ce, int q, int lane,
                                            int mt, int kb, float Dh) {
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
    const float ai = a[i];
    const int j0 = 32 * kb;
    if (kb < diag_band) {
      const float rf = ex2_approx(ai - a[j0 + 31]);
      const float4 *c4 = reinterpret_cast<const float4 *>(cf + j0);
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 f = c4[e >> 2];
        pk[e >> 1] = pack_bf16x2(v[e] * rf * f.x, v[e + 1] * rf * f.y);
        pk[(e >> 1) + 1] = pack_bf16x2(v[e + 2] * rf * f.z, v[e + 3] * rf * f.w);
      }
    } else if (a[j0] - a[j0 + 31] < 100.f) {
      const float g = ex2_approx(ai - a[j0]);
      const float4 *e4 = reinterpret_cast<const float4 *>(ce + j0);
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 f = e4[e >> 2];
        const int j = j0 + e;
        float l0 = j <= i ? v[e] * g * f.x : 0.f;
        float l1 = j + 1 <= i ? v[e + 1] * g * f.y : 0.f;
        float l2 = j + 2 <= i ? v[e + 2] * g * f.z : 0.f;
        float l3 = j + 3 <= i ? v[e + 3] * g * f.w : 0.f;
        if (j == i) l0 += Dh;
        if (j + 1 == i) l1 += Dh;
        if (j + 2 == i) l2 += Dh;
        if (j + 3 == i) l3 += Dh;
        pk[e >> 1] = pack_bf16x2(l0, l1);
        pk[(e >> 1) + 1] = pack_bf16x2(l2, l3);
      }
    } else {
      const float4 *a4 = reinterpret_cast<const float4 *>(a + j0);
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 f = a4[e >> 2];
        const int j = j0 + e;
        float l0 = j <= i ? v[e] * ex2_approx(ai - f.x) : 0.f;
        float l1 = j + 1 <= i ? v[e + 1] * ex2_approx(ai - f.y) : 0.f;
        float l2 = j + 2 <= i ? v[e + 2] * ex2_approx(ai - f.z) : 0.f;
        float l3 = j + 3 <= i ? v[e + 3] * ex2_approx(ai - f.w) : 0.f;
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

// The body of one CTA: head range bx of chunk c of batch row b.  FLAGGED:
// the heads bx, bx + heads_per_cta, bx + 2 heads_per_cta, ... (interleaved, so
// that the few heads a long decay flags spread evenly over the CTAs), and of
// those only the ones whose byte in only_flagged is 0 (the heads left by the
// head-pair kernel); their decays come from u, the per-token log2 decays
// softplus(dt) A log2(e) with each head's tokens contiguous.  Otherwise every
// head of the range bx heads_per_cta ... (bx + 1) heads_per_cta - 1.
// Warps 0-17 take part (warps past them, in a wider launch, only wait).
template <int Q, int P, bool FLAGGED>
__device__ __forceinline__ void scan_hl_body(
    int bx, int c, int b, const CUtensorMap &mapC32, const CUtensorMap &mapB,
    const CUtensorMap &mapX, const CUtensorMap &mapH, const CUtensorMap &mapY,
    const float *__restrict__ dt, const float *__restrict__ A, const float *__restrict__ D,
    int64_t T, int H, int GB, int GC, int nc, int heads_per_cta, int softplus,
    const uint8_t *__restrict__ only_flagged, const float *__restrict__ u) {
  using L = ScanHL<Q, P>;
  constexpr int N = L::N, MT = L::MT, KMAX = FLAGGED ? L::kMaxFlaggedHeads : L::kMaxHeads;
  constexpr int CW = kScanComputeWarps;
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *Ct = smem;
  uint8_t *Bt = Ct + L::kC;  // B tile, then the A2 blocks (and the y staging)
  uint8_t *Xt = Bt + L::kU;
  uint8_t *Ht = Xt + L::kX;
  // tables[buf][t][Q]: t = 0 a = cs*log2(e), 1 exp(cs), 2 2^(a_{j|31}-a_j), 3 2^(a_{j&~31}-a_j)
  float *tables = reinterpret_cast<float *>(Ht + L::kH);
  float *D_s = tables + 2 * L::kTables * Q;            // D of this CTA's heads
  uint64_t *bars = reinterpret_cast<uint64_t *>(D_s + KMAX);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + L::kBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
  int *hlist = reinterpret_cast<int *>(tslot + 4);  // FLAGGED: the heads this CTA computes
  int *nh_s = hlist + KMAX;

  const int h_begin = FLAGGED ? bx : bx * heads_per_cta;
  const int h_step = FLAGGED ? heads_per_cta : 1;  // the stride of the CTA's heads
  const int nh_all = FLAGGED ? (H - bx + heads_per_cta - 1) / heads_per_cta
                             : min(H, h_begin + heads_per_cta) - h_begin;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hpg_b = H / GB, hpg_c = H / GC;
  auto head_at = [&](int k) { return FLAGGED ? hlist[k] : h_begin + k; };
  auto new_group_at = [&](int k) {
    const int h = head_at(k), hp = FLAGGED ? (k > 0 ? hlist[k - 1] : h) : h - 1;
    return k == 0 || h / hpg_b != hp / hpg_b || h / hpg_c != hp / hpg_c;
  };

  if (tid == 0) {
    for (int i = 0; i < L::kBars; ++i) {
      const bool per_warp = i == kBarA2a || i == kBarA2b || i == kBarYFree ||
                            i == kBarTabEmpty0 || i == kBarTabEmpty1 || i == kBarYStaged;
      mbar_init(&bars[i], per_warp ? CW : 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // the heads to compute: all of the range, or (FLAGGED) those a preceding
  // kernel flagged 0, selected in parallel and compacted by thread 0
  if (FLAGGED) {
    for (int k = tid; k < nh_all; k += blockDim.x) {
      const int h = h_begin + k * h_step;
      hlist[k] = only_flagged[(static_cast<int64_t>(b) * nc + c) * H + h] == 0;
      D_s[k] = D ? D[h] : 0.f;
    }
  } else if (tid < nh_all) {
    D_s[tid] = D ? D[h_begin + tid] : 0.f;
  }
  if (warp == kScanControlWarp) tmem_alloc(tslot, L::kAlloc);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  int nh = nh_all;
  if (FLAGGED) {
    if (tid == 0) {
      int n = 0;
      for (int k = 0; k < nh_all; ++k) {
        if (hlist[k]) {
          hlist[n] = h_begin + k * h_step;
          D_s[n] = D_s[k];
          ++n;
        }
      }
      *nh_s = n;
    }
    __syncthreads();
    nh = *nh_s;
  }
  const uint32_t tmem = *tslot;

  if (warp == kScanAuxWarp) {
    // ================================================================ aux
    // Decay tables of head k into buffer k & 1, one head ahead of the compute
    // warps: lane owns Q/32 consecutive tokens; running sum, then a warp scan.
    // It also writes each head's y: once the compute warps have staged it in
    // the x tile, one TMA store per 64 columns, and it frees the x tile for
    // the next head as soon as the store has read it.
    constexpr int PER = Q / 32;
    const int64_t t0 = static_cast<int64_t>(c) * Q + lane * PER;
    for (int k = 0; k <= nh; ++k) {
      if (k < nh) {
        const int h = head_at(k), s = k & 1;
        float z[PER];
        const float *uh = FLAGGED ? u + (static_cast<int64_t>(b) * H + h) * T : nullptr;
#pragma unroll
        for (int e = 0; e < PER; ++e)
          z[e] = t0 + e >= T ? 0.f
                 : FLAGGED  ? uh[t0 + e]
                            : dt[(static_cast<int64_t>(b) * T + t0 + e) * H + h];
        const float Ah = A[h];
        if (k >= 2 && !mbar_wait(&bars[kBarTabEmpty0 + s], ((k - 2) >> 1) & 1, abort_flag)) break;
        float v[PER];
        float run = 0.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
          if (FLAGGED) run += z[e];  // already in log2 units; 0 past T
          else if (t0 + e < T) run += (softplus ? softplus_f32(z[e]) : z[e]) * Ah;
          v[e] = run;
        }
        float incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float o = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += o;
        }
        const float base = incl - run;
        float *ta = tables + s * L::kTables * Q;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
          const float av = FLAGGED ? v[e] + base : (v[e] + base) * kLog2e;
          ta[lane * PER + e] = av;
          ta[Q + lane * PER + e] = ex2_approx(av);
        }
        __syncwarp();
#pragma unroll
        for (int e = 0; e < PER; ++e) {
          const int j = lane * PER + e;
          const float av = ta[j];
          ta[2 * Q + j] = ex2_approx(ta[j | 31] - av);
          ta[3 * Q + j] = ex2_approx(ta[j & ~31] - av);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarTabFull0 + s]);
      }
      if (k >= 1) {
        const int kp = k - 1;
        const bool ok = mbar_wait(&bars[kBarYStaged], kp & 1, abort_flag);
        if (lane == 0) {
          if (ok && !*abort_flag) {
#pragma unroll
            for (int s = 0; s < P / 64; ++s)
              tma_store_4d(&mapY, Xt + s * Q * 128, 64 * s, head_at(kp), c * Q, b);
            bulk_commit();
            bulk_wait_read0();
          }
          mbar_arrive(&bars[kBarXFree]);
        }
        __syncwarp();
        if (!ok) break;
      }
    }
    if (lane == 0) bulk_wait_all();
  } else if (warp == kScanControlWarp) {
    // ================================================================ control
    if (lane == 0 && nh > 0) {
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
      load_x(head_at(0));
      load_h(head_at(0));
      int group = -1;
      for (int k = 0; k < nh && !*abort_flag; ++k) {
        const int h = head_at(k);
        const bool more = k + 1 < nh;
        if (new_group_at(k)) {
          ++group;
          // every earlier reader of C, B/A2 and S has finished (MMA2 of k - 1 waited below)
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
        if (more) load_h(head_at(k + 1));
        // MMA2: Y_mt += A2_mt x, the last row tile first (its mask is written first)
        if (!mbar_wait(&bars[kBarX], k & 1, abort_flag)) break;
        bool failed = false;
#pragma unroll
        for (int mi = 0; mi < MT; ++mi) {
          const int mt = MT - 1 - mi;
          if (!mbar_wait(&bars[mt == MT - 1 ? kBarA2b : kBarA2a], k & 1, abort_flag)) {
            failed = true;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a2 = bt + 128 * 128 * 2 * (mt * (mt + 1) / 2);
#pragma unroll
          for (int ks = 0; ks < 8 * (mt + 1); ++ks) {
            const uint64_t ad = sdesc_sw128(a2 + (ks >> 2) * (128 * 128) + (ks & 3) * 32, 16, 1024);
            mma_bf16(tmem + L::kSCols + mt * P, ad, sdesc_sw128(xt + ks * 2048, Q * 128, 1024),
                     idesc_y, 1u);
          }
          if (mi + 1 < MT) mma_commit(&bars[kBarM2a]);
        }
        if (failed) break;
        mma_commit(&bars[kBarM2]);
        if (!mbar_wait(&bars[kBarM2], k & 1, abort_flag)) break;
        // the x tile now holds this head's y until its store has read it
        if (more) {
          if (!mbar_wait(&bars[kBarXFree], k & 1, abort_flag)) break;
          load_x(head_at(k + 1));
        }
      }
    }
    __syncwarp();
  } else if (warp < CW) {
    // ================================================================ compute
    const int q = warp & 3, hs = warp >> 2;  // TMEM lane quarter, sub-warp of the quarter
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    float *a_tab = tables, *e_tab = tables + Q, *cf_tab = tables + 2 * Q, *ce_tab = tables + 3 * Q;
    auto mask_band = [&](int mt, int kb, float Dh) {
      scan_mask_band<MT>(Bt, tmem + lane_base, a_tab, cf_tab, ce_tab, q, lane, mt, kb, Dh);
    };
    constexpr int CPW = P / 4;  // Y columns per warp of a quarter

    int group = -1;
    for (int k = 0; k < nh; ++k) {
      const int tb = k & 1;  // this head's table buffer
      a_tab = tables + tb * L::kTables * Q;
      e_tab = a_tab + Q;
      cf_tab = a_tab + 2 * Q;
      ce_tab = a_tab + 3 * Q;
      const bool new_group = new_group_at(k);
      if (new_group) ++group;
      bool ok_s = !new_group || mbar_wait(&bars[kBarS], group & 1, abort_flag);
      ok_s = ok_s && mbar_wait(&bars[kBarTabFull0 + tb], (k >> 1) & 1, abort_flag);
      const bool ok = __all_sync(0xffffffffu, ok_s) && !*abort_flag;
      tc_fence_after_sync();
      const float Dh = D_s[k];
      // ---- last row tile's mask first: its MMA2 then overlaps the other tile's mask
      if (ok && MT == 2) {
        mask_band(1, hs, Dh);
        mask_band(1, hs + 4, Dh);
      }
      if (ok && MT == 1) mask_band(0, hs, Dh);
      // ---- Y *= exp(cs_i) once MMA3 (Y = C Hin) is done
      bool ok3 = ok && mbar_wait(&bars[kBarM3], k & 1, abort_flag);
      ok3 = __all_sync(0xffffffffu, ok3);
      tc_fence_after_sync();
      if (ok3) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const float e_i = e_tab[scan_row<MT>(128 * mt + 32 * q + lane)];
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
      if (lane == 0) mbar_arrive(&bars[kBarA2b]);
      if (MT == 2) {
        if (ok3) mask_band(0, hs, Dh);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarA2a]);
      }
      // ---- this head's decay tables are no longer needed
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarTabEmpty0 + tb]);
      // ---- output: after every MMA2 (the x tile is then free), Y -> bf16 -> x tile
      bool ok2 = ok3 && mbar_wait(&bars[kBarM2], k & 1, abort_flag);
      ok2 = __all_sync(0xffffffffu, ok2);
      tc_fence_after_sync();
      if (ok2) {
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int row = scan_row<MT>(128 * mt + 32 * q + lane);  // chunk row
#pragma unroll
          for (int cc = 0; cc < CPW; cc += 16) {
            float v[16];
            tmem_ld16(tmem + lane_base + L::kSCols + mt * P + CPW * hs + cc, v);
            const int col = CPW * hs + cc;
#pragma unroll
            for (int e = 0; e < 16; e += 8)
              *reinterpret_cast<uint4 *>(Xt + ((col + e) >> 6) * Q * 128 +
                                         sw128_offset(row, (col + e) & 63)) =
                  make_uint4(pack_bf16x2(v[e], v[e + 1]), pack_bf16x2(v[e + 2], v[e + 3]),
                             pack_bf16x2(v[e + 4], v[e + 5]), pack_bf16x2(v[e + 6], v[e + 7]));
          }
        }
      }
      tc_fence_before_sync();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kBarYFree]);
        mbar_arrive(&bars[kBarYStaged]);
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kScanControlWarp) tmem_dealloc(tmem, L::kAlloc);
}

template <int Q, int P>
__global__ void __launch_bounds__(kScanThreads, 1)
    chunk_scan_hl(const __grid_constant__ CUtensorMap mapC32, const __grid_constant__ CUtensorMap mapB,
                  const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapH,
                  const __grid_constant__ CUtensorMap mapY, const float *__restrict__ dt,
                  const float *__restrict__ A, const float *__restrict__ D, int64_t T, int H,
                  int GB, int GC, int nc, int heads_per_cta, int softplus) {
  scan_hl_body<Q, P, false>(blockIdx.x, blockIdx.y, blockIdx.z, mapC32, mapB, mapX, mapH, mapY,
                            dt, A, D, T, H, GB, GC, nc, heads_per_cta, softplus, nullptr,
                            nullptr);
}

}  // namespace ssd
