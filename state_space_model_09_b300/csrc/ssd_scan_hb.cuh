// ssd_scan_hb.cuh -- chunk_scan for 256-token chunks, 64-wide heads and one
// (B, C) group, two heads per MMA.
//
// Same result as chunk_scan_hl (ssd_scan.cuh): for one (batch b, chunk c) and
// each head h, with a = cs * log2(e) the in-chunk inclusive running sum of
// softplus(dt) * A_h in log2 units (summed here from u = softplus(dt) A
// log2(e), written by dt_decay_kernel) and Hin the chunk's true initial state,
//   y_i = sum_{j <= i} 2^(a_i - a_j) S_ij x_j + 2^(a_i) (C Hin)_i + D_h x_i,   S = C B^T
// (Mamba-2 page, section "SSD算法": the orange diagonal block in quadratic
// form and the blue term from the true initial state).
//
// Scaled form.  Taking 2^(a_i - r) out of row i, for a reference r <= 0 of
// the (batch, chunk, head),
//   y_i = 2^(a_i - r) [ sum_{j <= i} S_ij (2^(r - a_j) x_j) + (C 2^r Hin)_i
//                       + D_h 2^(r - a_i) x_i ],
// the masked matrix (j <= i) o S no longer depends on the head: it is formed
// once per CTA and is the A operand of every head's second MMA, while the
// head's decay rides on its x rows (x_j 2^(r - a_j), the B operand).  Two
// heads share every MMA (N = 2 x 64): C [2^r Hin_h | 2^r' Hin_h'] and the three
// masked blocks of S times [x~_h | x~_h'].  No per-head mask, half the MMA
// instructions of a 64-column head.
//
// Range.  r = min(0, a_last + 96) (scaled_form_ref, ssd_tc.cuh) keeps every
// factor within 2^-96 .. 2^96 while a_last >= -192; the chunk-state kernel,
// which runs first, records that per (batch, chunk, head) (flags[(b nc + c) H
// + h] = 1, else 0) and stores those chunk states already multiplied by 2^r.
// The other heads -- chunks whose decay falls below 2^-192 -- are computed by
// the per-head kernel body (scan_hl_body) in the same launch: the launch's
// first CTAs take head-pair items, the rest take the flagged heads of (batch,
// chunk, head set) items -- head set r of R: heads r, r + R, r + 2R, ..., so
// that each set gets about as many of the flagged heads, which a head's decay
// rate makes cluster -- and the flagged items fill the SMs the head-pair
// items leave.
//
// Tensor memory (512 columns): the masked S blocks as packed bf16 pairs --
// rows 0-127 x columns 0-127 ("b00"), rows 128-255 x columns 0-127 ("b10",
// nothing masked), rows 128-255 x columns 128-255 ("b11") -- then C (the A
// operand of the C Hin product), 64 columns per 128-row tile, then Y of one
// row tile for the two heads (128 columns, also the f32 scratch of each S
// piece while the blocks are built).  Shared memory: two 64 KB buffers (C and
// the B tile while S is built; then each head pair's scaled x) and two Hin
// pair buffers.  A pair's tile 1 (rows 128-255) is computed and read out
// first; while tile 0's MMAs run, the compute warps scale the next pair's x,
// which was loaded a pair earlier.  y leaves by TMA stores, staged where
// nothing else is needed any more: tile 1's rows in place of the x rows
// 128-255 (tile 0's MMAs read only rows 0-127), tile 0's rows in the pair's
// Hin buffer (both C Hin products are done by then).  So the x buffer is
// free for the x two pairs ahead once tile 0 is written and tile 1's store
// (issued a tile earlier) has read its rows, and the Hin buffer once tile 0's
// store has read it.
//
// Warp roles: warps 0-15 build the S blocks, copy C, scale x and write y
// (four per TMEM lane quarter); warp 16 (one lane) issues the C/B/Hin and the
// first x loads and every MMA; warp 17 computes each pair's decay tables up
// to two pairs ahead, fetching the next pair's u while it works; warp 18
// (one lane) stores each pair's y and loads the x and Hin two pairs ahead.
// Every wait is bounded in time.
#pragma once

#include "ssd_scan.cuh"

namespace ssd {
constexpr int kHbStoreWarp = kScanComputeWarps + 2;
constexpr int kHbThreads = 32 * (kScanComputeWarps + 3);
constexpr int kHbMaxPairs = 64;  // head pairs per CTA

struct ScanHB {
  static constexpr int Q = 256, P = 64, N = kTcN;
  static constexpr int kXS = 2 * P * Q * 2;  // one buffer: C or B tile, or a scaled x / y pair
  static constexpr int kH = 2 * P * N * 2;   // one Hin pair
  static_assert(kXS == N * Q * 2, "the C and B tiles fill an x buffer");
  static constexpr int kTab = 2 * 2 * Q;     // per buffer: [head][t = 2^-a, e = 2^a][Q]
  // + D and mode of the pair, per buffer; + one mode byte per head of the CTA
  static constexpr int kFloats = 2 * kTab + 8 + 2 * kHbMaxPairs / 4;
  static constexpr int kBars = 24;
  static constexpr int kBytes = 2 * kXS + 2 * kH + kFloats * 4 + kBars * 8 + 16 + 1024;
  // tensor memory columns
  static constexpr uint32_t kA00 = 0, kA10 = 64, kA11 = 128;  // masked S blocks (packed)
  static constexpr uint32_t kC0 = 192, kC1 = 256;             // C row tiles (packed)
  static constexpr uint32_t kY = 320;                         // Y of one row tile, 2 heads
  static constexpr uint32_t kAlloc = 512;
  static_assert(kY + 2 * P <= kAlloc, "TMEM map");
  static_assert(kBytes <= 227 * 1024, "shared memory");
};

enum : int {
  kHbCB = 0, kHbS, kHbConv, kHbX0, kHbX1, kHbH0, kHbH1, kHbXScaled, kHbM2, kHbYFree,
  kHbYStaged, kHbTabFull0, kHbTabFull1, kHbTabEmpty0, kHbTabEmpty1, kHbY1Staged0, kHbY1Staged1,
  kNumHbBars
};
static_assert(kNumHbBars <= ScanHB::kBars, "barrier slots");

__device__ __forceinline__ void tmem_st16_u32(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 "
      "[%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], bf16 inputs, f32 accumulation.  One thread.
// A is M x K with row m in TMEM lane m and K packed two bf16 per column
// (the lower half holds the even element).
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem,
                                                uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 f32 columns of S for the calling thread's row -> 16 packed bf16 pairs,
// column j kept when j <= lim (pass lim >= 31 to keep every column).
__device__ __forceinline__ void hb_mask_pack(const float (&v)[32], int lim, uint32_t (&pk)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e)
    pk[e] = pack_bf16x2(2 * e <= lim ? v[2 * e] : 0.f, 2 * e + 1 <= lim ? v[2 * e + 1] : 0.f);
}

// The body of one head-pair CTA: pair range bx of chunk c of batch row b.
__device__ __forceinline__ void scan_hb_body(
    int bx, int c, int b, const CUtensorMap &mapC32, const CUtensorMap &mapB,
    const CUtensorMap &mapX, const CUtensorMap &mapH, const CUtensorMap &mapY128,
    const float *__restrict__ u, const float *__restrict__ D, const uint8_t *__restrict__ flags,
    int64_t T, int H, int nc, int pairs_per_cta) {
  using L = ScanHB;
  constexpr int Q = L::Q, P = L::P, N = L::N;
  constexpr int CW = kScanComputeWarps;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *Xs = smem;                // two buffers, each [head][Q rows][128 B]
  uint8_t *Hb = Xs + 2 * L::kXS;     // two Hin pair buffers, each [head][N rows][128 B]
  // tab[buf][head][0] = 2^-a_j (0 for a head left to chunk_scan_hl), [1] = 2^a_j
  float *tab = reinterpret_cast<float *>(Hb + 2 * L::kH);
  float *misc = tab + 2 * L::kTab;  // [buf][4]: D of the two heads, their modes
  uint8_t *modes = reinterpret_cast<uint8_t *>(misc + 8);  // [pair][head]: 1 = y written here
  uint64_t *bars = reinterpret_cast<uint64_t *>(modes + 2 * kHbMaxPairs);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + L::kBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);

  const int h_begin = bx * 2 * pairs_per_cta;
  const int h_end = min(H, h_begin + 2 * pairs_per_cta);
  const int npairs = (h_end - h_begin + 1) / 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < L::kBars; ++i) {
      const bool per_warp = i == kHbConv || i == kHbXScaled || i == kHbYFree ||
                            i == kHbYStaged || i == kHbTabEmpty0 || i == kHbTabEmpty1 ||
                            i == kHbY1Staged0 || i == kHbY1Staged1;
      mbar_init(&bars[i], per_warp ? CW : 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kScanControlWarp) tmem_alloc(tslot, L::kAlloc);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;
  auto nheads_of = [&](int pr) { return min(2, h_end - (h_begin + 2 * pr)); };
  // x of pair pr into buffer pr & 1 (issued by one thread)
  auto load_x = [&](int pr) {
    const int n = nheads_of(pr);
    uint64_t *bar = &bars[kHbX0 + (pr & 1)];
    mbar_arrive_expect_tx(bar, n * P * Q * 2);
    for (int hh = 0; hh < n; ++hh)
      tma_load_4d(Xs + (pr & 1) * L::kXS + hh * Q * 128, &mapX, bar, 0, h_begin + 2 * pr + hh,
                  c * Q, b);
  };

  // chunk states of pair pr into Hin buffer pr & 1 (issued by one thread)
  auto load_h = [&](int pr) {
    const int n = nheads_of(pr);
    uint64_t *bar = &bars[kHbH0 + (pr & 1)];
    mbar_arrive_expect_tx(bar, n * P * N * 2);
    for (int hh = 0; hh < n; ++hh)
      tma_load_3d(Hb + (pr & 1) * L::kH + hh * N * 128, &mapH, bar, 0, 0,
                  (b * nc + c) * H + h_begin + 2 * pr + hh);
  };

  if (warp == kScanAuxWarp) {
    // ================================================================ tables
    // Tables of pair pr into buffer pr & 1 (lane owns Q/32 consecutive tokens
    // of the per-token log2 decays u = softplus(dt) A log2(e); running sum,
    // then a warp scan).  The next pair's u, D and modes are fetched before
    // this pair's buffer is waited for.
    constexpr int PER = Q / 32;
    const int64_t t0 = static_cast<int64_t>(c) * Q + lane * PER;
    float z[2][PER], zn[2][PER], Dp[2], Dn[2];
    int Fp[2], Fn[2];
    auto fetch = [&](int pr, float (&zz)[2][PER], float (&dd)[2], int (&ff)[2]) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = min(h_begin + 2 * pr + hh, H - 1);
        const float *uh = u + (static_cast<int64_t>(b) * H + h) * T;
#pragma unroll
        for (int e = 0; e < PER; ++e) zz[hh][e] = t0 + e < T ? uh[t0 + e] : 0.f;
        dd[hh] = D ? D[h] : 0.f;
        ff[hh] = flags[(static_cast<int64_t>(b) * nc + c) * H + h];
      }
    };
    grid_dep_wait();  // u and the flags come from the kernels before this one
    if (npairs > 0) fetch(0, zn, Dn, Fn);
    for (int pr = 0; pr < npairs; ++pr) {
      const int s = pr & 1, n = nheads_of(pr);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        Dp[hh] = Dn[hh];
        Fp[hh] = Fn[hh];
#pragma unroll
        for (int e = 0; e < PER; ++e) z[hh][e] = zn[hh][e];
      }
      if (pr + 1 < npairs) fetch(pr + 1, zn, Dn, Fn);
      if (pr >= 2 && !mbar_wait(&bars[kHbTabEmpty0 + s], ((pr - 2) >> 1) & 1, abort_flag)) break;
      float *tb = tab + s * L::kTab;
      for (int hh = 0; hh < n; ++hh) {
        float v[PER];
        float run = 0.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
          run += z[hh][e];  // 0 past T
          v[e] = run;
        }
        float incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float o = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += o;
        }
        const float base = incl - run;
        const int fast = Fp[hh] != 0;
        // the reference r of the scaled form, from the chunk's total decay
        // (the same running sums as the chunk-state kernel, which stored this
        // head's chunk state times 2^r)
        const float r = scaled_form_ref(__shfl_sync(0xffffffffu, v[PER - 1] + base, 31));
        float *tt = tb + hh * 2 * Q;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
          const float av = v[e] + base;
          tt[lane * PER + e] = fast ? ex2_approx(r - av) : 0.f;
          tt[Q + lane * PER + e] = ex2_approx(av - r);
        }
        if (lane == 0) {
          misc[4 * s + hh] = Dp[hh];
          misc[4 * s + 2 + hh] = fast ? 1.f : 0.f;
          modes[2 * pr + hh] = static_cast<uint8_t>(fast);
        }
      }
      if (n < 2 && lane == 0) {
        misc[4 * s + 3] = 0.f;
        modes[2 * pr + 1] = 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kHbTabFull0 + s]);
    }
  } else if (warp == kHbStoreWarp) {
    // ================================================================ y out, x in
    if (lane == 0) {
      const bool tile1 = static_cast<int64_t>(c) * Q + 128 < T;  // rows 128-255 exist
      for (int pr = 0; pr < npairs; ++pr) {
        const int s = pr & 1, n = nheads_of(pr);
        // tile 1 (rows 128-255), staged in the x buffer
        if (!mbar_wait(&bars[kHbY1Staged0 + s], (pr >> 1) & 1, abort_flag) || *abort_flag) break;
        for (int hh = 0; hh < n && tile1; ++hh)
          if (modes[2 * pr + hh])
            tma_store_4d(&mapY128, Xs + s * L::kXS + hh * Q * 128 + 128 * 128, 0,
                         h_begin + 2 * pr + hh, c * Q + 128, b);
        bulk_commit();
        // tile 0 (rows 0-127), staged in the Hin buffer
        if (!mbar_wait(&bars[kHbYStaged], pr & 1, abort_flag) || *abort_flag) break;
        for (int hh = 0; hh < n; ++hh)
          if (modes[2 * pr + hh])
            tma_store_4d(&mapY128, Hb + s * L::kH + hh * N * 128, 0, h_begin + 2 * pr + hh,
                         c * Q, b);
        bulk_commit();
        bulk_wait_read1();  // tile 1's store has read the x buffer
        if (pr + 2 < npairs) load_x(pr + 2);
        bulk_wait_read0();  // tile 0's store has read the Hin buffer
        if (pr + 2 < npairs) load_h(pr + 2);
      }
      bulk_wait_all();
    }
    __syncwarp();
  } else if (warp == kScanControlWarp) {
    // ================================================================ control
    if (lane == 0 && npairs > 0) {
      prefetch_tensormap(&mapC32);
      prefetch_tensormap(&mapB);
      prefetch_tensormap(&mapH);
      prefetch_tensormap(&mapX);
      prefetch_tensormap(&mapY128);
      const uint32_t xs = smem_u32(Xs), hb = smem_u32(Hb);
      // C into buffer 0, B into buffer 1 (one group: group index 0)
      mbar_arrive_expect_tx(&bars[kHbCB], 2 * L::kXS);
#pragma unroll
      for (int s = 0; s < N / 64; ++s) {
#pragma unroll
        for (int rb = 0; rb < Q / 32; ++rb)
          tma_load_4d(Xs + s * Q * 128 + rb * 32 * 128, &mapC32, &bars[kHbCB], 64 * s, 0,
                      c * Q + 32 * rb, b);
        tma_load_4d(Xs + L::kXS + s * Q * 128, &mapB, &bars[kHbCB], 64 * s, 0, c * Q, b);
      }
      bool ok = mbar_wait(&bars[kHbCB], 0, abort_flag);
      // three S pieces (C0 B0^T, C1 B0^T, C1 B1^T) through the Y columns, each
      // packed by the compute warps before the next
      for (int p = 0; p < 3 && ok; ++p) {
        tc_fence_after_sync();
        const uint32_t arow = p == 0 ? 0u : 128u * 128u, brow = p == 2 ? 128u * 128u : 0u;
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks) {
          const uint32_t koff = (ks >> 2) * Q * 128 + (ks & 3) * 32;
          mma_bf16(tmem + L::kY, sdesc_sw128(xs + koff + arow, 16, 1024),
                   sdesc_sw128(xs + L::kXS + koff + brow, 16, 1024),
                   idesc_bf16(128, 128, false, false), ks > 0 ? 1u : 0u);
        }
        mma_commit(&bars[kHbS]);
        ok = mbar_wait(&bars[kHbConv], p & 1, abort_flag);
      }
      // the set-up above reads inputs only; the chunk states come from the
      // chunk-state kernel, which may still be running when this CTA starts
      grid_dep_wait();
      if (ok) {
        load_h(0);
        if (npairs > 1) load_h(1);
      }
      // C and B are consumed: both buffers take x
      if (ok) {
        load_x(0);
        if (npairs > 1) load_x(1);
      }
      constexpr uint32_t idesc_y = idesc_bf16(128, 2 * P, false, true);
      for (int pr = 0; pr < npairs && ok && !*abort_flag; ++pr) {
        const uint32_t hk = hb + (pr & 1) * L::kH, xk = xs + (pr & 1) * L::kXS;
        if (!mbar_wait(&bars[kHbH0 + (pr & 1)], (pr >> 1) & 1, abort_flag)) break;
        // ---- row tile 1: Y = C1 [Hin | Hin'] + b10 x~[0:128] + b11 x~[128:256]
        if (pr > 0 && !mbar_wait(&bars[kHbYFree], 1, abort_flag)) break;
        tc_fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks)
          mma_bf16_tmem_a(tmem + L::kY, tmem + L::kC1 + 8 * ks,
                          sdesc_sw128(hk + ks * 2048, N * 128, 1024), idesc_y, ks > 0 ? 1u : 0u);
        if (!mbar_wait(&bars[kHbXScaled], pr & 1, abort_flag)) break;
        tc_fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16_tmem_a(tmem + L::kY, tmem + L::kA10 + 8 * ks,
                          sdesc_sw128(xk + ks * 2048, Q * 128, 1024), idesc_y, 1u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16_tmem_a(tmem + L::kY, tmem + L::kA11 + 8 * ks,
                          sdesc_sw128(xk + 128 * 128 + ks * 2048, Q * 128, 1024), idesc_y, 1u);
        mma_commit(&bars[kHbM2]);
        // ---- row tile 0: Y = C0 [Hin | Hin'] + b00 x~[0:128]
        if (!mbar_wait(&bars[kHbYFree], 0, abort_flag)) break;
        tc_fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks)
          mma_bf16_tmem_a(tmem + L::kY, tmem + L::kC0 + 8 * ks,
                          sdesc_sw128(hk + ks * 2048, N * 128, 1024), idesc_y, ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16_tmem_a(tmem + L::kY, tmem + L::kA00 + 8 * ks,
                          sdesc_sw128(xk + ks * 2048, Q * 128, 1024), idesc_y, 1u);
        mma_commit(&bars[kHbM2]);
      }
    }
    __syncwarp();
  } else if (npairs > 0) {
    // ================================================================ compute
    const int q = warp & 3, hs = warp >> 2;  // TMEM lane quarter, sub-warp of the quarter
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const int r = 32 * q + lane;  // row inside a row tile (= TMEM lane)
    bool ok = true;
    // ---- S pieces -> masked, packed blocks; C -> tensor memory
    for (int p = 0; p < 3 && ok; ++p) {
      // (the C copy below reads the TMA-written tile: wait on its barrier too)
      bool w = (p > 0 || mbar_wait(&bars[kHbCB], 0, abort_flag)) &&
               mbar_wait(&bars[kHbS], p & 1, abort_flag);
      ok = __all_sync(0xffffffffu, w) && !*abort_flag;
      if (ok) {
        tc_fence_after_sync();
        float v[32];
        uint32_t pk[16];
        tmem_ld32(tmem + lane_base + L::kY + 32 * hs, v);
        hb_mask_pack(v, p == 1 ? 31 : r - 32 * hs, pk);
        tmem_st16_u32(tmem + lane_base + (p == 0 ? L::kA00 : p == 1 ? L::kA10 : L::kA11) + 16 * hs,
                      pk);
        if (p == 0) {
          // C row tiles: row 128 t + r, state columns 32 hs .. + 31 (atom hs / 2)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            uint32_t cw[16];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
              const uint4 u = *reinterpret_cast<const uint4 *>(
                  Xs + (hs >> 1) * Q * 128 + sw128_offset(128 * t + r, 32 * (hs & 1) + 8 * g));
              cw[4 * g] = u.x; cw[4 * g + 1] = u.y; cw[4 * g + 2] = u.z; cw[4 * g + 3] = u.w;
            }
            tmem_st16_u32(tmem + lane_base + (t == 0 ? L::kC0 : L::kC1) + 16 * hs, cw);
          }
        }
        tmem_st_wait();
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kHbConv]);
    }
    // x rows of pair pr *= 2^-a_j in place (16-byte chunks, eight per thread);
    // returns the pair's row factors, D and modes, then frees its tables
    float e[2][2], Dh[2], on[2];
    auto scale = [&](int pr) -> bool {
      const int s = pr & 1;
      bool w = mbar_wait(&bars[kHbTabFull0 + s], (pr >> 1) & 1, abort_flag);
      w = w && mbar_wait(&bars[kHbX0 + s], (pr >> 1) & 1, abort_flag);
      if (!(__all_sync(0xffffffffu, w) && !*abort_flag)) return false;
      const float *tb = tab + s * L::kTab;
      uint8_t *xb = Xs + s * L::kXS;
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const int u = tid + 512 * m;
        const int hh = u >> 11, j = (u >> 3) & 255, cc = u & 7;
        uint4 *p = reinterpret_cast<uint4 *>(xb + hh * Q * 128 + sw128_offset(j, 8 * cc));
        *p = scale_bf16x8(*p, tb[hh * 2 * Q + j]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kHbXScaled]);
      const float *md = misc + 4 * s;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        e[hh][0] = tb[hh * 2 * Q + Q + r];
        e[hh][1] = tb[hh * 2 * Q + Q + 128 + r];
        Dh[hh] = md[hh];
        on[hh] = md[2 + hh];
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kHbTabEmpty0 + s]);
      return true;
    };
    // y rows of row tile t of pair pr = 2^(a_i - r) (Y + D x~) -> bf16, staged
    // for the TMA stores: tile 1 in place of x~, tile 0 in the Hin buffer
    auto output = [&](int pr, int t, const float (&ee)[2][2], const float (&dd)[2],
                      const float (&oo)[2]) -> bool {
      bool w = mbar_wait(&bars[kHbM2], t == 1 ? 0 : 1, abort_flag);
      if (!(__all_sync(0xffffffffu, w) && !*abort_flag)) return false;
      tc_fence_after_sync();
      uint8_t *xb = Xs + (pr & 1) * L::kXS;
      uint8_t *yb = t == 1 ? xb : Hb + (pr & 1) * L::kH;  // [head][rows][128 B]
      const int yhead = t == 1 ? Q * 128 : N * 128;
      const int i = 128 * t + r;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        if (oo[hh] == 0.f) continue;
        float v[16];
        tmem_ld16(tmem + lane_base + L::kY + 64 * hh + 16 * hs, v);
        const float f = ee[hh][t], d = dd[hh];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const uint4 xv = *reinterpret_cast<const uint4 *>(
              xb + hh * Q * 128 + sw128_offset(i, 16 * hs + 8 * g));
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
          uint32_t o[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 xf = unpack_bf16x2(xw[k]);
            o[k] = pack_bf16x2(f * fmaf(d, xf.x, v[8 * g + 2 * k]),
                               f * fmaf(d, xf.y, v[8 * g + 2 * k + 1]));
          }
          *reinterpret_cast<uint4 *>(yb + hh * yhead + sw128_offset(t == 1 ? i : r, 16 * hs + 8 * g)) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      tc_fence_before_sync();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kHbYFree]);
        mbar_arrive(&bars[t == 0 ? kHbYStaged : kHbY1Staged0 + (pr & 1)]);
      }
      return true;
    };
    if (ok) ok = scale(0);
    for (int pr = 0; pr < npairs && ok; ++pr) {
      float ce[2][2] = {{e[0][0], e[0][1]}, {e[1][0], e[1][1]}};
      float cd[2] = {Dh[0], Dh[1]}, co[2] = {on[0], on[1]};
      if (!(ok = output(pr, 1, ce, cd, co))) break;
      if (pr + 1 < npairs && !(ok = scale(pr + 1))) break;
      if (!(ok = output(pr, 0, ce, cd, co))) break;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kScanControlWarp) tmem_dealloc(tmem, L::kAlloc);
}

// Shared memory of the combined launch: the larger of the two bodies.
constexpr int kHbLaunchBytes =
    ScanHB::kBytes > ScanHL<256, 64>::kBytes ? ScanHB::kBytes : ScanHL<256, 64>::kBytes;

// One launch for the chunk outputs of 256-token chunks of one (B, C) group:
// blocks 0 .. hb_ranges nc batch - 1 are head-pair items (pair range, chunk,
// batch row, range fastest); the rest are the flagged heads of (head set,
// chunk, batch row) items, computed per head (head set r of flagged_sets:
// heads r, r + flagged_sets, ...).
__global__ void __launch_bounds__(kHbThreads, 1)
    chunk_scan_hb(const __grid_constant__ CUtensorMap mapC32,
                  const __grid_constant__ CUtensorMap mapB,
                  const __grid_constant__ CUtensorMap mapX,
                  const __grid_constant__ CUtensorMap mapH,
                  const __grid_constant__ CUtensorMap mapY,
                  const __grid_constant__ CUtensorMap mapY128, const float *__restrict__ dt,
                  const float *__restrict__ A, const float *__restrict__ D,
                  const float *__restrict__ u, const uint8_t *__restrict__ flags, int64_t T,
                  int batch, int H, int nc, int pairs_per_cta, int hb_ranges,
                  int flagged_sets, int softplus) {
  const int64_t i = blockIdx.x;
  const int64_t n_hb = static_cast<int64_t>(hb_ranges) * nc * batch;
  if (i < n_hb) {
    scan_hb_body(static_cast<int>(i % hb_ranges), static_cast<int>((i / hb_ranges) % nc),
                 static_cast<int>(i / (static_cast<int64_t>(hb_ranges) * nc)), mapC32, mapB, mapX,
                 mapH, mapY128, u, D, flags, T, H, nc, pairs_per_cta);
  } else {
    grid_dep_wait();  // the flags, u and the chunk states of the kernels before
    const int64_t j = i - n_hb;
    const int set = static_cast<int>(j % flagged_sets), c = static_cast<int>((j / flagged_sets) % nc);
    const int bb = static_cast<int>(j / (static_cast<int64_t>(flagged_sets) * nc));
    // a block whose heads were all computed by the pass before leaves at once,
    // before any set-up (usually all of them: long-decay chunks are rare)
    int any = 0;
    for (int h = set + static_cast<int>(threadIdx.x) * flagged_sets; h < H;
         h += static_cast<int>(blockDim.x) * flagged_sets)
      any |= flags[(static_cast<int64_t>(bb) * nc + c) * H + h] == 0;
    if (!__syncthreads_or(any)) return;
    scan_hl_body<256, 64, true>(set, c, bb, mapC32, mapB, mapX, mapH, mapY, dt, A, D, T, H, 1, 1,
                                nc, flagged_sets, softplus, flags, u);
  }
}

}  // namespace ssd
