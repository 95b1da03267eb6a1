// ssd_fused_hb.cuh -- the chunked SSD prefill in one pass over the sequence,
// for 256-token chunks, 64-wide heads and one (B, C) group: two heads per MMA,
// the running state kept on chip from the first chunk to the last.
//
// The four steps of the chunked algorithm (Mamba-2 page, section "SSD算法"):
// the diagonal blocks in quadratic form (orange), each chunk's state from a
// zero start (green), the scan of states across chunks (yellow) and each
// chunk's output from its true initial state (blue).  Here one CTA takes a
// (batch row, head pair) -- or a segment of its chunks -- and walks its
// chunks in order, so the state that enters a chunk is already in registers
// when the chunk is reached: the blue term needs no chunk states in memory,
// and x is read once.  Each 256-token chunk is taken as two 128-token stages
// (the chunk's diagonal block split in two, with the state carried from the
// first stage to the second -- the same decomposition one level down).
//
// Per stage (128 tokens; a = running log2 decay from the stage start, a_j
// inclusive; r a reference <= 0 per (stage, head)), for each head of the pair:
//   x~_j = bf16(2^(r - a_j) x_j)                                   (scale)
//   P    = C B^T, masked to j <= i, as bf16 pairs in tensor memory  (mask)
//   Y    = C H~ + P x~,  H~ = bf16(2^r state)                       (two MMAs)
//   y_i  = 2^(a_i - r) (Y_i + D x~_i)                               (epilogue)
//   S    = B^T x~                                                   (MMA)
//   state <- 2^(a_last) state + 2^(a_last - r) S                     (fold)
// which is exact algebra for y_i = sum_{j<=i} 2^(a_i - a_j) (C_i.B_j) x_j +
// 2^(a_i) C_i.state + D x_i and for the state recurrence.  The masked P does
// not depend on the head, so both heads share every MMA (N = 2 x 64).
//
// Range.  With r = min(0, a_last + 96) every factor stays within 2^-96 ..
// 2^96 as long as a_last >= -192 (ssd_tc.cuh).  A (chunk, head) in which
// either stage decays further is flagged: both its stages take r = a_last
// (factors <= 1, so the state is still exact), its y is left unwritten, and
// the chunk's entering state (bf16), its per-token log2 decays u and a flag
// byte 0 are stored for the per-head chunk-scan body, which computes that
// (chunk, head) in the launch after this one; every other (chunk, head) gets
// flag byte 1.
//
// Segments.  To fill the SMs, the (batch row, head pair) items of a last,
// partly filled wave (or all items, when they are fewer than the SMs) are
// split into `nseg` segments of `cps` chunks.  A prepass launch of this
// kernel (FULL = false: the state path alone) computes for every segment but
// the last its final state from a zero start (segment 0 from h0) and its
// total decay; the segment's CTA in the full launch then starts from
//   T_s = sum_{s' < s} (prod_{s' < k < s} Lambda_k) F_s'
// (the yellow scan one level up) and needs no correction afterwards.
//
// Shared memory: three x stage slots (x of both heads, 32 KB each; a slot
// later holds that stage's y for its TMA store), one C landing slot (copied
// into tensor memory on arrival, the A operand of C B^T and of C H~), one B
// slot (a second one in the prepass, which has no C), the H~ pair (32 KB) and
// four stage-table buffers.  Tensor memory (512 columns): Y (128), S (128),
// the f32 C B^T (128), the masked P (64, packed) and C (64, packed).
//
// Warp roles: warps 0-15 mask, fold, write H~, copy C, scale x and write y
// (four per TMEM lane quarter, thread = one row, 32 columns); warp 16 (one
// lane) issues every MMA and the B and C loads; warps 17 and 18 compute the
// decay tables of one head each, a chunk at a time, from dt; warp 19 (one
// lane) stores y and loads x three stages ahead.  Every wait is bounded.
#pragma once

#include "ssd_scan.cuh"
#include "ssd_scan_hb.cuh"

namespace ssd {

constexpr int kFuWarps = 20;
constexpr int kFuComputeThreads = 32 * 16;
// a barrier among the sixteen compute warps only (threads 0..511)
__device__ __forceinline__ void compute_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kFuComputeThreads) : "memory");
}
constexpr int kFuThreads = 32 * kFuWarps;
constexpr int kFuCompute = 16;
constexpr int kFuControl = 16;
constexpr int kFuTables = 17;  // 17, 18
constexpr int kFuLoader = 19;

struct FusedHB {
  static constexpr int Q = 256, S = 128, P = 64, N = kTcN;
  static constexpr int kTile = 2 * S * 128;  // one stage tile: x pair, or C / B (two 64-column atoms)
  static constexpr int kXSlots = 3;
  static constexpr int kHt = 2 * N * 128;    // H~ pair: [head][N rows][128 B]
  static constexpr int kTabBufs = 4;
  static constexpr int kTabFloats = 4 * S;   // t[head][S] then e[head][S]
  static constexpr int kScal = 16;           // per head: 8 scalars (see below)
  static constexpr int kBars = 40;
  static constexpr int kBytes = 1024 + (kXSlots + 2) * kTile + kHt +
                                kTabBufs * (kTabFloats + kScal) * 4 + 16 + kBars * 8 + 32;
  // tensor memory columns
  static constexpr uint32_t kY = 0, kS = 128, kP = 256, kM = 384, kC = 448, kAlloc = 512;
  static_assert(kBytes <= 227 * 1024, "shared memory");
};
// per-head stage scalars: sfac = 2^(a_last - r), dec = 2^(a_last), hsc = 2^r,
// D, yw (1: this kernel writes the (chunk, head)'s y), hin (1: flagged, store
// the entering state)
enum : int { kScSfac = 0, kScDec, kScHsc, kScD, kScYw, kScHin };

enum : int {
  kFuXfull0 = 0, kFuXready0 = 3, kFuYstaged0 = 6, kFuXfree0 = 9,
  kFuCfull = 12, kFuCcopied, kFuBfull0, kFuBfull1, kFuBfree0, kFuBfree1,
  kFuSready, kFuSfree, kFuPready, kFuMready, kFuHready, kFuHfree, kFuYready, kFuYfree,
  kFuTabFull0, kFuTabEmpty0 = kFuTabFull0 + 4, kNumFuBars = kFuTabEmpty0 + 4
};
static_assert(kNumFuBars <= FusedHB::kBars, "barrier slots");

// FULL: the whole layer for items whole.. and split segments; otherwise the
// prepass of the split items' segments 0 .. nseg - 2 (final states, decays).
// HP: heads per item -- 2 (two 64-wide heads sharing one (B, C) group, their
// 128 columns side by side) or 1 (one 128-wide head, its two 64-column
// halves side by side; B and C of its own groups).  SPC: 128-token stages per
// chunk (2: 256-token chunks, 1: 128-token chunks); the flags, the flagged
// units' states and u are kept per chunk.
template <bool FULL, int HP, int SPC>
__global__ void __launch_bounds__(kFuThreads, 1)
    chunk_fused_hb(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapC, const __grid_constant__ CUtensorMap mapY,
                   const float *__restrict__ dt, const float *__restrict__ A,
                   const float *__restrict__ D, const float *__restrict__ h0,
                   float *__restrict__ h_final, __nv_bfloat16 *__restrict__ Hin,
                   uint8_t *__restrict__ flags, float *__restrict__ u, int64_t T, int H, int GB,
                   int GC, int nc, int softplus, int whole, int nseg, int cps, int64_t bh0,
                   float *__restrict__ Fseg, float *__restrict__ Lseg, int nsm) {
  using L = FusedHB;
  constexpr int S = L::S, N = L::N;
  constexpr int P = 128 / HP;  // the width of one head
  static_assert(HP == 1 || HP == 2, "heads per item");
  static_assert(SPC == 1 || SPC == 2, "stages per chunk");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *Xs = smem;                            // [slot][head][S rows][128 B]
  uint8_t *Cl = Xs + L::kXSlots * L::kTile;      // C landing [atom][S rows][128 B] (prepass: B slot 1)
  uint8_t *Bs = Cl + L::kTile;                   // B [atom][S rows][128 B]
  uint8_t *Ht = Bs + L::kTile;                   // H~ [head][N rows][128 B]
  float *tab = reinterpret_cast<float *>(Ht + L::kHt);  // [buf][t: head, S | e: head, S]
  float *scal = tab + L::kTabBufs * L::kTabFloats;       // [buf][head][8]
  uint8_t *ystore = reinterpret_cast<uint8_t *>(scal + L::kTabBufs * L::kScal);  // [slot][head]
  uint64_t *bars = reinterpret_cast<uint64_t *>(ystore + 16);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + L::kBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);

  const int ipb = (H + HP - 1) / HP;  // items per batch row
  const int cta = blockIdx.x;
  bool split;
  int item, seg;
  if (FULL) {
    split = cta >= whole;
    item = split ? whole + (cta - whole) / nseg : cta;
    seg = split ? (cta - whole) % nseg : 0;
  } else {
    split = true;
    item = whole + cta / (nseg - 1);
    seg = cta % (nseg - 1);
  }
  const int b = item / ipb;
  const int hb0 = HP * (item % ipb), nh = min(HP, H - hb0);
  const int gb = hb0 / (H / GB), gc = hb0 / (H / GC);  // the item's B and C groups
  const int c_begin = split ? seg * cps : 0;
  const int ncl = split ? min(nc, c_begin + cps) - c_begin : nc;
  const int nstages = SPC * ncl;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto stage_t0 = [&](int g) { return (SPC * c_begin + g) * S; };
  // column atom a (64 columns) of the item's 128: which head, which columns
  auto atom_head = [&](int a) { return HP == 2 ? hb0 + a : hb0; };
  auto atom_col = [&](int a) { return HP == 2 ? 0 : 64 * a; };
  const int natoms = HP == 2 ? nh : 2;

  if (tid == 0) {
    for (int i = 0; i < L::kBars; ++i) {
      const bool per_warp = (i >= kFuXready0 && i < kFuXready0 + 3) ||
                            (i >= kFuYstaged0 && i < kFuYstaged0 + 3) || i == kFuCcopied ||
                            i == kFuSfree || i == kFuMready || i == kFuHready || i == kFuYfree ||
                            (i >= kFuTabEmpty0 && i < kFuTabEmpty0 + 4);
      const bool tables = i >= kFuTabFull0 && i < kFuTabFull0 + 4;
      mbar_init(&bars[i], per_warp ? kFuCompute : tables ? 2 : 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kFuControl) tmem_alloc(tslot, L::kAlloc);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;
  // the launch after this one (the flagged heads, or the full pass after the
  // prepass) may start its set-up; it waits for this one's end before reading
  grid_dep_trigger();

  if (warp == kFuTables || warp == kFuTables + 1) {
    // ================================================================ tables
    // One head per warp (the second warp idles when an item has one head),
    // two stages at a time: lane owns 8 consecutive tokens (lanes 0-15 the
    // first stage, 16-31 the second); z = softplus(dt) A log2(e), running
    // sums, a scan within each half-warp.
    const int hh = warp - kFuTables;
    const bool mine = hh < nh;
    const int h = hb0 + min(hh, nh - 1);
    constexpr float kLog2e = 1.4426950408889634f;
    const float Ah = A[h] * kLog2e, Dh = D ? D[h] : 0.f;
    const int st = lane >> 4, sl = lane & 15;
    const int npair = (nstages + 1) / 2;
    float raw[8], rawn[8];
    auto fetch = [&](int lp, float (&rr)[8]) {
      const int64_t t0 = static_cast<int64_t>(stage_t0(2 * lp)) + lane * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        rr[e] = t0 + e < T ? dt[(static_cast<int64_t>(b) * T + t0 + e) * H + h] : 0.f;
    };
    float prod = 1.f;  // prepass: the segment's total decay
    if (npair > 0) fetch(0, rawn);
    for (int lp = 0; lp < npair; ++lp) {
      const int g0 = 2 * lp, gs = g0 + st;  // this half-warp's stage
      const bool have = gs < nstages;
      const int c = c_begin + gs / SPC;     // and its chunk
      const int64_t t0 = static_cast<int64_t>(stage_t0(g0)) + lane * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) raw[e] = rawn[e];
      if (lp + 1 < npair) fetch(lp + 1, rawn);
      float z[8], v[8];
      float run = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        z[e] = t0 + e < T ? (softplus ? softplus_f32(raw[e]) : raw[e]) * Ah : 0.f;
        run += z[e];
        v[e] = run;
      }
      float incl = run;
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if (sl >= off) incl += o;
      }
      const float base = incl - run;
      const float last0 = __shfl_sync(0xffffffffu, incl, 15);
      const float last1 = __shfl_sync(0xffffffffu, incl, 31);
      // the scaled form holds for a chunk when it holds for each of its stages
      const bool ok0 = scaled_form_ok(last0), ok1 = scaled_form_ok(last1);
      const bool fast = FULL && (SPC == 2 ? ok0 && ok1 : (st ? ok1 : ok0));
      const float a_last = st ? last1 : last0;
      const float r = fast ? scaled_form_ref(a_last) : a_last;
      bool ok = true;
      for (int s2 = 0; s2 < 2 && ok; ++s2) {
        const int g = g0 + s2;
        if (g >= L::kTabBufs)
          ok = mbar_wait(&bars[kFuTabEmpty0 + g % L::kTabBufs], ((g >> 2) - 1) & 1, abort_flag);
      }
      if (!ok) break;
      if (mine && have) {
        float *tb = tab + (gs % L::kTabBufs) * L::kTabFloats;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float av = v[e] + base;
          tb[hh * S + sl * 8 + e] = ex2_approx(r - av);
          tb[2 * S + hh * S + sl * 8 + e] = fast ? ex2_approx(av - r) : 0.f;
        }
        if (sl == 0) {
          float *sc = scal + (gs % L::kTabBufs) * L::kScal + hh * 8;
          sc[kScSfac] = ex2_approx(a_last - r);
          sc[kScDec] = ex2_approx(a_last);
          sc[kScHsc] = ex2_approx(r);
          sc[kScD] = Dh;
          sc[kScYw] = fast ? 1.f : 0.f;
          sc[kScHin] = fast ? 0.f : 1.f;
        }
        if (FULL) {
          if (sl == 0 && (SPC == 1 || st == 0))
            flags[(static_cast<int64_t>(b) * nc + c) * H + h] = fast ? 1 : 0;
          if (!fast) {  // the per-token log2 decays, for the per-head body
            float *uh = u + (static_cast<int64_t>(b) * H + h) * T;
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (t0 + e < T) uh[t0 + e] = z[e];
          }
        } else if (sl == 0) {
          prod *= ex2_approx(a_last);
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kFuTabFull0 + g0 % L::kTabBufs]);
        mbar_arrive(&bars[kFuTabFull0 + (g0 + 1) % L::kTabBufs]);
      }
    }
    // the prepass: the segment's total decay, the two half-warps' products
    prod *= __shfl_sync(0xffffffffu, prod, 16);
    if (!FULL && mine && lane == 0)
      Lseg[(static_cast<int64_t>(b) * H + h - bh0) * nseg + seg] = prod;
  } else if (warp == kFuControl) {
    // ================================================================ MMA issue, B and C loads
    if (lane == 0 && nstages > 0) {
      prefetch_tensormap(&mapB);
      if (FULL) prefetch_tensormap(&mapC);
      auto load_B = [&](int g) {
        const int k = FULL ? 0 : (g & 1);
        uint8_t *dst = FULL ? Bs : (k ? Cl : Bs);
        uint64_t *bar = &bars[kFuBfull0 + k];
        mbar_arrive_expect_tx(bar, L::kTile);
        tma_load_4d(dst, &mapB, bar, 0, gb, stage_t0(g), b);
        tma_load_4d(dst + S * 128, &mapB, bar, 64, gb, stage_t0(g), b);
      };
      auto load_C = [&](int g) {
        mbar_arrive_expect_tx(&bars[kFuCfull], L::kTile);
        tma_load_4d(Cl, &mapC, &bars[kFuCfull], 0, gc, stage_t0(g), b);
        tma_load_4d(Cl + S * 128, &mapC, &bars[kFuCfull], 64, gc, stage_t0(g), b);
      };
      load_B(0);
      if (FULL) load_C(0);
      else if (nstages > 1) load_B(1);
      constexpr uint32_t id_p = idesc_bf16(128, 128, false, false);  // C (TMEM) B^T (smem, K-major)
      // N = the item's 128 columns (two heads, or one 128-wide head)
      constexpr uint32_t id_s = idesc_bf16(128, 128, true, true);    // B^T (MN-major) x~ (MN-major)
      constexpr uint32_t id_y = idesc_bf16(128, 128, false, true);   // C or P (TMEM) H~ / x~ (MN-major)
      const uint32_t hs_ = smem_u32(Ht);
      for (int g = 0; g < nstages && !*abort_flag; ++g) {
        const int xk = g % L::kXSlots, bk = FULL ? 0 : (g & 1);
        const uint32_t xs = smem_u32(Xs + xk * L::kTile);
        const uint32_t bs = smem_u32(FULL ? Bs : (bk ? Cl : Bs));
        const uint32_t bpar = FULL ? (g & 1) : ((g >> 1) & 1);
        if (!mbar_wait(&bars[kFuBfull0 + bk], bpar, abort_flag)) break;
        if (FULL) {
          // ---- P = C B^T (C copied into tensor memory by the compute warps)
          if (!mbar_wait(&bars[kFuCcopied], g & 1, abort_flag)) break;
          tc_fence_after_sync();
#pragma unroll
          for (int ks = 0; ks < N / 16; ++ks) {
            const uint32_t koff = (ks >> 2) * S * 128 + (ks & 3) * 32;
            mma_bf16_tmem_a(tmem + L::kP, tmem + L::kC + 8 * ks, sdesc_sw128(bs + koff, 16, 1024),
                            id_p, ks > 0 ? 1u : 0u);
          }
          mma_commit(&bars[kFuPready]);
          if (g + 1 < nstages) load_C(g + 1);  // the landing slot was copied out
        }
        // ---- S = B^T x~
        if (!mbar_wait(&bars[kFuXready0 + xk], (g / L::kXSlots) & 1, abort_flag)) break;
        if (g > 0 && !mbar_wait(&bars[kFuSfree], (g - 1) & 1, abort_flag)) break;
        tc_fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < S / 16; ++ks)
          mma_bf16(tmem + L::kS, sdesc_sw128(bs + ks * 2048, S * 128, 1024),
                   sdesc_sw128(xs + ks * 2048, S * 128, 1024), id_s, ks > 0 ? 1u : 0u);
        mma_commit(&bars[kFuSready]);
        mma_commit(&bars[kFuBfree0 + bk]);
        if (!FULL) {
          mma_commit(&bars[kFuXfree0 + xk]);
          if (g + 2 < nstages) {
            if (!mbar_wait(&bars[kFuBfree0 + bk], (g >> 1) & 1, abort_flag)) break;
            load_B(g + 2);
          }
          continue;
        }
        // ---- Y = C H~ (after the epilogue has read the previous Y)
        if (!mbar_wait(&bars[kFuHready], g & 1, abort_flag)) break;
        if (g > 0 && !mbar_wait(&bars[kFuYfree], (g - 1) & 1, abort_flag)) break;
        tc_fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks)
          mma_bf16_tmem_a(tmem + L::kY, tmem + L::kC + 8 * ks,
                          sdesc_sw128(hs_ + ks * 2048, N * 128, 1024), id_y, ks > 0 ? 1u : 0u);
        mma_commit(&bars[kFuHfree]);
        // B is free once S and P are done: the next stage's B
        if (g + 1 < nstages) {
          if (!mbar_wait(&bars[kFuBfree0], g & 1, abort_flag)) break;
          load_B(g + 1);
        }
        // ---- Y += P x~
        if (!mbar_wait(&bars[kFuMready], g & 1, abort_flag)) break;
        tc_fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < S / 16; ++ks)
          mma_bf16_tmem_a(tmem + L::kY, tmem + L::kM + 8 * ks,
                          sdesc_sw128(xs + ks * 2048, S * 128, 1024), id_y, 1u);
        mma_commit(&bars[kFuYready]);
      }
    }
    __syncwarp();
  } else if (warp == kFuLoader) {
    // ================================================================ y out, x in
    if (lane == 0 && nstages > 0) {
      prefetch_tensormap(&mapX);
      if (FULL) prefetch_tensormap(&mapY);
      auto load_x = [&](int g) {
        const int xk = g % L::kXSlots;
        uint64_t *bar = &bars[kFuXfull0 + xk];
        mbar_arrive_expect_tx(bar, natoms * S * 128);
        for (int a = 0; a < natoms; ++a)
          tma_load_4d(Xs + xk * L::kTile + a * S * 128, &mapX, bar, atom_col(a), atom_head(a),
                      stage_t0(g), b);
      };
      // The whole item most likely to start on an SM next (CTAs start in
      // index order, one per SM, so about nsm after this one): its first two
      // stages of x and its h0 into L2, a few stages before this item ends.
      auto prefetch_next = [&]() {
        const int nxt = cta + nsm;
        if (!FULL || split || nxt >= whole) return;
        const int bn = nxt / ipb, hn = HP * (nxt % ipb), nhn = min(HP, H - hn);
        for (int gs = 0; gs < 2 && gs * S < T; ++gs)
          for (int a = 0; a < (HP == 2 ? nhn : 2); ++a)
            tma_prefetch_4d(&mapX, HP == 2 ? 0 : 64 * a, HP == 2 ? hn + a : hn, gs * S, bn);
        if (h0) {
          const float *src = h0 + (static_cast<int64_t>(bn) * H + hn) * N * P;
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                           reinterpret_cast<uint64_t>(src)),
                       "r"(static_cast<uint32_t>(nhn * N * P * 4))
                       : "memory");
        }
      };
      for (int g = 0; g < min(L::kXSlots, nstages); ++g) load_x(g);
      for (int g = 0; g < nstages; ++g) {
        const int xk = g % L::kXSlots;
        if (g == max(0, nstages - 4)) prefetch_next();
        const uint32_t par = (g / L::kXSlots) & 1;
        if (FULL) {
          if (!mbar_wait(&bars[kFuYstaged0 + xk], par, abort_flag) || *abort_flag) break;
          for (int a = 0; a < natoms; ++a)
            if (ystore[2 * xk + a])
              tma_store_4d(&mapY, Xs + xk * L::kTile + a * S * 128, atom_col(a), atom_head(a),
                           stage_t0(g), b);
          bulk_commit();
          bulk_wait_read0();  // the slot's y has been read
        } else if (!mbar_wait(&bars[kFuXfree0 + xk], par, abort_flag)) {
          break;
        }
        if (g + L::kXSlots < nstages) load_x(g + L::kXSlots);
      }
      bulk_wait_all();
    }
    __syncwarp();
  } else {
    // ================================================================ compute
    const int q = warp & 3, hs = warp >> 2;       // TMEM lane quarter; 32-column block
    // the block's 64-column atom and its columns inside it (shared memory),
    // its head (tables) and its first column inside that head (global memory)
    const int atom = hs >> 1, pa = 32 * (hs & 1);
    const int hh = HP == 2 ? atom : 0, p0 = HP == 2 ? pa : 32 * hs;
    const int n = 32 * q + lane;                  // state row (S), token row (Y, P)
    const bool valid = hh < nh;
    const int h = hb0 + min(hh, nh - 1);
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const int64_t rel = static_cast<int64_t>(b) * H + h - bh0;  // split rows only
    bool ok = nstages > 0;
    float st[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) st[e] = 0.f;
    // The item's state moves between global memory and the threads' rows
    // through the H~ buffer (idle before the first stage and after the
    // last): one 64-column half of the item's 128 columns (a head of a pair,
    // or half of a wide head) at a time, fully coalesced on the global side,
    // 16-byte chunks XOR-swizzled by row on the shared side; round r serves
    // the warps whose columns lie in that half (hs / 2 == r).
    float *stage_f = reinterpret_cast<float *>(Ht);  // [128 rows][64 floats]
    auto half_base = [&](float *base, int r) {       // the half's [128][64] block
      return HP == 2 ? base + ((static_cast<int64_t>(b) * H + hb0 + r) * N) * P
                     : base + (static_cast<int64_t>(b) * H + hb0) * N * P + 64 * r;
    };
    const int nhalves = HP == 2 ? nh : 2;
    // both halves' global loads are issued first (one memory latency): the
    // first half lands in ta, the second in st[16..31], whose owners fill st
    // last; the first half's owners park their row's second 16 floats in ta
    auto load_state_staged = [&](const float *base) {
      float ta[16];
      auto gload = [&](int r, float *dst) {
        const float *src = half_base(const_cast<float *>(base), r);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int f = i * 32 * kFuCompute + tid, row = f >> 4, c = f & 15;
          const float4 v = *reinterpret_cast<const float4 *>(src + static_cast<int64_t>(row) * P + 4 * c);
          dst[4 * i] = v.x; dst[4 * i + 1] = v.y; dst[4 * i + 2] = v.z; dst[4 * i + 3] = v.w;
        }
      };
      auto sstore = [&](const float *src) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int f = i * 32 * kFuCompute + tid, row = f >> 4, c = f & 15;
          *reinterpret_cast<float4 *>(stage_f + row * 64 + 4 * (c ^ (row & 7))) =
              make_float4(src[4 * i], src[4 * i + 1], src[4 * i + 2], src[4 * i + 3]);
        }
      };
      // own row, 16-byte chunks j0 .. j0 + 3 of the thread's eight, into dst
      auto sread = [&](int j0, float *dst) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = 8 * (hs & 1) + j0 + j;
          const float4 v = *reinterpret_cast<const float4 *>(stage_f + n * 64 + 4 * (c ^ (n & 7)));
          dst[4 * j] = v.x; dst[4 * j + 1] = v.y; dst[4 * j + 2] = v.z; dst[4 * j + 3] = v.w;
        }
      };
      gload(0, ta);
      if (nhalves > 1) gload(1, st + 16);
      sstore(ta);
      compute_bar_sync();
      if ((hs >> 1) == 0) {
        sread(0, st);
        sread(4, ta);
      }
      compute_bar_sync();
      if (nhalves > 1) {
        sstore(st + 16);
        compute_bar_sync();
        if ((hs >> 1) == 1) {
          sread(0, st);
          sread(4, st + 16);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) st[16 + e] = ta[e];
        }
        compute_bar_sync();  // every row read before the first H~ is written
      } else if ((hs >> 1) == 0) {
#pragma unroll
        for (int e = 0; e < 16; ++e) st[16 + e] = ta[e];
      }
    };
    // half(r): the global [128][64] block of round r (row stride P)
    auto store_state_staged = [&](auto half, bool write) {
#pragma unroll 1
      for (int r = 0; r < nhalves; ++r) {
        float *dst = half(r);
        compute_bar_sync();  // the buffer is free
        if ((hs >> 1) == r) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int c = 8 * (hs & 1) + j;
            *reinterpret_cast<float4 *>(stage_f + n * 64 + 4 * (c ^ (n & 7))) =
                make_float4(st[4 * j], st[4 * j + 1], st[4 * j + 2], st[4 * j + 3]);
          }
        }
        compute_bar_sync();
        if (write) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int f = i * 32 * kFuCompute + tid, row = f >> 4, c = f & 15;
            *reinterpret_cast<float4 *>(dst + static_cast<int64_t>(row) * P + 4 * c) =
                *reinterpret_cast<const float4 *>(stage_f + row * 64 + 4 * (c ^ (row & 7)));
          }
        }
      }
    };
    if (seg == 0 && h0) {
      load_state_staged(h0);
    } else if (FULL && split && seg > 0 && valid) {
      // the true entering state from the prepass: T = Lambda T + F over s' < seg
      // (a thread's 32 columns of a state row, one 128-byte line, at a time)
      grid_dep_wait();
      for (int s2 = 0; s2 < seg; ++s2) {
        const float Ls = Lseg[rel * nseg + s2];
        float v[32];
        ld_row32(Fseg + (rel * nseg + s2) * N * P + static_cast<int64_t>(n) * P + p0, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) st[e] = fmaf(Ls, st[e], v[e]);
      }
    }
    // a wait for the whole warp: every lane waits on the same phase, so they
    // agree unless one ran out of time (which sets the abort flag for all)
    auto wait_all = [&](uint64_t *bar, uint32_t par) -> bool {
      const bool w = mbar_wait(bar, par, abort_flag);
      return __all_sync(0xffffffffu, w);
    };
    auto tables_ready = [&](int g) {
      return wait_all(&bars[kFuTabFull0 + g % L::kTabBufs], (g >> 2) & 1);
    };
    auto sc_of = [&](int g) { return scal + (g % L::kTabBufs) * L::kScal + min(hh, nh - 1) * 8; };
    // stage g's x rows *= t_j in place (16-byte chunks, four per thread)
    auto scale = [&](int g) -> bool {
      const int xk = g % L::kXSlots;
      // (the full pass calls it right after enter(g), which waited for the tables)
      if ((!FULL && !tables_ready(g)) || !wait_all(&bars[kFuXfull0 + xk], (g / L::kXSlots) & 1))
        return false;
      const float *tb = tab + (g % L::kTabBufs) * L::kTabFloats;
      uint8_t *xb = Xs + xk * L::kTile;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int uu = tid + kFuCompute * 32 * m;
        const int x_h = uu >> 10, j = (uu >> 3) & (S - 1), cc = uu & 7;
        uint4 *ptr = reinterpret_cast<uint4 *>(xb + x_h * S * 128 + sw128_offset(j, 8 * cc));
        const float t = tb[(HP == 2 ? x_h : 0) * S + j];
        *ptr = scale_bf16x8(*ptr, t);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kFuXready0 + xk]);
      return true;
    };
    // the entering state of stage g: H~ = bf16(2^r state) for the C H~ MMA,
    // the stage's C copied into tensor memory, and, at a flagged chunk's
    // start, the unscaled state for the per-head body
    auto enter = [&](int g) -> bool {
      if (!tables_ready(g) || !wait_all(&bars[kFuCfull], g & 1)) return false;
      const float *sc = sc_of(g);
      const float f = sc[kScHsc];
      uint8_t *hrow = Ht + atom * N * 128;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t w4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          w4[i] = pack_bf16x2(f * st[8 * k + 2 * i], f * st[8 * k + 2 * i + 1]);
        *reinterpret_cast<uint4 *>(hrow + sw128_offset(n, pa + 8 * k)) =
            make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      if (g % SPC == 0 && valid && sc[kScHin] != 0.f) {  // a flagged chunk's start
        __nv_bfloat16 *dst =
            Hin + (((static_cast<int64_t>(b) * nc + c_begin + g / SPC) * H + h) * N + n) * P + p0;
#pragma unroll
        for (int e = 0; e < 32; e += 16) {
          uint32_t w8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) w8[k] = pack_bf16x2(st[e + 2 * k], st[e + 2 * k + 1]);
          st_global_v8(dst + e, w8);
        }
      }
      // C rows n, state columns 32 hs .. + 31 (atom hs / 2) -> tensor memory
      uint32_t cw[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 cv = *reinterpret_cast<const uint4 *>(
            Cl + (hs >> 1) * S * 128 + sw128_offset(n, 32 * (hs & 1) + 8 * k));
        cw[4 * k] = cv.x; cw[4 * k + 1] = cv.y; cw[4 * k + 2] = cv.z; cw[4 * k + 3] = cv.w;
      }
      tmem_st16_u32(tmem + lane_base + L::kC + 16 * hs, cw);
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kFuHready]);
        mbar_arrive(&bars[kFuCcopied]);
      }
      return true;
    };
    // P of stage g -> masked bf16 pairs (j <= i) in tensor memory.  The full
    // pass waits for S instead: its commit follows P's MMAs (same thread, in
    // order), so one wait covers mask and fold
    auto mask = [&](int g) -> bool {
      if (!wait_all(&bars[FULL ? kFuSready : kFuPready], g & 1)) return false;
      // (row quarter q, column block hs): below the diagonal block (q > hs)
      // nothing is masked, on it (q == hs) columns j <= i are kept, and above
      // it (q < hs) the block stays zero from the start
      if (q >= hs) {
        tc_fence_after_sync();
        float v[32];
        uint32_t pk[16];
        tmem_ld32(tmem + lane_base + L::kP + 32 * hs, v);
        if (q > hs) {
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(v[2 * e], v[2 * e + 1]);
        } else {
          hb_mask_pack(v, lane, pk);
        }
        tmem_st16_u32(tmem + lane_base + L::kM + 16 * hs, pk);
        tmem_st_wait();
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kFuMready]);
      return true;
    };
    // state <- dec state + sfac S (stage g's S; the full pass has waited in mask)
    auto fold = [&](int g) -> bool {
      if (!FULL && !wait_all(&bars[kFuSready], g & 1)) return false;
      tc_fence_after_sync();
      float sv[32];
      tmem_ld32(tmem + lane_base + L::kS + 32 * hs, sv);
      const float *sc = sc_of(g);
      const float dec = sc[kScDec], sf = sc[kScSfac];
#pragma unroll
      for (int e = 0; e < 32; ++e) st[e] = fmaf(dec, st[e], sf * sv[e]);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kFuSfree]);
      return true;
    };
    // y rows of stage g = 2^(a_i - r) (Y + D x~) -> bf16 in place of x~ in
    // the stage's slot, for the loader's TMA store
    auto epilogue = [&](int g) -> bool {
      if (!wait_all(&bars[kFuYready], g & 1)) return false;
      tc_fence_after_sync();
      const int xk = g % L::kXSlots;
      const float *sc = sc_of(g);
      const bool yw = valid && sc[kScYw] != 0.f;
      if (yw) {
        const float f = tab[(g % L::kTabBufs) * L::kTabFloats + 2 * S + hh * S + n];
        const float d = sc[kScD];
        uint8_t *xrow = Xs + xk * L::kTile + atom * S * 128;
        float v32[32];
        tmem_ld32(tmem + lane_base + L::kY + 32 * hs, v32);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const float *v = v32 + 16 * half;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            uint4 *ptr =
                reinterpret_cast<uint4 *>(xrow + sw128_offset(n, pa + 16 * half + 8 * k));
            const uint4 xv = *ptr;
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float2 xf = unpack_bf16x2(xw[i]);
              o[i] = pack_bf16x2(f * fmaf(d, xf.x, v[8 * k + 2 * i]),
                                 f * fmaf(d, xf.y, v[8 * k + 2 * i + 1]));
            }
            *ptr = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
      if (warp == 0 && lane < 2) {  // which atoms' y the loader stores
        const float *s0 = scal + (g % L::kTabBufs) * L::kScal;
        ystore[2 * xk + lane] = lane < natoms && s0[8 * (HP == 2 ? lane : 0) + kScYw] != 0.f;
      }
      tc_fence_before_sync();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kFuYfree]);
        mbar_arrive(&bars[kFuYstaged0 + xk]);
        mbar_arrive(&bars[kFuTabEmpty0 + g % L::kTabBufs]);
      }
      return true;
    };

    if (FULL) {
      if (q < hs) {  // the masked C B^T's blocks above the diagonal: zero throughout
        const uint32_t z[16] = {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0};
        tmem_st16_u32(tmem + lane_base + L::kM + 16 * hs, z);
        tmem_st_wait();
      }
      ok = ok && enter(0) && scale(0);
      for (int g = 0; g < nstages && ok; ++g) {
        if (g > 0 && !(ok = epilogue(g - 1))) break;
        if (!(ok = mask(g))) break;
        if (!(ok = fold(g))) break;
        if (g + 1 < nstages) {
          if (!(ok = wait_all(&bars[kFuHfree], g & 1))) break;  // C H~ of stage g is done
          if (!(ok = enter(g + 1) && scale(g + 1))) break;
        }
      }
      if (ok) ok = epilogue(nstages - 1);
    } else {
      ok = ok && scale(0);
      for (int g = 0; g < nstages && ok; ++g) {
        if (!(ok = fold(g))) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kFuTabEmpty0 + g % L::kTabBufs]);
        if (g + 1 < nstages && !(ok = scale(g + 1))) break;
      }
    }
    // the final state: the sequence's (whole items, last segments) or, in the
    // prepass, the segment's from its own start (the H~ buffer is free once
    // the last C H~ product is done)
    if (FULL && nstages > 0) ok = ok && wait_all(&bars[kFuHfree], (nstages - 1) & 1);
    if (!FULL) {  // segment states: [(row - bh0) nseg + seg][N][P]
      store_state_staged(
          [&](int r) {
            const int64_t row = static_cast<int64_t>(b) * H + hb0 + (HP == 2 ? r : 0) - bh0;
            return Fseg + (row * nseg + seg) * N * P + (HP == 2 ? 0 : 64 * r);
          },
          ok);
    } else if (h_final && (!split || seg == nseg - 1)) {
      store_state_staged([&](int r) { return half_base(h_final, r); }, ok);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kFuControl) tmem_dealloc(tmem, L::kAlloc);
}

// The (chunk, head) units the one-pass kernel left to the per-head chunk-scan
// body (their decay falls outside its scaled form's range): one block per
// (head set, chunk, batch row) -- set r of `sets` holds heads r, r + sets,
// ... -- computing the set's flagged heads; a block with none leaves before
// any set-up (usually all of them: such chunks are rare).
template <int Q, int P>
__global__ void __launch_bounds__(kScanThreads, 1)
    chunk_scan_flagged(const __grid_constant__ CUtensorMap mapC32,
                       const __grid_constant__ CUtensorMap mapB,
                       const __grid_constant__ CUtensorMap mapX,
                       const __grid_constant__ CUtensorMap mapH,
                       const __grid_constant__ CUtensorMap mapY, const float *__restrict__ dt,
                       const float *__restrict__ A, const float *__restrict__ D,
                       const float *__restrict__ u, const uint8_t *__restrict__ flags, int64_t T,
                       int H, int GB, int GC, int nc, int sets, int softplus) {
  grid_dep_wait();  // the flags, u and the states of the one-pass kernel
  const int64_t j = blockIdx.x;
  const int set = static_cast<int>(j % sets), c = static_cast<int>((j / sets) % nc);
  const int bb = static_cast<int>(j / (static_cast<int64_t>(sets) * nc));
  int any = 0;
  for (int h = set + static_cast<int>(threadIdx.x) * sets; h < H;
       h += static_cast<int>(blockDim.x) * sets)
    any |= flags[(static_cast<int64_t>(bb) * nc + c) * H + h] == 0;
  if (!__syncthreads_or(any)) return;
  scan_hl_body<Q, P, true>(set, c, bb, mapC32, mapB, mapX, mapH, mapY, dt, A, D, T, H, GB, GC, nc,
                           sets, softplus, flags, u);
}

}  // namespace ssd
