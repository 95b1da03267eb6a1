// ssd_state_hb.cuh -- chunk states and state passing for 256-token chunks,
// 64-wide heads and one B group, two heads per MMA.
//
// Same result as chunk_state_pass_tc (ssd_state.cuh): for one (batch b, head
// pair) and every chunk c in order, with a = cs * log2(e) the in-chunk
// inclusive running sum of softplus(dt) * A_h in log2 units (summed here from
// u = softplus(dt) * A * log2(e), written by dt_decay_kernel),
//   S_c   = B_c^T diag(w) x_c,     w_j = 2^(a_last - a_j)             (green step)
//   Hin_c = state entering chunk c                                   (stored, bf16)
//   state = 2^(a_last) * state + S_c                                 (yellow step)
// (Mamba-2 page, section "SSD算法": the chunk-final states by batched matmul
// and the scan over chunks with the chunk decays).  The running state starts
// at h0 (or zero) and its last value is h_final; sequence segments and their
// hand-off (Fseg, Lseg, Dc) work as in chunk_state_pass_tc.
//
// Items.  Item i is (batch i / npairs, head pair i % npairs).  The first
// `whole` CTAs take items 0 .. whole - 1 over the whole sequence; the CTAs
// after them take the remaining items in `nseg` segments of `cps` chunks
// each (CTA whole + k nseg + s: item whole + k, segment s).  The host splits
// only the items of a last, partly filled wave, so that wave ends as soon as
// the full ones; the hand-off arrays then cover the split items' heads alone,
// indexed from the first of them (bh0 = its b H + h).
//
// Schedule.  B is the A operand of every head's MMA, so two heads share one
// MMA chain (N = 2 x 64).  Each chunk arrives as two 128-token stages (the B
// half and both heads' x halves, 64 KB) through a ring of three shared-memory
// slots, loaded 1.5 chunks ahead; the compute warps scale a stage's x rows
// by w_j in place and the control warp's MMAs for it run while the next
// stage is scaled.  The two chunk accumulators alternate in tensor memory:
// chunk c + 1 accumulates while the compute warps fold chunk c into the
// running state (registers: thread = one state row, 32 columns of one head).
// A table warp computes each chunk's decays up to two chunks ahead.
//
// With `flags` (the head-pair chunk scan follows), the (batch, chunk, head)
// decay-range flags of that scan are recorded here too -- 1 when
// a_last >= -kScaledRangeMax -- and each flagged-1 chunk state is stored
// multiplied by 2^r, r = scaled_form_ref(a_last), the factor the scan's
// scaled form applies to it (ssd_tc.cuh); the per-chunk decay products Dc of a
// split item carry the same factor, so the fix-up keeps it.
//
// Warp roles: warps 0-15 scale x, fold states and store chunk states (four
// per TMEM lane quarter); warp 16 (one lane) issues every TMA load and MMA;
// warps 17 and 18 compute the tables, one head each.  Every wait is bounded
// in time.
#pragma once

#include "ssd_state.cuh"

namespace ssd {

constexpr int kShWarps = 19;  // 16 compute + control + two table warps
constexpr int kShThreads = 32 * kShWarps;
constexpr int kShCompute = 16;
constexpr int kShControl = 16;
constexpr int kShTables = 17;

struct StateHB {
  static constexpr int Q = 256, P = 64, N = kTcN, HALF = Q / 2;
  static constexpr int kStage = N * HALF * 2 + 2 * P * HALF * 2;  // B half + x pair half
  static constexpr int kSlots = 3;
  static constexpr int kTabBufs = 3;
  static constexpr int kTab = 2 * Q;  // per buffer: w_j for the two heads
  static constexpr int kFloats = kTabBufs * (kTab + 4);  // + the two chunk decays and state factors
  static constexpr int kBars = 20;
  static constexpr int kBytes = kSlots * kStage + kFloats * 4 + kBars * 8 + 16 + 1024;
  static constexpr uint32_t kAlloc = 256;  // two chunk accumulators of 128 columns
  static_assert(kBytes <= 227 * 1024, "shared memory");
};

enum : int {
  kShFull0 = 0, kShFull1, kShFull2, kShEmpty0, kShEmpty1, kShEmpty2, kShScaled0, kShScaled1,
  kShScaled2, kShAccFull0, kShAccFull1, kShAccFree0, kShAccFree1, kShTabFull0, kShTabFull1,
  kShTabFull2, kShTabEmpty0, kShTabEmpty1, kShTabEmpty2, kNumShBars
};
static_assert(kNumShBars <= StateHB::kBars, "barrier slots");

__global__ void __launch_bounds__(kShThreads, 1)
    chunk_state_hb(const __grid_constant__ CUtensorMap mapB128,
                   const __grid_constant__ CUtensorMap mapX128, const float *__restrict__ u,
                   const float *__restrict__ h0, __nv_bfloat16 *__restrict__ Hin,
                   float *__restrict__ h_final, int64_t T, int H, int nc, int whole, int nseg,
                   int cps, int64_t bh0, float *__restrict__ Fseg,
                   float *__restrict__ Lseg, float *__restrict__ Dc,
                   uint8_t *__restrict__ flags) {
  using L = StateHB;
  constexpr int Q = L::Q, P = L::P, N = L::N, HALF = L::HALF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  // slot s: [B state cols 0-63 | B cols 64-127 | x head 0 | x head 1], each [HALF rows][128 B]
  uint8_t *slots = smem;
  // tables of chunk lc in buffer lc % 3: [buf][head][Q] w_j, [buf][head] decay
  float *tab = reinterpret_cast<float *>(slots + L::kSlots * L::kStage);
  float *dec = tab + L::kTabBufs * L::kTab;  // [buf][head] chunk decay 2^a_last
  float *hsc = dec + 2 * L::kTabBufs;        // [buf][head] factor of the stored chunk state
  uint64_t *bars = reinterpret_cast<uint64_t *>(hsc + 2 * L::kTabBufs);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + L::kBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);

  const int npairs = (H + 1) / 2;
  const int cta = blockIdx.x;
  const bool split = cta >= whole;  // a segment of a split item
  const int item = split ? whole + (cta - whole) / nseg : cta;
  const int seg = split ? (cta - whole) % nseg : 0;
  const int b = item / npairs, pair = item % npairs;
  const int hb0 = 2 * pair, nh = min(2, H - hb0);  // the CTA's heads hb0, hb0 + 1
  const int c_begin = split ? seg * cps : 0;
  const int ncl = split ? min(nc, c_begin + cps) - c_begin : nc;
  const int nstages = 2 * ncl;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < L::kBars; ++i) {
      const bool per_warp = (i >= kShScaled0 && i <= kShScaled2) || i == kShAccFree0 ||
                            i == kShAccFree1 || (i >= kShTabEmpty0 && i <= kShTabEmpty2);
      const bool tables = i >= kShTabFull0 && i <= kShTabFull2;
      mbar_init(&bars[i], per_warp ? kShCompute : tables ? 2 : 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kShControl) tmem_alloc(tslot, L::kAlloc);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;
  // the kernels after this one may start their set-up (they wait for its end)
  grid_dep_trigger();

  if (warp >= kShTables) {
    // ================================================================ tables
    // Head hh = warp - kShTables: chunk lc's w_j = 2^(a_last - a_j) and decay
    // 2^(a_last) into buffer lc % 3 (lane owns Q/32 consecutive tokens of the
    // per-token log2 decays u; running sum, then a warp scan); the next
    // chunk's u is fetched first.
    constexpr int PER = Q / 32;
    const int hh = warp - kShTables;
    const bool mine = hh < nh;
    const int h = hb0 + min(hh, nh - 1);
    const float *uh = u + (static_cast<int64_t>(b) * H + h) * T;
    float z[PER], zn[PER];
    float prod = 1.f;  // decays of this segment's chunks so far
    auto fetch = [&](int lc, float (&zz)[PER]) {
      const int64_t t0 = static_cast<int64_t>(c_begin + lc) * Q + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) zz[e] = t0 + e < T ? uh[t0 + e] : 0.f;
    };
    grid_dep_wait();  // u comes from dt_decay_kernel, which may still be running
    if (ncl > 0 && mine) fetch(0, zn);
    for (int lc = 0; lc < ncl; ++lc) {
      const int s = lc % L::kTabBufs, c = c_begin + lc;
#pragma unroll
      for (int e = 0; e < PER; ++e) z[e] = zn[e];
      if (mine && lc + 1 < ncl) fetch(lc + 1, zn);
      if (lc >= L::kTabBufs &&
          !mbar_wait(&bars[kShTabEmpty0 + s], ((lc - L::kTabBufs) / L::kTabBufs) & 1, abort_flag))
        break;
      if (mine) {
        float v[PER];
        float run = 0.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
          run += z[e];  // 0 past T
          v[e] = run;
        }
        float incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float o = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += o;
        }
        const float base = incl - run;
        const float a_last = __shfl_sync(0xffffffffu, v[PER - 1] + base, 31);
        float *tw = tab + s * L::kTab + hh * Q;
#pragma unroll
        for (int e = 0; e < PER; ++e) tw[lane * PER + e] = ex2_approx(a_last - (v[e] + base));
        if (lane == 0) {
          const float decay = ex2_approx(a_last);
          const bool scaled = flags && scaled_form_ok(a_last);
          const float f = scaled ? ex2_approx(scaled_form_ref(a_last)) : 1.f;
          dec[2 * s + hh] = decay;
          hsc[2 * s + hh] = f;
          const int64_t rel = static_cast<int64_t>(b) * H + h - bh0;  // split items only
          if (flags) flags[(static_cast<int64_t>(b) * nc + c) * H + h] = scaled;
          if (split) Dc[rel * nc + c] = prod * f;
          prod *= decay;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kShTabFull0 + s]);
    }
    if (mine && lane == 0 && split)
      Lseg[(static_cast<int64_t>(b) * H + h - bh0) * nseg + seg] = prod;
  } else if (warp == kShControl) {
    // ================================================================ control
    if (lane == 0 && nstages > 0) {
      prefetch_tensormap(&mapB128);
      prefetch_tensormap(&mapX128);
      // stage g: half g & 1 of local chunk g >> 1, in slot g % 3
      auto load_stage = [&](int g) {
        const int sl = g % L::kSlots;
        const int t0 = (c_begin + (g >> 1)) * Q + (g & 1) * HALF;
        uint8_t *base = slots + sl * L::kStage;
        uint64_t *bar = &bars[kShFull0 + sl];
        mbar_arrive_expect_tx(bar, N * HALF * 2 + nh * P * HALF * 2);
#pragma unroll
        for (int a = 0; a < N / 64; ++a)
          tma_load_4d(base + a * HALF * 128, &mapB128, bar, 64 * a, 0, t0, b);
        for (int hh = 0; hh < nh; ++hh)
          tma_load_4d(base + (2 + hh) * HALF * 128, &mapX128, bar, 0, hb0 + hh, t0, b);
      };
      for (int g = 0; g < min(L::kSlots, nstages); ++g) load_stage(g);
      constexpr uint32_t idesc = idesc_bf16(128, 2 * P, true, true);
      for (int g = 0; g < nstages && !*abort_flag; ++g) {
        const int sl = g % L::kSlots, lc = g >> 1, half = g & 1;
        // the previous stage's slot takes stage g + 2 once its MMAs are done
        if (g >= 1 && g + 2 < nstages) {
          if (!mbar_wait(&bars[kShEmpty0 + (g - 1) % L::kSlots], ((g - 1) / L::kSlots) & 1,
                         abort_flag))
            break;
          load_stage(g + 2);
        }
        // chunk lc's accumulator is free once chunk lc - 2 has been folded
        if (half == 0 && lc >= 2 &&
            !mbar_wait(&bars[kShAccFree0 + (lc & 1)], ((lc - 2) >> 1) & 1, abort_flag))
          break;
        if (!mbar_wait(&bars[kShScaled0 + sl], (g / L::kSlots) & 1, abort_flag)) break;
        tc_fence_after_sync();
        const uint32_t bb = smem_u32(slots + sl * L::kStage), xb = bb + 2 * HALF * 128;
        // S (+)= B_half^T [x~_h | x~_h']: M = 128 state rows (two 64-row atoms
        // HALF * 128 bytes apart), N = 128 (two heads, the same), K = 128 tokens
#pragma unroll
        for (int ks = 0; ks < HALF / 16; ++ks)
          mma_bf16(tmem + 128 * (lc & 1), sdesc_sw128(bb + ks * 2048, HALF * 128, 1024),
                   sdesc_sw128(xb + ks * 2048, HALF * 128, 1024), idesc,
                   (half > 0 || ks > 0) ? 1u : 0u);
        mma_commit(&bars[kShEmpty0 + sl]);
        if (half == 1) mma_commit(&bars[kShAccFull0 + (lc & 1)]);
      }
    }
    __syncwarp();
  } else if (warp < kShCompute) {
    // ================================================================ compute
    const int q = warp & 3, hs = warp >> 2;  // TMEM lane quarter; 32-column block
    const int hh = hs >> 1, p0 = 32 * (hs & 1);  // this thread's head and first column
    const int n = 32 * q + lane;                 // state row
    const bool valid = hh < nh;
    const int h = hb0 + min(hh, nh - 1);
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    float st[32];
    const int64_t srow = ((static_cast<int64_t>(b) * H + h) * N + n) * P + p0;
    if (h0 && seg == 0 && valid) {
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 v = *reinterpret_cast<const float4 *>(h0 + srow + e);
        st[e] = v.x; st[e + 1] = v.y; st[e + 2] = v.z; st[e + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) st[e] = 0.f;
    }
    // stage g's x rows *= w_j in place (16-byte chunks, four per thread)
    auto scale = [&](int g) -> bool {
      const int sl = g % L::kSlots, lc = g >> 1, half = g & 1;
      bool w = mbar_wait(&bars[kShFull0 + sl], (g / L::kSlots) & 1, abort_flag);
      if (!(__all_sync(0xffffffffu, w) && !*abort_flag)) return false;
      const float *tw = tab + (lc % L::kTabBufs) * L::kTab + half * HALF;
      uint8_t *xb = slots + sl * L::kStage + 2 * HALF * 128;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int u = tid + kShCompute * 32 * m;
        const int x_h = u >> 10, j = (u >> 3) & (HALF - 1), cc = u & 7;
        uint4 *ptr = reinterpret_cast<uint4 *>(xb + x_h * HALF * 128 + sw128_offset(j, 8 * cc));
        *ptr = scale_bf16x8(*ptr, tw[x_h * Q + j]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kShScaled0 + sl]);
      return true;
    };
    auto tables_ready = [&](int lc) -> bool {
      bool w = mbar_wait(&bars[kShTabFull0 + lc % L::kTabBufs], (lc / L::kTabBufs) & 1, abort_flag);
      return __all_sync(0xffffffffu, w) && !*abort_flag;
    };
    // the state entering local chunk lc -> Hin (bf16), times the scan's factor;
    // issued right after the fold that produced it, so that the stores drain
    // while the next chunk's x is scaled (tables of lc are ready)
    auto store_hin = [&](int lc) {
      if (!valid) return;
      const float f = hsc[2 * (lc % L::kTabBufs) + hh];
      __nv_bfloat16 *dst =
          Hin + (((static_cast<int64_t>(b) * nc + c_begin + lc) * H + h) * N + n) * P + p0;
#pragma unroll
      for (int e = 0; e < 32; e += 16) {
        uint32_t v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = pack_bf16x2(f * st[e + 2 * k], f * st[e + 2 * k + 1]);
        st_global_v8(dst + e, v);  // 32-byte aligned: row n, columns p0 + e
      }
    };
    bool ok = ncl > 0 && tables_ready(0);
    if (ok) store_hin(0);
    ok = ok && scale(0) && scale(1);
    for (int lc = 0; lc < ncl && ok; ++lc) {
      // the next chunk's x first, so that its MMAs queue behind this chunk's
      if (lc + 1 < ncl && !(ok = tables_ready(lc + 1) && scale(2 * lc + 2) && scale(2 * lc + 3)))
        break;
      // fold local chunk lc: state = decay * state + S_c
      bool w = mbar_wait(&bars[kShAccFull0 + (lc & 1)], (lc >> 1) & 1, abort_flag);
      if (!(ok = __all_sync(0xffffffffu, w) && !*abort_flag)) break;
      tc_fence_after_sync();
      float sv[32];
      tmem_ld32(tmem + lane_base + 128 * (lc & 1) + 32 * hs, sv);
      const float decay = dec[2 * (lc % L::kTabBufs) + min(hh, nh - 1)];
#pragma unroll
      for (int e = 0; e < 32; ++e) st[e] = fmaf(decay, st[e], sv[e]);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[kShAccFree0 + (lc & 1)]);
        mbar_arrive(&bars[kShTabEmpty0 + lc % L::kTabBufs]);
      }
      if (lc + 1 < ncl) store_hin(lc + 1);
    }
    // the sequence's final state, or this segment's (from its own start state)
    if (ok && valid && (split || h_final)) {
      float *fin = !split ? h_final + srow
                          : Fseg + ((static_cast<int64_t>(b) * H + h - bh0) * nseg + seg) * N * P +
                                static_cast<int64_t>(n) * P + p0;
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4 *>(fin + e) = make_float4(st[e], st[e + 1], st[e + 2], st[e + 3]);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kShControl) tmem_dealloc(tmem, L::kAlloc);
}

// ----------------------------------------------------------------------------
// dt -> per-token log2 decays for the head-pair kernels:
//   u[b, h, t] = softplus(dt[b, t, h]) * A_h * log2(e)
// (the modified A factors of the Mamba-2 page, section "SSD算法", in log2
// units), written with each head's tokens contiguous so that a table warp
// reads a chunk of one head in 1 KB.  A 32-token x 32-head tile per block
// through shared memory (reads coalesced over heads, writes over tokens).
// (A tile of 32 tokens x all heads per block, one wave of 512 blocks at the
// 2.7B shape, measured slower: 10.4 against 8.7 us.)
// grid (ceil(T / 32), ceil(H / 32), batch), 256 threads.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) dt_decay_kernel(const float *__restrict__ dt,
                                                       const float *__restrict__ A,
                                                       float *__restrict__ u, int64_t T, int H,
                                                       int softplus) {
  __shared__ float tile[32][33];
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * 32;
  const int h0 = blockIdx.y * 32, b = blockIdx.z;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  constexpr float kLog2e = 1.4426950408889634f;
  grid_dep_trigger();  // the chunk-state kernel may start loading x and B
  const int h = h0 + tx;
  float z[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {  // every load first, so that the four are in flight at once
    const int64_t t = t0 + ty + 8 * k;
    z[k] = t < T && h < H ? dt[(static_cast<int64_t>(b) * T + t) * H + h] : 0.f;
  }
  const float Ah = h < H ? A[h] : 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = ty + 8 * k;
    tile[r][tx] = t0 + r < T && h < H ? (softplus ? softplus_f32(z[k]) : z[k]) * Ah * kLog2e : 0.f;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int r = ty + 8 * k;
    const int h = h0 + r;
    const int64_t t = t0 + tx;
    if (h < H && t < T) u[(static_cast<int64_t>(b) * H + h) * T + t] = tile[tx][r];
  }
}

}  // namespace ssd
