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
// Kernels: cp_tile_decay_kernel and cp_tile_prefix_kernel (a_t as a scan
// within 128-token tiles plus the sum of the tiles before; Lambda = 2^(sum of
// all tiles)),
// cp_combine_kernel (H_in(r) and h_final,
// elementwise over the states), cp_correct_tc (the C H_in product on the
// tensor cores, bf16 C with N = 128 and P in {64, 128}) or cp_correct_simt
// (every other shape, float32 CUDA cores).
#pragma once

#include "ssd_tc.cuh"

namespace ssd {

// Tokens per tile of the running decay (the token tile of cp_correct_tc).
constexpr int kCpTile = 128;

// ----------------------------------------------------------------------------
// Running log2 decays of a segment, tiled over tokens:
//   u_t = softplus(dt[b, t, h]) A_h log2(e)   (or dt A_h log2(e)),
//   a[b, h, t] = sum of u over t's 128-token tile up to t (inclusive),
//   tot[b, h, k] = sum of u over tile k,
// so that the running decay from the segment's start is a[b, h, t] plus the
// totals of the tiles before t's (cp_tile_prefix_kernel turns tot into those
// sums).  Block: one tile x 32 heads; dt is read
// coalesced over heads, each warp scans four heads (a lane holds four
// consecutive tokens).  grid (ntiles, ceil(H / 32), b), 256 threads.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cp_tile_decay_kernel(const float *__restrict__ dt,
                                                            const float *__restrict__ A,
                                                            float *__restrict__ a,
                                                            float *__restrict__ tot, int64_t T,
                                                            int H, int ntiles, int softplus) {
  __shared__ float tile[32][kCpTile + 4];
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kCpTile;
  const int h0 = blockIdx.y * 32, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr float kLog2e = 1.4426950408889634f;
  const int h = h0 + lane;
  float z[kCpTile / 8];
#pragma unroll
  for (int k = 0; k < kCpTile / 8; ++k) {  // every load first: all 16 are in flight at once
    const int64_t t = t0 + warp + 8 * k;
    z[k] = t < T && h < H ? dt[(static_cast<int64_t>(b) * T + t) * H + h] : 0.f;
  }
  const float Ah = h < H ? A[h] : 0.f;
#pragma unroll
  for (int k = 0; k < kCpTile / 8; ++k) {
    const int r = warp + 8 * k;
    tile[lane][r] = t0 + r < T ? (softplus ? softplus_f32(z[k]) : z[k]) * Ah * kLog2e : 0.f;
  }
  __syncthreads();
  for (int j = warp; j < 32 && h0 + j < H; j += 8) {
    const float4 q = *reinterpret_cast<const float4 *>(&tile[j][4 * lane]);
    const float v[4] = {q.x, q.x + q.y, q.x + q.y + q.z, q.x + q.y + q.z + q.w};
    float incl = v[3];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    const float before = incl - v[3];
    const int64_t row = static_cast<int64_t>(b) * H + h0 + j;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t t = t0 + 4 * lane + k;
      if (t < T) a[row * T + t] = before + v[k];
    }
    if (lane == 31) tot[row * ntiles + blockIdx.x] = incl;
  }
}

// In place: tot[row, k] <- sum of tot[row, 0 .. k) (the decay over the tiles
// before tile k; one warp per row, 32 tiles per step with a running carry);
// decay[row] = 2^(sum over all tiles), the segment's total decay Lambda,
// when given.
__global__ void __launch_bounds__(256) cp_tile_prefix_kernel(float *__restrict__ tot, int ntiles,
                                                             int64_t rows,
                                                             float *__restrict__ decay) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int lane = threadIdx.x & 31;
  float *r = tot + row * ntiles;
  float carry = 0.f;
  for (int k0 = 0; k0 < ntiles; k0 += 32) {
    const float v = k0 + lane < ntiles ? r[k0 + lane] : 0.f;
    float incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    if (k0 + lane < ntiles) r[k0 + lane] = carry + incl - v;
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (decay && lane == 0) decay[row] = ex2_approx(carry);
}

// ----------------------------------------------------------------------------
// H_in(rank) from the gathered segment decays and final states, and this
// rank's true final state:
//   H = 0; for r' < rank: H = Lambda_r' H + F_r';   h_in = H;
//   h_final = Lambda_rank H + F_rank
// decays [nranks, BH], finals [nranks, BH, NP]; one float4 per thread.
// h_in_op (when given) receives H rounded to bf16 in the operand image
// cp_correct_tc copies as is: per (b, h), P / 64 atoms of N rows x 128 bytes,
// element (n, p) of atom p / 64 at sw128_offset(n, p % 64) -- the layout of
// a 128-byte-swizzled tile at a 1024-byte-aligned shared-memory address.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cp_combine_kernel(const float *__restrict__ decays,
                                                         const float *__restrict__ finals,
                                                         int rank, int64_t BH, int NP, int P,
                                                         float *__restrict__ h_in,
                                                         uint8_t *__restrict__ h_in_op,
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
  if (h_in_op) {
    const int e = static_cast<int>(i4 * 4 - bh * NP), n = e / P, p = e % P;
    const int N = NP / P;
    *reinterpret_cast<uint2 *>(h_in_op + bh * NP * 2 + (p >> 6) * N * 128 + sw128_offset(n, p & 63)) =
        make_uint2(pack_bf16x2(H.x, H.y), pack_bf16x2(H.z, H.w));
  }
  if (h_final) {
    const float L = decays[static_cast<int64_t>(rank) * BH + bh];
    const float4 F =
        reinterpret_cast<const float4 *>(finals + static_cast<int64_t>(rank) * BH * NP)[i4];
    reinterpret_cast<float4 *>(h_final)[i4] =
        make_float4(fmaf(L, H.x, F.x), fmaf(L, H.y, F.y), fmaf(L, H.z, F.z), fmaf(L, H.w, F.w));
  }
}

// ----------------------------------------------------------------------------
// y[b, t, h, :] += 2^(a_t) (C[b, t, g(h), :] H_in[b, h]) on the tensor cores,
// streamed: a persistent CTA per SM walks work units (batch row, 128-token
// tile, run of hpc heads sharing a C group; the run is the fastest index, so
// CTAs working at the same time share C tiles in L2 and touch neighbouring
// y rows), one job per (unit, head).  Warp roles:
//   warp 4 (one lane), loads: per unit the C tile (128 tokens x 128 state
//     columns, TMA, two buffers), per job the head's H_in operand image (one
//     bulk copy of what cp_combine_kernel wrote, kHBufs buffers) and the head's
//     y tile (TMA, a ring of kYSlots tiles), each as soon as its buffer is
//     free, so that several jobs' y is in flight;
//   warp 5 (one lane), MMAs: C (K-major A) x H_in (MN-major B) into one of two
//     128 x P float32 accumulators in tensor memory;
//   warps 0-3, rows: thread t owns token t of the tile: it reads its
//     accumulator row, scales by 2^(a_t) and adds it into its y row in shared
//     memory; each warp then stores its 32 rows with one TMA store per
//     64-column atom.  Tokens past T are zero-filled on load and not stored.
// Every wait is bounded in time.
// ----------------------------------------------------------------------------
template <int P>
struct CpTc {
  static constexpr int N = kTcN, TQ = 128;
  static constexpr int kCBytes = TQ * N * 2;   // one C tile, two 64-column atoms
  static constexpr int kHBytes = N * P * 2;    // one head's H_in operand image
  static constexpr int kYBytes = TQ * P * 2;   // one head's y tile, P / 64 atoms
  static constexpr int kHBufs = P == 64 ? 4 : 2;   // H_in copies in flight
  static constexpr int kYSlots = P == 64 ? 5 : 3;  // y tiles in flight
  static constexpr int kThreads = 192;
  // barriers: C in / C free (two buffers), product done and accumulator read
  // by the 128 row threads (two accumulators), H in / H free (kHBufs
  // buffers), y in / y stored by the four row warps (kYSlots slots)
  static constexpr int kCin = 0, kCfree = 2, kDone = 4, kFree = 6, kHin = 8,
                       kHfree = kHin + kHBufs, kYin = kHfree + kHBufs, kYfree = kYin + kYSlots,
                       kBars = kYfree + kYSlots;
  static constexpr int kBytes =
      1024 + 2 * kCBytes + kHBufs * kHBytes + kYSlots * kYBytes + kBars * 8 + 16;
};

template <int P>
__global__ void __launch_bounds__(CpTc<P>::kThreads, 1)
    cp_correct_tc(const __grid_constant__ CUtensorMap mapC,
                  const __grid_constant__ CUtensorMap mapYl,
                  const __grid_constant__ CUtensorMap mapYs, const uint8_t *__restrict__ h_in_op,
                  const float *__restrict__ a, const float *__restrict__ pre, int ntiles, int64_t T,
                  int H, int GC, int hpc, int64_t nunits) {
  using L = CpTc<P>;
  constexpr int N = L::N, TQ = L::TQ, HB = L::kHBytes, YB = L::kYBytes, NY = L::kYSlots,
                NH = L::kHBufs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *Cs = smem;                    // 2 x [two atoms of TQ rows x 128 B]
  uint8_t *Hs = Cs + 2 * L::kCBytes;     // NH x [P / 64 atoms of N rows x 128 B]
  uint8_t *Ys = Hs + NH * HB;            // NY x [P / 64 atoms of TQ rows x 128 B]
  uint64_t *bars = reinterpret_cast<uint64_t *>(Ys + NY * YB);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + L::kBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nrun = H / hpc;
  const int per_group = H / GC;
  // this CTA's units: blockIdx.x, + gridDim.x, ...; jobs = units x hpc
  const int64_t my_units =
      nunits > blockIdx.x ? (nunits - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  struct Unit { int b, run; int64_t tile; };
  auto unit_of = [&](int64_t k) {  // k-th unit of this CTA
    const int64_t u = blockIdx.x + k * gridDim.x;
    Unit r;
    r.run = static_cast<int>(u % nrun);
    const int64_t bt = u / nrun;
    r.tile = bt % ntiles;
    r.b = static_cast<int>(bt / ntiles);
    return r;
  };

  if (tid == 0) {
    for (int i = 0; i < L::kBars; ++i) {
      const bool rows = i == L::kFree || i == L::kFree + 1;
      const bool warps = i >= L::kYfree;
      mbar_init(&bars[i], rows ? 128 : warps ? 4 : 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, 2 * P);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tslot;

  // Every role walks the same jobs in the same order: units k = 0, 1, ... of
  // this CTA (decoded once each), heads j = 0 .. hpc - 1 within; the ring
  // positions advance by increments (no division per job).
  if (warp == 4) {
    // ---------------- loads ----------------
    if (lane == 0) {
      prefetch_tensormap(&mapC);
      prefetch_tensormap(&mapYl);
      int hb = 0, hr = 0, ys = 0, yr = 0;  // ring slots and rounds of H_in and y
      bool ok = true;
      for (int64_t k = 0; k < my_units && ok; ++k) {
        const Unit U = unit_of(k);
        const int t0 = static_cast<int>(U.tile * TQ), cb = static_cast<int>(k & 1);
        if (k >= 2 && !mbar_wait(&bars[L::kCfree + cb], ((k >> 1) - 1) & 1, abort_flag)) break;
        const int g = (U.run * hpc) / per_group;
        mbar_arrive_expect_tx(&bars[L::kCin + cb], L::kCBytes);
        tma_load_4d(Cs + cb * L::kCBytes, &mapC, &bars[L::kCin + cb], 0, g, t0, U.b);
        tma_load_4d(Cs + cb * L::kCBytes + TQ * 128, &mapC, &bars[L::kCin + cb], 64, g, t0, U.b);
        for (int j = 0; j < hpc; ++j) {
          const int h = U.run * hpc + j;
          // H_in buffer hb: free once the product of its previous job is done
          if (hr > 0 && !mbar_wait(&bars[L::kHfree + hb], (hr - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars[L::kHin + hb], HB);
          bulk_load(Hs + hb * HB, h_in_op + (static_cast<int64_t>(U.b) * H + h) * HB, HB,
                    &bars[L::kHin + hb]);
          // y slot ys: free once its previous job's rows are stored
          if (yr > 0 && !mbar_wait(&bars[L::kYfree + ys], (yr - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars[L::kYin + ys], YB);
#pragma unroll
          for (int at = 0; at < P / 64; ++at)
            tma_load_4d(Ys + ys * YB + at * TQ * 128, &mapYl, &bars[L::kYin + ys], 64 * at, h,
                        t0, U.b);
          if (++hb == NH) hb = 0, ++hr;
          if (++ys == NY) ys = 0, ++yr;
        }
      }
    }
  } else if (warp == 5) {
    // ---------------- MMAs ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, P, false, true);
      int64_t q = 0;
      int hb = 0, hr = 0;
      bool ok = true;
      for (int64_t k = 0; k < my_units && ok; ++k) {
        const int cb = static_cast<int>(k & 1);
        if (!mbar_wait(&bars[L::kCin + cb], (k >> 1) & 1, abort_flag)) break;
        for (int j = 0; j < hpc; ++j, ++q) {
          const int s = static_cast<int>(q & 1);
          if (!mbar_wait(&bars[L::kHin + hb], hr & 1, abort_flag) ||
              (q >= 2 && !mbar_wait(&bars[L::kFree + s], ((q - 2) >> 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t ca = smem_u32(Cs + cb * L::kCBytes), ha = smem_u32(Hs + hb * HB);
#pragma unroll
          for (int ks = 0; ks < N / 16; ++ks) {
            const uint32_t koff = (ks >> 2) * TQ * 128 + (ks & 3) * 32;
            mma_bf16(tmem + s * P, sdesc_sw128(ca + koff, 16, 1024),
                     sdesc_sw128(ha + ks * 2048, N * 128, 1024), idesc, ks > 0 ? 1u : 0u);
          }
          mma_commit(&bars[L::kDone + s]);
          mma_commit(&bars[L::kHfree + hb]);
          if (j == hpc - 1) mma_commit(&bars[L::kCfree + cb]);  // the unit is done with its C
          if (++hb == NH) hb = 0, ++hr;
        }
      }
    }
  } else {
    // ---------------- rows (warps 0-3) ----------------
    const int row = tid;  // token t0 + row; tensor-memory lane `row`
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    auto decay_of = [&](const Unit &U, int j) -> float {  // running log2 decay of the row's token
      const int64_t t = U.tile * TQ + row;
      if (t >= T) return 0.f;
      const int64_t bh = static_cast<int64_t>(U.b) * H + U.run * hpc + j;
      return a[bh * T + t] + pre[bh * ntiles + U.tile];
    };
    int64_t q = 0;
    int ys = 0, yr = 0, ys_prev = NY - 1;
    bool ok = true;
    Unit U = unit_of(0);
    float fnext = my_units > 0 ? decay_of(U, 0) : 0.f;
    for (int64_t k = 0; k < my_units && ok; ++k) {
      const Unit Un = k + 1 < my_units ? unit_of(k + 1) : U;
      for (int j = 0; j < hpc; ++j, ++q) {
        const float f = ex2_approx(fnext);
        fnext = j + 1 < hpc ? decay_of(U, j + 1) : k + 1 < my_units ? decay_of(Un, 0) : 0.f;
        const int s = static_cast<int>(q & 1);
        const bool w = mbar_wait(&bars[L::kYin + ys], yr & 1, abort_flag) &&
                       mbar_wait(&bars[L::kDone + s], (q >> 1) & 1, abort_flag);
        if (!__all_sync(0xffffffffu, w)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint8_t *yt = Ys + ys * YB;
#pragma unroll
        for (int c = 0; c < P; c += 32) {
          float acc[32];
          tmem_ld32(tmem + lane_base + s * P + c, acc);
          uint8_t *rowp = yt + (c >> 6) * TQ * 128 + row * 128;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {  // four 16-byte chunks of 8 columns
            const int cc = ((c & 63) >> 3) + k4;
            uint4 *ch = reinterpret_cast<uint4 *>(rowp + (((cc ^ row) & 7) << 4));
            uint4 u = *ch;
            uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 yv = unpack_bf16x2(wv[e]);
              wv[e] = pack_bf16x2(fmaf(f, acc[8 * k4 + 2 * e], yv.x),
                                  fmaf(f, acc[8 * k4 + 2 * e + 1], yv.y));
            }
            *ch = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
        tc_fence_before_sync();
        mbar_arrive(&bars[L::kFree + s]);  // the accumulator may take job q + 2's product
        fence_proxy_async_smem();          // the updated rows are visible to the TMA store
        __syncwarp();
        if (lane == 0) {
          const int64_t tw = U.tile * TQ + 32 * warp;
          if (tw < T) {
#pragma unroll
            for (int at = 0; at < P / 64; ++at)
              tma_store_4d(&mapYs, yt + at * TQ * 128 + 32 * warp * 128, 64 * at,
                           U.run * hpc + j, static_cast<int>(tw), U.b);
          }
          bulk_commit();
          bulk_wait_read1();  // the previous job's store has read its slot
          if (q >= 1) mbar_arrive(&bars[L::kYfree + ys_prev]);
        }
        __syncwarp();
        ys_prev = ys;
        if (++ys == NY) ys = 0, ++yr;
      }
      U = Un;
    }
    if (lane == 0) bulk_wait_all();
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 2 * P);
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
                                                       const float *__restrict__ pre,
                                                       int ntiles, IO *__restrict__ y,
                                                       int64_t T, int H, int GC, int N, int P,
                                                       int PS) {
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
  const float f = exp2f(a[bh * T + t] + pre[bh * ntiles + t0 / kCpTile]);
  IO *row = y + ((static_cast<int64_t>(b) * T + t) * H + h) * P + p0 + tx * ncol;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < ncol) row[j] = from_f32<IO>(fmaf(f, acc[j], to_f32(row[j])));
}

}  // namespace ssd
