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
//
// Long sequences with few (batch, head) pairs are cut into nseg segments of
// cps chunks that run in parallel (Mamba-2 page, section "深入解析分块与状态
// 传递机制": the same chunk/state split, one level up).  Segment 0 starts from
// h0, the others from zero; each CTA then also writes its segment's final
// state (Fseg), the product of its chunk decays (Lseg) and, per chunk, the
// product of the decays before it within the segment (Dc).  state_fixup_kernel
// turns these into the true chunk states.
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
                        int H, int GB, int nc, int P, int softplus, int nseg, int cps,
                        float *__restrict__ Fseg, float *__restrict__ Lseg,
                        float *__restrict__ Dc) {
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

  const int p0 = blockIdx.x * PS, h = blockIdx.y, b = blockIdx.z / nseg, seg = blockIdx.z % nseg;
  const int c_begin = seg * cps, ncl = min(nc, c_begin + cps) - c_begin;  // this CTA's chunks
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

  auto issue_loads = [&](int c) {  // global chunk index
    mbar_arrive_expect_tx(&bars[0], L::kB + L::kX);
#pragma unroll
    for (int s = 0; s < N / 64; ++s) tma_load_4d(Bt + s * Q * 128, &mapB, &bars[0], 64 * s, gb, c * Q, b);
    tma_load_4d(Xt, &mapX, &bars[0], p0, h, c * Q, b);
  };
  auto load_dt = [&](int c) {
    const int64_t t = static_cast<int64_t>(c) * Q + tid;
    return (tid < Q && t < T) ? dt[(static_cast<int64_t>(b) * T + t) * H + h] : 0.f;
  };
  // cumsum of softplus(dt) * A_h over chunk c into buffer lc & 1 (one token per thread)
  auto cumsum = [&](int c, int lc, float z) {
    float *cs = csb + (lc & 1) * Q, *w = wb + (lc & 1) * Q;
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
    if (tid == 0) decay_s[lc & 1] = __expf(cl);
    // readers of w / decay synchronise later in the loop
  };

  const int64_t srow = ((static_cast<int64_t>(b) * H + h) * N + n) * P + p0 + cbase;
  float st[32];
  if (h0 && seg == 0) {
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
      const float4 v = *reinterpret_cast<const float4 *>(h0 + srow + e);
      st[e] = v.x; st[e + 1] = v.y; st[e + 2] = v.z; st[e + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) st[e] = 0.f;
  }

  // product of the decays of this segment's chunks so far (Dc, Lseg)
  const bool track = Dc != nullptr && blockIdx.x == 0 && tid == 0;
  float prod = 1.f;
  if (tid == 0) issue_loads(c_begin);
  cumsum(c_begin, 0, load_dt(c_begin));
  float z_next = ncl > 1 ? load_dt(c_begin + 1) : 0.f;
  for (int lc = 0; lc < ncl; ++lc) {
    const int c = c_begin + lc;
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
    const float *w = wb + (lc & 1) * Q;
    if (track) {
      Dc[(static_cast<int64_t>(b) * H + h) * nc + c] = prod;
      prod *= decay_s[lc & 1];
    }
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars[0], lc & 1, abort_flag));
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
    if (lc + 1 < ncl) {
      cumsum(c + 1, lc + 1, z_next);
      if (lc + 2 < ncl) z_next = load_dt(c + 2);
    }
    ok = !*abort_flag && mbar_wait(&bars[1], lc & 1, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after_sync();
    if (tid == 0 && ok && lc + 1 < ncl) issue_loads(c + 1);  // the tiles are free again
    if (ok) {
      const float decay = decay_s[lc & 1];
      float sv[32];
      tmem_ld32(taddr, sv);
#pragma unroll
      for (int e = 0; e < 32; ++e) st[e] = fmaf(decay, st[e], sv[e]);
    }
    tc_fence_before_sync();
  }
  // the sequence's final state, or this segment's (from its own start state)
  float *fin = nseg == 1 ? h_final
                         : Fseg + ((static_cast<int64_t>(b) * H + h) * nseg + seg) * N * P +
                               static_cast<int64_t>(n) * P + p0 + cbase;
  if (fin) {
    if (nseg == 1) fin += srow;
#pragma unroll
    for (int e = 0; e < 32; e += 4)
      *reinterpret_cast<float4 *>(fin + e) = make_float4(st[e], st[e + 1], st[e + 2], st[e + 3]);
  }
  if (track && nseg > 1) Lseg[(static_cast<int64_t>(b) * H + h) * nseg + seg] = prod;
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, PS);
}

// ----------------------------------------------------------------------------
// True chunk states of a segmented state pass.  With T_s the true state at the
// start of segment s (T_1 = Fseg_0, since segment 0 started from h0):
//   Hin_c += Dc_c * T_s           for every chunk c of segment s >= 1
//   T_{s+1} = Lseg_s * T_s + Fseg_s,   h_final = T_nseg
// for the split (batch, head) rows bh0, bh0 + 1, ... (row = b H + h), whose
// hand-off arrays are indexed from bh0.  Elementwise over (row, n, p);
// thread = 4 consecutive elements; grid (ceil(N P / 1024), rows), 256 threads.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) state_fixup_kernel(
    const float *__restrict__ Fseg, const float *__restrict__ Lseg, const float *__restrict__ Dc,
    __nv_bfloat16 *__restrict__ Hin, float *__restrict__ h_final, int H, int nc, int cps,
    int nseg, int NP, int64_t bh0) {
  const int64_t r = blockIdx.y;  // row relative to bh0
  const int64_t bh = bh0 + r;
  const int64_t b = bh / H;
  const int h = static_cast<int>(bh % H);
  const int e = 4 * (blockIdx.x * 256 + threadIdx.x);
  grid_dep_trigger();  // the chunk scan may start its set-up
  grid_dep_wait();     // the segment results of the chunk-state kernel
  if (e >= NP) return;
  float4 Ts = *reinterpret_cast<const float4 *>(Fseg + r * nseg * NP + e);
  for (int s = 1; s < nseg; ++s) {
    const int c0 = s * cps, c1 = min(nc, c0 + cps);
    const int64_t cstride = static_cast<int64_t>(H) * NP;  // one chunk further in Hin
    uint2 *base = reinterpret_cast<uint2 *>(Hin + ((b * nc + c0) * H + h) * NP + e);
    // eight chunks per round, loads first, so that many reads are in flight
    for (int c = c0; c < c1; c += 8) {
      uint2 v[8];
      float d[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (c + u < c1) {
          v[u] = *reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(base) + (c - c0 + u) * cstride);
          d[u] = Dc[r * nc + c + u];
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (c + u < c1) {
          const float2 lo = unpack_bf16x2(v[u].x), hi = unpack_bf16x2(v[u].y);
          uint2 o;
          o.x = pack_bf16x2(fmaf(d[u], Ts.x, lo.x), fmaf(d[u], Ts.y, lo.y));
          o.y = pack_bf16x2(fmaf(d[u], Ts.z, hi.x), fmaf(d[u], Ts.w, hi.y));
          *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(base) + (c - c0 + u) * cstride) = o;
        }
      }
    }
    const float l = Lseg[r * nseg + s];
    const float4 f = *reinterpret_cast<const float4 *>(Fseg + (r * nseg + s) * NP + e);
    Ts = make_float4(fmaf(l, Ts.x, f.x), fmaf(l, Ts.y, f.y), fmaf(l, Ts.z, f.z), fmaf(l, Ts.w, f.w));
  }
  if (h_final) *reinterpret_cast<float4 *>(h_final + bh * NP + e) = Ts;
}

}  // namespace ssd
