// ssd_kernels.cuh -- CUDA-core kernels of libssd:
//   dt_cumsum_kernel      softplus(dt) * A and its in-chunk inclusive running sum
//   state_passing_kernel  the scan of chunk-final states across chunks
//   chunk_state_simt / chunk_scan_simt
//                         float32-accurate chunk kernels (the fp32 I/O path and
//                         shapes outside the tensor-core kernels' envelope)
//   multistep_kernel      K-token verification decode from a cached state, and
//                         the fused recompute + verify + cache step
#pragma once

#include <type_traits>

#include "ssd_device.cuh"

namespace ssd {

// ----------------------------------------------------------------------------
// dt -> cs.  cs[b,h,c,i] = sum_{k<=i} softplus(dt[b, cQ+k, h]) * A_h, inclusive,
// within chunk c (the in-chunk "segment sums" whose differences give the decay
// mask L and whose last entry gives the chunk decay; Mamba-2 page, section
// "SSD算法", the modified A factors of the state-passing step).  Positions past
// T contribute 0, so a short last chunk keeps its last valid value.
// grid (nc, batch, ceil(H/32)), 256 threads: the block stages the chunk's
// dt rows for 32 heads (coalesced), then warp w scans heads w, w+8, ...
// ----------------------------------------------------------------------------
template <int Q>
__global__ void __launch_bounds__(256) dt_cumsum_kernel(const float *__restrict__ dt,
                                                         const float *__restrict__ A,
                                                         float *__restrict__ cs, int64_t T, int H,
                                                         int nc, int softplus) {
  constexpr int PER = Q / 32;
  __shared__ float tile[Q][33];
  const int c = blockIdx.x, b = blockIdx.y, h0 = blockIdx.z * 32;
  const int nh = min(32, H - h0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tc = static_cast<int64_t>(c) * Q;
  for (int idx = threadIdx.x; idx < Q * 32; idx += 256) {
    const int t = idx >> 5, hh = idx & 31;
    float d = 0.f;
    if (hh < nh && tc + t < T) {
      const float z = dt[(static_cast<int64_t>(b) * T + tc + t) * H + h0 + hh];
      d = (softplus ? softplus_f32(z) : z) * A[h0 + hh];
    }
    tile[t][hh] = d;
  }
  __syncthreads();
  for (int hh = warp; hh < nh; hh += 8) {
    float v[PER];
    float run = 0.f;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      run += tile[lane * PER + k][hh];
      v[k] = run;
    }
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    const float excl = incl - run;
    float *out = cs + ((static_cast<int64_t>(b) * H + h0 + hh) * nc + c) * Q + lane * PER;
#pragma unroll
    for (int k = 0; k < PER; ++k) out[k] = v[k] + excl;
  }
}

// ----------------------------------------------------------------------------
// State passing across chunks (Mamba-2 page, "SSD算法", the 1-semiseparable
// scan): Hin[0] = h0 (or 0), Hin[c+1] = exp(cs_last(c)) * Hin[c] + S[c],
// h_final = Hin[nc].  Every (b, h, n, p) element is an independent scan over
// the nc chunks; each thread carries 4 consecutive elements.
// S, Hin: [b, nc, H, N*P]; grid (ceil(NP/1024), H, batch), 256 threads.
// ----------------------------------------------------------------------------
template <typename HT>
__device__ __forceinline__ void store4(HT *dst, float4 v);
template <> __device__ __forceinline__ void store4<float>(float *dst, float4 v) {
  *reinterpret_cast<float4 *>(dst) = v;
}
template <> __device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *dst, float4 v) {
  uint2 u;
  u.x = pack_bf16x2(v.x, v.y);
  u.y = pack_bf16x2(v.z, v.w);
  *reinterpret_cast<uint2 *>(dst) = u;
}

template <typename HT>
__global__ void __launch_bounds__(256) state_passing_kernel(
    const float *__restrict__ S, const float *__restrict__ cs, const float *__restrict__ h0,
    HT *__restrict__ Hin, float *__restrict__ h_final, int H, int nc, int Q, int NP) {
  const int b = blockIdx.z, h = blockIdx.y;
  const int e = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (e >= NP) return;
  const int64_t bh = static_cast<int64_t>(b) * H + h;
  float4 st = make_float4(0.f, 0.f, 0.f, 0.f);
  if (h0) st = *reinterpret_cast<const float4 *>(h0 + bh * NP + e);
  const float *csl = cs + bh * nc * Q + (Q - 1);
#pragma unroll 4
  for (int c = 0; c < nc; ++c) {
    const int64_t off = ((static_cast<int64_t>(b) * nc + c) * H + h) * NP + e;
    const float4 s = __ldcs(reinterpret_cast<const float4 *>(S + off));
    const float decay = expf(csl[static_cast<int64_t>(c) * Q]);
    store4<HT>(Hin + off, st);
    st.x = fmaf(decay, st.x, s.x);
    st.y = fmaf(decay, st.y, s.y);
    st.z = fmaf(decay, st.z, s.z);
    st.w = fmaf(decay, st.w, s.w);
  }
  if (h_final) *reinterpret_cast<float4 *>(h_final + bh * NP + e) = st;
}

// ----------------------------------------------------------------------------
// Chunk-final states from a zero initial state, on CUDA cores in float32
// (Mamba-2 page, "SSD算法", the green step):
//   S[b,c,h][n][p] = sum_j exp(cs_last - cs_j) B[cQ+j, n] x[cQ+j, p].
// One block computes a 64 x 64 tile of S (rows n0.., columns p0..) of one
// (batch, chunk, head); grid (ceil(N/64) * ceil(P/64) * nc, H, batch), 256
// threads, each a 4 x 4 register tile.  Tokens go through shared memory 32 at
// a time as float32: w_j B_j (the weight folded into B) and x_j.
// ----------------------------------------------------------------------------
constexpr int kSimtTok = 32;  // tokens per shared-memory block

template <typename IO>
__global__ void __launch_bounds__(256) chunk_state_simt(
    const IO *__restrict__ x, const IO *__restrict__ Bm, const float *__restrict__ cs,
    float *__restrict__ S, int64_t T, int H, int GB, int N, int P, int Q, int nc) {
  __shared__ float w_s[256];
  __shared__ __align__(16) float Bw[kSimtTok][64];
  __shared__ __align__(16) float Xs[kSimtTok][64];
  const int tilesP = (P + 63) / 64, tilesN = (N + 63) / 64;
  const int tile = blockIdx.x % (tilesN * tilesP), c = blockIdx.x / (tilesN * tilesP);
  const int n0 = 64 * (tile / tilesP), p0 = 64 * (tile % tilesP);
  const int h = blockIdx.y, b = blockIdx.z;
  const int gb = h / (H / GB);
  const int tid = threadIdx.x, tn = tid >> 4, tp = tid & 15;
  const int64_t t0 = static_cast<int64_t>(c) * Q;
  const int L = static_cast<int>(T - t0 < Q ? T - t0 : static_cast<int64_t>(Q));
  const float *csc = cs + ((static_cast<int64_t>(b) * H + h) * nc + c) * Q;
  const float cl = csc[Q - 1];
  for (int j = tid; j < Q; j += 256) w_s[j] = j < L ? expf(cl - csc[j]) : 0.f;
  float acc[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[r][e] = 0.f;
  for (int j0 = 0; j0 < L; j0 += kSimtTok) {
    __syncthreads();  // w_s written; previous block consumed
    for (int idx = tid; idx < kSimtTok * 64; idx += 256) {
      const int jj = idx >> 6, cc = idx & 63, j = j0 + jj;
      const bool in_t = j < L;
      const int64_t t = t0 + j;
      Bw[jj][cc] = in_t && n0 + cc < N
                       ? w_s[j] * to_f32(Bm[((static_cast<int64_t>(b) * T + t) * GB + gb) * N + n0 + cc])
                       : 0.f;
      Xs[jj][cc] = in_t && p0 + cc < P
                       ? to_f32(x[((static_cast<int64_t>(b) * T + t) * H + h) * P + p0 + cc])
                       : 0.f;
    }
    __syncthreads();
#pragma unroll 4
    for (int jj = 0; jj < kSimtTok; ++jj) {
      const float4 bv = *reinterpret_cast<const float4 *>(&Bw[jj][4 * tn]);
      const float4 xv = *reinterpret_cast<const float4 *>(&Xs[jj][4 * tp]);
      const float bn[4] = {bv.x, bv.y, bv.z, bv.w}, xp[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[r][e] = fmaf(bn[r], xp[e], acc[r][e]);
    }
  }
  float *Sc = S + ((static_cast<int64_t>(b) * nc + c) * H + h) * N * P;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int n = n0 + 4 * tn + r, p = p0 + 4 * tp;
    if (n < N && p < P)
      *reinterpret_cast<float4 *>(Sc + static_cast<int64_t>(n) * P + p) =
          make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  }
}

// ----------------------------------------------------------------------------
// Chunk outputs on CUDA cores in float32 (Mamba-2 page, "SSD算法": the orange
// diagonal block in quadratic form plus the blue term from the chunk's true
// initial state, and the D skip):
//   y_i = sum_{j<=i} exp(cs_i - cs_j) (C_i . B_j) x_j + exp(cs_i) C_i^T Hin + D x_i
// One block computes 32 rows i0.. x 64 columns p0.. of one (batch, chunk,
// head); grid (ceil(Q/32) * ceil(P/64) * nc, H, batch), 256 threads, thread
// (row ri, column group pg) owns 8 columns of one row.  Shared memory (floats):
// cs[Q], C rows [32][Np] (zero-padded to Np = N rounded up to 32), then per
// 32-token block the B rows [32][Np + 1] (odd stride: the score loop reads a
// column of it across the lanes), the masked scores G[32][33] and x (or, for
// the C Hin term, Hin rows) [32][64].
// ----------------------------------------------------------------------------
__host__ __device__ constexpr int scan_simt_smem_floats(int Q, int N) {
  return Q + 32 * ((N + 31) / 32 * 32) + 32 * ((N + 31) / 32 * 32 + 1) + 32 * 33 + kSimtTok * 64;
}

template <typename IO, typename HT>
__global__ void __launch_bounds__(256) chunk_scan_simt(
    const IO *__restrict__ x, const IO *__restrict__ Bm, const IO *__restrict__ Cm,
    const float *__restrict__ cs, const HT *__restrict__ Hin, const float *__restrict__ D,
    IO *__restrict__ y, int64_t T, int H, int GB, int GC, int N, int P, int Q, int nc) {
  extern __shared__ __align__(16) float sm_f[];
  const int Np = (N + 31) / 32 * 32;
  float *csq = sm_f;            // [Q]
  float *Ct = csq + Q;          // [32][Np]
  const int Bst = Np + 1;
  float *Bs = Ct + 32 * Np;     // [32][Bst]
  float *G = Bs + 32 * Bst;     // [32][33]
  float *Ws = G + 32 * 33;      // [32][64]: x block or Hin block (offset a multiple of 4 floats)
  const int rowT = (Q + 31) / 32, tilesP = (P + 63) / 64;
  const int per_c = rowT * tilesP;
  const int c = blockIdx.x / per_c, rem = blockIdx.x % per_c;
  const int i0 = 32 * (rem / tilesP), p0 = 64 * (rem % tilesP);
  const int h = blockIdx.y, b = blockIdx.z;
  const int gb = h / (H / GB), gc = h / (H / GC);
  const int tid = threadIdx.x, ri = tid >> 3, pg = tid & 7;
  const int i = i0 + ri;
  const int64_t t0 = static_cast<int64_t>(c) * Q;
  const int L = static_cast<int>(T - t0 < Q ? T - t0 : static_cast<int64_t>(Q));
  const float *csc = cs + ((static_cast<int64_t>(b) * H + h) * nc + c) * Q;
  for (int j = tid; j < Q; j += 256) csq[j] = csc[j];
  for (int idx = tid; idx < 32 * Np; idx += 256) {
    const int ii = idx / Np, n = idx % Np;
    Ct[idx] = i0 + ii < L && n < N
                  ? to_f32(Cm[((static_cast<int64_t>(b) * T + t0 + i0 + ii) * GC + gc) * N + n])
                  : 0.f;
  }
  float accd[8], acco[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) accd[e] = acco[e] = 0.f;
  auto accumulate = [&](const float *coef, int coef_stride, float (&acc)[8]) {
    // acc[e] += sum_k coef[k] * Ws[k][8 pg + e], k over the 32-row block
#pragma unroll 4
    for (int k = 0; k < 32; ++k) {
      const float g = coef[k * coef_stride];
      const float4 w0 = *reinterpret_cast<const float4 *>(&Ws[k * 64 + 8 * pg]);
      const float4 w1 = *reinterpret_cast<const float4 *>(&Ws[k * 64 + 8 * pg + 4]);
      acc[0] = fmaf(g, w0.x, acc[0]); acc[1] = fmaf(g, w0.y, acc[1]);
      acc[2] = fmaf(g, w0.z, acc[2]); acc[3] = fmaf(g, w0.w, acc[3]);
      acc[4] = fmaf(g, w1.x, acc[4]); acc[5] = fmaf(g, w1.y, acc[5]);
      acc[6] = fmaf(g, w1.z, acc[6]); acc[7] = fmaf(g, w1.w, acc[7]);
    }
  };
  // ---- C Hin, 32 state rows at a time
  const HT *Hc = Hin + ((static_cast<int64_t>(b) * nc + c) * H + h) * N * P;
  for (int nb = 0; nb < N; nb += 32) {
    __syncthreads();
    for (int idx = tid; idx < 32 * 64; idx += 256) {
      const int k = idx >> 6, cc = idx & 63;
      Ws[idx] = nb + k < N && p0 + cc < P ? to_f32(Hc[static_cast<int64_t>(nb + k) * P + p0 + cc]) : 0.f;
    }
    __syncthreads();
    accumulate(Ct + ri * Np + nb, 1, acco);
  }
  // ---- diagonal block, 32 tokens at a time (causal: tokens j <= i0 + 31)
  const int jmax = min(i0 + 32, L);
  for (int j0 = 0; j0 < jmax; j0 += kSimtTok) {
    __syncthreads();
    for (int idx = tid; idx < 32 * Np; idx += 256) {
      const int jj = idx / Np, n = idx % Np, j = j0 + jj;
      Bs[jj * Bst + n] = j < L && n < N
                    ? to_f32(Bm[((static_cast<int64_t>(b) * T + t0 + j) * GB + gb) * N + n])
                    : 0.f;
    }
    for (int idx = tid; idx < 32 * 64; idx += 256) {
      const int k = idx >> 6, cc = idx & 63, j = j0 + k;
      Ws[idx] = j < L && p0 + cc < P
                    ? to_f32(x[((static_cast<int64_t>(b) * T + t0 + j) * H + h) * P + p0 + cc])
                    : 0.f;
    }
    __syncthreads();
    // masked scores G[ii][jj] = exp(cs_i - cs_j) C_i . B_j for j <= i (4 per thread)
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int e = tid + 256 * q4, ii = e >> 5, jj = e & 31;
      const int gi = i0 + ii, gj = j0 + jj;
      float g = 0.f;
      if (gj <= gi && gi < L && gj < L) {
        float dot = 0.f;
        for (int n = 0; n < N; ++n) dot = fmaf(Ct[ii * Np + n], Bs[jj * Bst + n], dot);
        g = dot * expf(csq[gi] - csq[gj]);
      }
      G[ii * 33 + jj] = g;
    }
    __syncthreads();
    accumulate(G + ri * 33, 1, accd);
  }
  // ---- y = diagonal + exp(cs_i) C Hin + D x
  if (i < L) {
    const float ei = expf(csq[i]);
    const float Dh = D ? D[h] : 0.f;
    const int64_t row = ((static_cast<int64_t>(b) * T + t0 + i) * H + h) * P;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int p = p0 + 8 * pg + e;
      if (p < P) y[row + p] = from_f32<IO>(accd[e] + ei * acco[e] + Dh * to_f32(x[row + p]));
    }
  }
}

// ----------------------------------------------------------------------------
// K-token multi-step decode ("Mamba in the Llama", 推测解码, MultiStep) and the
// fused verifier step (same page, 硬件特定优化).
// One warp serves one item (head blockIdx.x of batch row b, p-slice of PS
// columns).  Lane (r, q) owns the 4 columns 4q..4q+3 of state rows r, r + R,
// r + 2R, ... (R = 32 / (PS/4) row groups).  Its rows stream through a
// lane-private ring of D float4 slots in shared memory filled by cp.async
// (D - 1 rows in flight without holding registers); the small per-call
// operands (B, C, x of the new tokens; B, x of the previous drafts) arrive
// the same way, raw, as one group ahead of them.
//
// The recurrence h_k = a_k h_{k-1} + B_k x_k^T is not stepped token by token:
// over a run of tokens lo..hi-1 it collapses to
//     h_hi = (prod_{lo<=m<hi} a_m) h_lo + sum_k (prod_{k<m<hi} a_m) B_k x_k^T,
// one scale and one rank-1 term per token, with the decay products folded
// into per-row coefficients W[n][k] = w_k B_k[n] once per item.  The outputs
// split the same way,
//     y_k = e_k C_k^T h_0 + sum_{m<=k} G[k][m] x_m + D x_k,
//     e_k = prod_{m<=k} a_m,  G[k][m] = (prod_{m<l<=k} a_l) C_k . B_m,
// so a state row only feeds K dot-product partials (coefficients e_k C_k[n])
// and the K x K matrix G is formed once per item from B and C.  Per state
// element that is 1 + (tokens folded) + K multiply-adds; the coefficients
// are float4 rows of shared memory, the lane's x columns sit in registers.
// For the decode instance (K fixed) the row loop is compiled once per
// accepted count, so each fold runs exactly its tokens with no predicates.
//
// Both modes fold with one routine (ms_fold) and form y with one routine, so
// a verifier chain (cache = the state before the previous drafts) and a
// multistep chain continuing from h_j produce identical bits.
// ----------------------------------------------------------------------------
constexpr int kMsThreads = 32;
constexpr int kMsMaxK = 16;

// ring of the state stream: DEPTH row slots per lane, filled two row steps
// per cp.async group (at most DEPTH / 2 groups outstanding)
__host__ __device__ constexpr int ms_depth(bool verify) { return verify ? 12 : 16; }

// dynamic shared memory per item (bytes).  float32: e C [N][KT], W [N][KW],
// G [KT][KT], decays [2][16], ring [DEPTH][32] float4.  io dtype, raw: B, C of
// the new tokens [KT][N + 16 B] (rows padded so that reads across tokens fall
// in distinct banks), x [KT][PS]; verify adds B_prev [KPT][N + 16 B] and
// x_prev [KPT][PS].
__host__ __device__ constexpr int ms_smem_bytes(int KT, int KPT, int N, int PS, bool verify,
                                                int io_bytes) {
  return 4 * (N * KT + N * (verify ? KPT : KT) + KT * KT + 2 * kMsMaxK) + 16 * 32 * ms_depth(verify) +
         io_bytes * (2 * KT * (N + 16 / io_bytes) + KT * PS +
                     (verify ? KPT * (N + 16 / io_bytes) + KPT * PS : 0));
}

// four consecutive elements as float (8- or 16-byte aligned; global or shared)
__device__ __forceinline__ float4 ms_ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 ms_ld4(const __nv_bfloat16 *p) {
  const uint2 v = *reinterpret_cast<const uint2 *>(p);
  const float2 a = unpack_bf16x2(v.x), c = unpack_bf16x2(v.y);
  return make_float4(a.x, a.y, c.x, c.y);
}
__device__ __forceinline__ void ms_st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void ms_st4(__nv_bfloat16 *p, float4 v) {
  *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

// asynchronous 16-byte copy global -> shared (cp.async, L2 only), and its
// group bookkeeping; a group completes in the order it was committed
__device__ __forceinline__ void ms_cp16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void ms_zero16(void *dst) {
  *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
}
__device__ __forceinline__ void ms_cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int NW>
__device__ __forceinline__ void ms_cp_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(NW) : "memory");
}

// prod_{lo <= l < hi} a[l], ascending; the one formula every decay product of
// both modes goes through (bit-identical folds)
__device__ __forceinline__ float ms_prod(const float *a, int lo, int hi) {
  float p = 1.f;
  for (int l = lo; l < hi; ++l) p *= a[l];
  return p;
}

// the coefficient w of token k when folding tokens lo..hi-1 (0 outside)
__device__ __forceinline__ float ms_weight(const float *a, int k, int lo, int hi) {
  return (k >= lo && k < hi) ? ms_prod(a, k + 1, hi) : 0.f;
}

__device__ __forceinline__ void ms_fma(float4 &s, float w, float4 v) {
  s.x = fmaf(w, v.x, s.x);
  s.y = fmaf(w, v.y, s.y);
  s.z = fmaf(w, v.z, s.z);
  s.w = fmaf(w, v.w, s.w);
}

// s = lam st + sum over tokens k in [lo, hi) of wrow[k] xr[k], ascending k.
// LO >= 0: the range is [LO, HI), fixed at compile time; LO < 0: [lo, hi).
template <int KW, int LO, int HI>
__device__ __forceinline__ float4 ms_fold(float lam, float4 st, const float *wrow,
                                          const float4 (&xr)[KW], int lo, int hi) {
  float4 s = make_float4(lam * st.x, lam * st.y, lam * st.z, lam * st.w);
#pragma unroll
  for (int k4 = 0; k4 < KW; k4 += 4) {
    if (LO >= 0 && (k4 + 4 <= LO || k4 >= HI)) continue;
    const float4 w = *reinterpret_cast<const float4 *>(wrow + k4);
    const float wk[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = k4 + u;
      if (LO >= 0 ? (k >= LO && k < HI) : (k >= lo && k < hi)) ms_fma(s, wk[u], xr[k]);
    }
  }
  return s;
}

// y partials: yp[k] += e_k C_k[n] st for the new tokens (crow: row n of e C);
// KX: K == KT
template <int KT, bool KX>
__device__ __forceinline__ void ms_ypart(float4 (&yp)[KT], const float *crow, float4 st, int K) {
#pragma unroll
  for (int k4 = 0; k4 < KT; k4 += 4) {
    const float4 c = *reinterpret_cast<const float4 *>(crow + k4);
    const float ck[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (KX || k4 + u < K) ms_fma(yp[k4 + u], ck[u], st);
  }
}

// KT: compile-time bound on K (8 or 16); KPT: on k_prev (verify).  NC: the
// state size N when fixed at compile time (0: taken from the arguments).  KX:
// K == KT exactly (the row loop is then specialised on the accepted count).
//
// Multistep (VF false): each state row yields the y partials, h_j (tokens
// 0..j-1 folded, ordinary stores: a speculative chain continues from it, so
// the next call finds it in L2) and h_K (tokens j..K-1 folded onto h_j).
// Verify (VF true): h_cache holds the state before the previous call's KP
// drafts (xp, dtp, Bp), jacc[b] of which were accepted; a row is folded
// through those, stored to h_next (the next call's cache) and then feeds the
// y partials of the K new drafts; h_j and h_K are not written.  Per state
// row that is one read and one write (multistep: one read, two writes).
template <typename IO, int KT, int KPT, int NC = 0, bool KX = false, bool VF = false>
__global__ void __launch_bounds__(kMsThreads, KT <= 8 ? 12 : 8) multistep_kernel(
    const IO *__restrict__ x, const float *__restrict__ dt, const float *__restrict__ A,
    const IO *__restrict__ Bm, const IO *__restrict__ Cm, const float *__restrict__ D,
    const float *__restrict__ h_cache, const int32_t *__restrict__ jacc, IO *__restrict__ y,
    float *__restrict__ h_j, float *__restrict__ h_K, int K_arg, int H, int GB, int GC, int N_arg,
    int P, int PS, int softplus, const IO *__restrict__ xp, const float *__restrict__ dtp,
    const IO *__restrict__ Bp, float *__restrict__ h_next, int KP, int nitems) {
  static_assert(!KX || KT == 8, "the specialised row loop covers accepted counts 0..8");
  constexpr int KW = VF ? KPT : KT;
  constexpr int DEPTH = ms_depth(VF);
  const int N = NC ? NC : N_arg;
  const int K = KX ? KT : K_arg;
  extern __shared__ float4 sm_ms4[];
  // Multistep: grid (SMs, rounds, P / PS).  CTAs are handed to the SMs in
  // index order, so an SM's CTAs are consecutive (b, h) items and mostly run
  // the same accepted-count specialisation of the row loop (fewer
  // instruction-cache misses).  Verify: grid (H, b, P / PS) -- the grouping
  // measured slower there.
  int h, b;
  if constexpr (VF) {
    h = blockIdx.x;
    b = blockIdx.y;
  } else {
    const int item = blockIdx.x * gridDim.y + blockIdx.y;
    if (item >= nitems) return;
    h = item % H;
    b = item / H;
  }
  const int p0 = blockIdx.z * PS;
  const int lane = threadIdx.x;
  const int NS = N + 16 / static_cast<int>(sizeof(IO));  // padded raw row
  float *sCe = reinterpret_cast<float *>(sm_ms4);  // e_k C_k [N][KT]
  float *sW = sCe + N * KT;                         // fold coefficients [N][KW]
  float *sG = sW + N * KW;                          // [KT][KT]
  float *sa = sG + KT * KT;                         // decays of the new tokens
  float *sap = sa + kMsMaxK;                        // verify: decays of the previous drafts
  float4 *ring = reinterpret_cast<float4 *>(sap + kMsMaxK);  // [DEPTH][32]
  IO *sBr = reinterpret_cast<IO *>(ring + DEPTH * kMsThreads);  // raw B [KT][NS]
  IO *sCr = sBr + KT * NS;                          // raw C [KT][NS]
  IO *sxr = sCr + KT * NS;                          // raw x [KT][PS]
  IO *sBpr = sxr + KT * PS;                         // verify: raw B_prev [KPT][NS]
  IO *sxpr = sBpr + KPT * NS;                       // verify: raw x_prev [KPT][PS]
  const int gb = h / (H / GB), gc = h / (H / GC);
  const int TP = PS / 4, R = kMsThreads / TP;
  const int q = lane % TP, r = lane / TP;
  const int rows = N / R;
  const int64_t base = (static_cast<int64_t>(b) * H + h) * N * P + p0 + 4 * q;

  // group 1: the per-call operands, raw, in 16-byte granules of GR elements;
  // rows past K (k_prev) zero
  constexpr int GR = 16 / static_cast<int>(sizeof(IO));
  const int NGB = N / GR, PG = PS / GR;
  for (int i = lane; i < KT * NGB; i += kMsThreads) {
    const int k = i / NGB, n = (i % NGB) * GR;
    if (k < K) {
      const int64_t ob = ((static_cast<int64_t>(b) * K + k) * GB + gb) * N + n;
      const int64_t oc = ((static_cast<int64_t>(b) * K + k) * GC + gc) * N + n;
      ms_cp16(sBr + k * NS + n, Bm + ob);
      ms_cp16(sCr + k * NS + n, Cm + oc);
    } else {
      ms_zero16(sBr + k * NS + n);
      ms_zero16(sCr + k * NS + n);
    }
  }
  for (int i = lane; i < KT * PG; i += kMsThreads) {
    const int k = i / PG, p = (i % PG) * GR;
    const int64_t ox = ((static_cast<int64_t>(b) * K + k) * H + h) * P + p0 + p;
    if (k < K) {
      ms_cp16(sxr + k * PS + p, x + ox);
    } else {
      ms_zero16(sxr + k * PS + p);
    }
  }
  if (VF) {
    for (int i = lane; i < KPT * NGB; i += kMsThreads) {
      const int k = i / NGB, n = (i % NGB) * GR;
      const int64_t ob = ((static_cast<int64_t>(b) * KP + k) * GB + gb) * N + n;
      if (k < KP) {
        ms_cp16(sBpr + k * NS + n, Bp + ob);
      } else {
        ms_zero16(sBpr + k * NS + n);
      }
    }
    for (int i = lane; i < KPT * PG; i += kMsThreads) {
      const int k = i / PG, p = (i % PG) * GR;
      const int64_t ox = ((static_cast<int64_t>(b) * KP + k) * H + h) * P + p0 + p;
      if (k < KP) {
        ms_cp16(sxpr + k * PS + p, xp + ox);
      } else {
        ms_zero16(sxpr + k * PS + p);
      }
    }
  }
  ms_cp_commit();
  // groups 2..DEPTH/2: the first DEPTH - 2 row steps of the state stream, two
  // per group
  constexpr int NGR = DEPTH / 2;
#pragma unroll
  for (int g = 0; g < NGR - 1; ++g) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int i = 2 * g + u;
      if (i < rows) ms_cp16(ring + i * kMsThreads + lane, h_cache + base + static_cast<int64_t>(r + R * i) * P);
    }
    ms_cp_commit();
  }

  int jb = jacc[b];
  if (jb < 0 || jb > (VF ? KP : K)) {
    if (lane == 0 && h == 0 && blockIdx.z == 0) report_error(kDevBadJ);
    jb = -1;
  }
  // verify: a batch row whose accepted count is out of range gets no outputs
  const bool run = !VF || jb >= 0;
  const int jf = jb < 0 ? 0 : jb;  // tokens folded into h_j (multistep) / h_next (verify)
  if (lane < kMsMaxK) {
    float av = 1.f;
    if (lane < K) {
      const float z = dt[(static_cast<int64_t>(b) * K + lane) * H + h];
      av = expf((softplus ? softplus_f32(z) : z) * A[h]);
    }
    sa[lane] = av;
    if (VF) {
      av = 1.f;
      if (lane < KP) {
        const float z = dtp[(static_cast<int64_t>(b) * KP + lane) * H + h];
        av = expf((softplus ? softplus_f32(z) : z) * A[h]);
      }
      sap[lane] = av;
    }
  }
  ms_cp_wait<NGR - 1>();  // group 1 has landed
  __syncwarp();

  // per-item coefficients, written as float4 rows: element 4i + u of e C
  // (or W) is token (4i) % KT + u of state index (4i) / KT; since
  // 128 % KT == 0 a lane keeps the same four tokens on every step
  {
    const int k0 = (4 * lane) % KT;
    float e[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) e[u] = k0 + u < K ? ms_prod(sa, 0, k0 + u + 1) : 0.f;
    for (int i = lane; i < N * KT / 4; i += kMsThreads) {
      const int n = (4 * i) / KT;
      *reinterpret_cast<float4 *>(sCe + 4 * i) =
          make_float4(e[0] * to_f32(sCr[k0 * NS + n]), e[1] * to_f32(sCr[(k0 + 1) * NS + n]),
                      e[2] * to_f32(sCr[(k0 + 2) * NS + n]), e[3] * to_f32(sCr[(k0 + 3) * NS + n]));
    }
    const int kw0 = (4 * lane) % KW;
    float w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int kw = kw0 + u;
      w[u] = VF ? ms_weight(sap, kw, 0, jf)
                : (kw < jf ? ms_weight(sa, kw, 0, jf) : ms_weight(sa, kw, jf, K));
    }
    // raw B times w (verify: of the previous drafts); the product commutes,
    // so both modes give a token's coefficient the same bits
    const IO *braw = VF ? sBpr : sBr;
    for (int i = lane; i < N * KW / 4; i += kMsThreads) {
      const int n = (4 * i) / KW;
      *reinterpret_cast<float4 *>(sW + 4 * i) =
          make_float4(w[0] * to_f32(braw[kw0 * NS + n]), w[1] * to_f32(braw[(kw0 + 1) * NS + n]),
                      w[2] * to_f32(braw[(kw0 + 2) * NS + n]), w[3] * to_f32(braw[(kw0 + 3) * NS + n]));
    }
    if constexpr (KT == 8) {
      // lane-split: the lane's partial C_k . B_m over its granules of four
      // state indices for all 64 (k, m), then a transposing butterfly: at
      // each level a lane keeps half of its values plus its partner's copy
      // of that half, so lane l ends with entries 2l and 2l + 1, summed
      // over the warp
      float pv[64];
#pragma unroll
      for (int e = 0; e < 64; ++e) pv[e] = 0.f;
      for (int n = 4 * lane; n < N; n += 4 * kMsThreads) {
        float4 bv[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) bv[m] = ms_ld4(sBr + m * NS + n);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const float4 cv = ms_ld4(sCr + kk * NS + n);
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            float &a = pv[kk * 8 + m];
            a = fmaf(cv.x, bv[m].x, a);
            a = fmaf(cv.y, bv[m].y, a);
            a = fmaf(cv.z, bv[m].z, a);
            a = fmaf(cv.w, bv[m].w, a);
          }
        }
      }
#pragma unroll
      for (int lv = 0; lv < 5; ++lv) {
        const int o = 16 >> lv, half = 32 >> lv;
        const bool hi = (lane & o) != 0;
#pragma unroll
        for (int e = 0; e < half; ++e) {
          const float lo_v = pv[e], hi_v = pv[e + half];
          const float recv = __shfl_xor_sync(0xffffffffu, hi ? lo_v : hi_v, o);
          pv[e] = (hi ? hi_v : lo_v) + recv;
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int t = 2 * lane + u, kk = t / 8, m = t % 8;
        sG[t] = (m <= kk && kk < K) ? pv[u] * ms_prod(sa, m + 1, kk + 1) : 0.f;
      }
    } else {
      for (int t = lane; t < KT * KT; t += kMsThreads) {
        const int kk = t / KT, m = t % KT;
        float g = 0.f;
        if (m <= kk && kk < K) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
          for (int n = 0; n < N; n += 4) {
            const float4 c = ms_ld4(sCr + kk * NS + n), bb = ms_ld4(sBr + m * NS + n);
            acc.x = fmaf(c.x, bb.x, acc.x);
            acc.y = fmaf(c.y, bb.y, acc.y);
            acc.z = fmaf(c.z, bb.z, acc.z);
            acc.w = fmaf(c.w, bb.w, acc.w);
          }
          g = ((acc.x + acc.y) + (acc.z + acc.w)) * ms_prod(sa, m + 1, kk + 1);
        }
        sG[t] = g;
      }
    }
  }
  __syncwarp();

  const float lam_j = ms_prod(VF ? sap : sa, 0, jf);  // decay of the folded tokens
  const float lam_K = VF ? 1.f : ms_prod(sa, jf, K);  // multistep: tokens j..K-1
  float4 xr[KW];  // the lane's columns of the folded tokens' x
#pragma unroll
  for (int k = 0; k < KW; ++k) xr[k] = ms_ld4((VF ? sxpr : sxr) + k * PS + 4 * q);

  float4 yp[KT];
#pragma unroll
  for (int k = 0; k < KT; ++k) yp[k] = make_float4(0.f, 0.f, 0.f, 0.f);

  // the row loop; JF >= 0: compiled for jf == JF (and K == KT)
  const auto row_loop = [&](auto jf_tag) {
    constexpr int JF = decltype(jf_tag)::value;
    constexpr int LO0 = JF >= 0 ? 0 : -1;       // the fold into h_j / h_next
    constexpr int LO1 = JF >= 0 ? JF : -1;      // multistep: the fold onto h_K
    const int64_t rstep = static_cast<int64_t>(R) * P;  // one row step in the state
    const float4 *rd = ring + lane;                                // slot of row step i2
    float4 *wr = ring + (DEPTH - 2) * kMsThreads + lane;           // slot of row step i2 + DEPTH - 2
    const float *src = h_cache + base + (DEPTH - 2) * rstep + static_cast<int64_t>(r) * P;
    float *out_a = (VF ? h_next : h_j) + base + static_cast<int64_t>(r) * P;
    float *out_b = h_K + base + static_cast<int64_t>(r) * P;     // multistep only
    const float *wrow = sW + r * KW, *crow = sCe + r * KT;
    for (int i2 = 0; i2 < rows; i2 += 2) {
      ms_cp_wait<NGR - 2>();  // row steps i2, i2 + 1 have landed (this lane's own copies)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (i2 + u < rows) {
          const float4 st = rd[u * kMsThreads];
          const float *wr_u = wrow + u * R * KW, *cr_u = crow + u * R * KT;
          if (VF) {
            const float4 s = ms_fold<KW, LO0, JF>(lam_j, st, wr_u, xr, 0, jf);
            *reinterpret_cast<float4 *>(out_a + u * rstep) = s;
            ms_ypart<KT, KX>(yp, cr_u, s, K);
          } else {
            ms_ypart<KT, KX>(yp, cr_u, st, K);
            const float4 sj = ms_fold<KW, LO0, JF>(lam_j, st, wr_u, xr, 0, jf);
            if (jb >= 0) *reinterpret_cast<float4 *>(out_a + u * rstep) = sj;
            __stcs(reinterpret_cast<float4 *>(out_b + u * rstep), ms_fold<KW, LO1, KT>(lam_K, sj, wr_u, xr, jf, K));
          }
        }
      }
      // refill the two slots read one step ago (their values are long consumed)
#pragma unroll
      for (int u = 0; u < 2; ++u)
        if (i2 + DEPTH - 2 + u < rows) ms_cp16(wr + u * kMsThreads, src + u * rstep);
      ms_cp_commit();
      rd += 2 * kMsThreads;
      if (rd == ring + DEPTH * kMsThreads + lane) rd = ring + lane;
      wr += 2 * kMsThreads;
      if (wr == ring + DEPTH * kMsThreads + lane) wr = ring + lane;
      src += 2 * rstep;
      out_a += 2 * rstep;
      out_b += 2 * rstep;
      wrow += 2 * R * KW;
      crow += 2 * R * KT;
    }
  };
  if (run) {
    if constexpr (KX) {
      switch (jf) {
        case 0: row_loop(std::integral_constant<int, 0>{}); break;
        case 1: row_loop(std::integral_constant<int, 1>{}); break;
        case 2: row_loop(std::integral_constant<int, 2>{}); break;
        case 3: row_loop(std::integral_constant<int, 3>{}); break;
        case 4: row_loop(std::integral_constant<int, 4>{}); break;
        case 5: row_loop(std::integral_constant<int, 5>{}); break;
        case 6: row_loop(std::integral_constant<int, 6>{}); break;
        case 7: row_loop(std::integral_constant<int, 7>{}); break;
        default: row_loop(std::integral_constant<int, 8>{}); break;
      }
    } else {
      row_loop(std::integral_constant<int, -1>{});
    }
  }
  ms_cp_wait<0>();  // no copy may outlive the block (a skipped row loop leaves some)
  if (!run) return;
  // sum the partials over the row groups (lanes q, q + TP, ...); lane (r, q)
  // then writes tokens k = r, r + R, ... of its four columns
  const float Dh = D ? D[h] : 0.f;
#pragma unroll
  for (int k = 0; k < KT; ++k) {
    if (k < K) {
      float4 v = yp[k];
      for (int o = TP; o < kMsThreads; o <<= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
        v.z += __shfl_xor_sync(0xffffffffu, v.z, o);
        v.w += __shfl_xor_sync(0xffffffffu, v.w, o);
      }
      if (k % R == r) {
        // sum_{m<=k} G[k][m] x_m: the part of y_k that does not see the state
        float4 loc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int m = 0; m <= k; ++m) ms_fma(loc, sG[k * KT + m], ms_ld4(sxr + m * PS + 4 * q));
        const float4 xk = ms_ld4(sxr + k * PS + 4 * q);
        ms_st4(y + ((static_cast<int64_t>(b) * K + k) * H + h) * P + p0 + 4 * q,
               make_float4(v.x + loc.x + Dh * xk.x, v.y + loc.y + Dh * xk.y,
                           v.z + loc.z + Dh * xk.z, v.w + loc.w + Dh * xk.w));
      }
    }
  }
}

}  // namespace ssd
