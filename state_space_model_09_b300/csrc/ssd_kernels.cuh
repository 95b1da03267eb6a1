// ssd_kernels.cuh -- CUDA-core kernels of libssd:
//   dt_cumsum_kernel      softplus(dt) * A and its in-chunk inclusive running sum
//   state_passing_kernel  the scan of chunk-final states across chunks
//   chunk_state_simt / chunk_scan_simt
//                         float32-accurate chunk kernels (the fp32 I/O path and
//                         shapes outside the tensor-core kernels' envelope)
//   multistep_kernel      K-token verification decode from a cached state
#pragma once

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
// K-token multi-step decode ("Mamba in the Llama", 推测解码, MultiStep).
// A block of 128 threads serves two items (heads 2 blockIdx.x and +1 of batch
// row b, p-slice of PS columns); 64 threads per item.  Thread (r, q) of an item
// handles the 4 columns 4q..4q+3 of state rows r, r + R, r + 2R, ...
// (R = 64 / (PS/4) row groups) and streams them: a row's 4 values are
// advanced through the K tokens (h = a h + B x^T; written to h_j after j
// tokens and to h_K after K) and add C_k[n] h to the thread's y partials,
// which stay in registers; loads run four rows ahead.  y = sum over rows
// (warp shuffles + shared memory) + D x.  The state is never held whole
// (42 MB of state would not fit the register file), so the whole grid is
// resident at once.
// dynamic smem per item: B[K][N], C[K][N], x[K][PS], a[16], y partials [K][2][PS].
// ----------------------------------------------------------------------------
constexpr int kMsThreads = 128;
// floats of shared memory per item: B, C [K][N], x [K][PS], decays, y partials
// [K][2][PS]; verify adds the previous drafts' B [KP][N], x [KP][PS], decays.
__host__ __device__ constexpr int ms_item_floats(int K, int N, int PS, bool verify, int KP = 0) {
  return 2 * K * N + K * PS + 16 + K * 2 * PS + (verify ? KP * N + KP * PS + 16 : 0);
}
constexpr int kMsItemThreads = 64;
constexpr int kMsMaxK = 16;

// KT: compile-time bound on K (8 or 16), K <= KT.  NC / PSC: the state size N
// and the column slice PS when fixed at compile time (0: taken from the
// arguments); with both fixed every shared-memory index of the row loop is a
// constant offset, which removes most of its integer work.
//
// VF (verify): the fused recompute + multistep + cache step ("Mamba in the
// Llama", 硬件特定优化: the verifier first recomputes the previous steps from
// the cache, then decodes the new drafts, then caches, in one kernel).  The
// cache h_cache then holds the state before the previous call's KP drafts
// (xp, dtp, Bp); jacc[b] of them were accepted.  Each state row is advanced
// through those jacc[b] tokens, stored to h_next (the next call's cache),
// and then through the K new drafts for y; h_j and h_K are not written.  Per
// row that is one state read and one state write instead of one and two.
template <typename IO, int KT, int NC = 0, int PSC = 0, bool VF = false>
__global__ void __launch_bounds__(128, 5) multistep_kernel(
    const IO *__restrict__ x, const float *__restrict__ dt, const float *__restrict__ A,
    const IO *__restrict__ Bm, const IO *__restrict__ Cm, const float *__restrict__ D,
    const float *__restrict__ h_cache, const int32_t *__restrict__ jacc, IO *__restrict__ y,
    float *__restrict__ h_j, float *__restrict__ h_K, int K, int H, int GB, int GC, int N_arg,
    int P, int PS_arg, int softplus, const IO *__restrict__ xp, const float *__restrict__ dtp,
    const IO *__restrict__ Bp, float *__restrict__ h_next, int KP) {
  const int N = NC ? NC : N_arg;
  const int PS = PSC ? PSC : PS_arg;
  extern __shared__ float sm_ms[];
  const int item = threadIdx.x / kMsItemThreads;  // 0 or 1
  const int h = 2 * blockIdx.x + item, b = blockIdx.y, p0 = blockIdx.z * PS;
  const int tid = threadIdx.x % kMsItemThreads, lane = threadIdx.x & 31;
  const int warp = tid >> 5;  // warp within the item: 0 or 1
  const int item_floats = ms_item_floats(K, N, PS, VF, KP);
  float *sB = sm_ms + item * item_floats;
  float *sC = sB + K * N;
  float *sx = sC + K * N;
  float *sa = sx + K * PS;
  float *red = sa + kMsMaxK;
  float *sBp = red + K * 2 * PS;  // verify: previous drafts' B, x and decays
  float *sxp = sBp + KP * N;
  float *sap = sxp + KP * PS;
  const bool live = h < H;
  const int hh = live ? h : H - 1;
  const int gb = hh / (H / GB), gc = hh / (H / GC);
  const int TP = PS / 4, R = kMsItemThreads / TP;
  const int q = tid % TP, r = tid / TP;

  for (int i = tid; i < K * N; i += kMsItemThreads) {
    const int k = i / N, n = i % N;
    sB[i] = to_f32(Bm[((static_cast<int64_t>(b) * K + k) * GB + gb) * N + n]);
    sC[i] = to_f32(Cm[((static_cast<int64_t>(b) * K + k) * GC + gc) * N + n]);
  }
  for (int i = tid; i < K * PS; i += kMsItemThreads) {
    const int k = i / PS, p = i % PS;
    sx[i] = to_f32(x[((static_cast<int64_t>(b) * K + k) * H + hh) * P + p0 + p]);
  }
  if (tid < K) {
    const float z = dt[(static_cast<int64_t>(b) * K + tid) * H + hh];
    sa[tid] = expf((softplus ? softplus_f32(z) : z) * A[hh]);
  }
  if (VF) {
    for (int i = tid; i < KP * N; i += kMsItemThreads) {
      const int k = i / N, n = i % N;
      sBp[i] = to_f32(Bp[((static_cast<int64_t>(b) * KP + k) * GB + gb) * N + n]);
    }
    for (int i = tid; i < KP * PS; i += kMsItemThreads) {
      const int k = i / PS, p = i % PS;
      sxp[i] = to_f32(xp[((static_cast<int64_t>(b) * KP + k) * H + hh) * P + p0 + p]);
    }
    if (tid < KP) {
      const float z = dtp[(static_cast<int64_t>(b) * KP + tid) * H + hh];
      sap[tid] = expf((softplus ? softplus_f32(z) : z) * A[hh]);
    }
  }
  int jb = jacc[b];
  if (jb < 0 || jb > (VF ? KP : K)) {
    if (tid == 0 && h == 0 && blockIdx.z == 0) report_error(kDevBadJ);
    jb = -1;
  }
  __syncthreads();
  // verify: a batch row whose accepted count is out of range gets no outputs
  const bool run = !VF || jb >= 0;

  float4 yp[KT];
#pragma unroll
  for (int k = 0; k < KT; ++k) yp[k] = make_float4(0.f, 0.f, 0.f, 0.f);

  if (live && run) {
    const int64_t base = (static_cast<int64_t>(b) * H + h) * N * P + p0 + 4 * q;
    const int rows = N / R;
    constexpr int PF = 4;  // rows in flight
    float4 buf[PF];
#pragma unroll
    for (int u = 0; u < PF; ++u)
      if (u < rows) buf[u] = __ldcs(reinterpret_cast<const float4 *>(h_cache + base + static_cast<int64_t>(r + R * u) * P));
    for (int i0 = 0; i0 < rows; i0 += PF) {
#pragma unroll
      for (int u = 0; u < PF; ++u) {
        const int i = i0 + u;
        if (i < rows) {
          const int n = r + R * i;
          float4 st = buf[u];
          if (i + PF < rows)
            buf[u] = __ldcs(reinterpret_cast<const float4 *>(h_cache + base + static_cast<int64_t>(n + R * PF) * P));
          const int64_t off = base + static_cast<int64_t>(n) * P;
          if (VF) {
            // recompute the accepted previous drafts, then cache the result
#pragma unroll
            for (int k = 0; k < kMsMaxK; ++k) {
              if (k < jb) {
                const float bn = sBp[k * N + n], a = sap[k];
                const float4 xk = *reinterpret_cast<const float4 *>(sxp + k * PS + 4 * q);
                st.x = fmaf(a, st.x, bn * xk.x);
                st.y = fmaf(a, st.y, bn * xk.y);
                st.z = fmaf(a, st.z, bn * xk.z);
                st.w = fmaf(a, st.w, bn * xk.w);
              }
            }
            *reinterpret_cast<float4 *>(h_next + off) = st;
          }
          // h_j with ordinary (L2-resident) stores: a speculative decode step
          // usually continues from it, so the next call finds it in L2
          if (!VF && jb == 0) *reinterpret_cast<float4 *>(h_j + off) = st;
#pragma unroll
          for (int k = 0; k < KT; ++k) {
            if (k < K) {
              const float bn = sB[k * N + n], cn = sC[k * N + n], a = sa[k];
              const float4 xk = *reinterpret_cast<const float4 *>(sx + k * PS + 4 * q);
              st.x = fmaf(a, st.x, bn * xk.x);
              st.y = fmaf(a, st.y, bn * xk.y);
              st.z = fmaf(a, st.z, bn * xk.z);
              st.w = fmaf(a, st.w, bn * xk.w);
              yp[k].x = fmaf(cn, st.x, yp[k].x);
              yp[k].y = fmaf(cn, st.y, yp[k].y);
              yp[k].z = fmaf(cn, st.z, yp[k].z);
              yp[k].w = fmaf(cn, st.w, yp[k].w);
              if (!VF && k + 1 == jb) *reinterpret_cast<float4 *>(h_j + off) = st;
            }
          }
          if (!VF) __stcs(reinterpret_cast<float4 *>(h_K + off), st);
        }
      }
    }
  }
  // reduce the y partials over row groups: lanes q, q + TP, ... of a warp, then 2 warps
#pragma unroll
  for (int k = 0; k < KT; ++k) {
    if (k < K) {
      float4 v = yp[k];
      for (int off = TP; off < 32; off <<= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, off);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, off);
        v.z += __shfl_xor_sync(0xffffffffu, v.z, off);
        v.w += __shfl_xor_sync(0xffffffffu, v.w, off);
      }
      if (lane < TP) *reinterpret_cast<float4 *>(red + (k * 2 + warp) * PS + 4 * lane) = v;
    }
  }
  __syncthreads();
  if (!live || !run) return;
  const float Dh = D ? D[h] : 0.f;
  for (int i = tid; i < K * PS; i += kMsItemThreads) {
    const int k = i / PS, p = i % PS;
    const float acc = red[(k * 2) * PS + p] + red[(k * 2 + 1) * PS + p];
    y[((static_cast<int64_t>(b) * K + k) * H + h) * P + p0 + p] = from_f32<IO>(acc + Dh * sx[i]);
  }
}

}  // namespace ssd
