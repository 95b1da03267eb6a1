// ssd_api.cu -- host side of libssd: argument validation, workspace layout,
// TMA descriptor encoding and kernel launches behind the C ABI of ssd.h.
//
// ssd_fwd runs the four steps of the chunked SSD algorithm (Mamba-2 page,
// section "SSD算法" and "深入解析分块与状态传递机制") as four kernels on the
// caller's stream:
//   0 dt_cumsum      softplus(dt) * A, in-chunk inclusive running sums
//   1 chunk_state    chunk-final states from zero initial state (green)
//   2 state_passing  scan of those states across chunks (yellow)
//   3 chunk_scan     diagonal blocks (orange) + output from the true initial
//                    state (blue) + D skip
// With bf16 I/O and a shape inside the tensor-core envelope (N = 128;
// Q in {128, 256}; P = 64, or P = 128 with Q = 128) steps 1 and 3 run on
// tcgen05 tensor cores; otherwise (fp32 I/O, other shapes) they run as
// float32 CUDA-core kernels.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>
#include <utility>

#include "../../include/ssd.h"
#include "ssd_cp.cuh"
#include "ssd_fused_hb.cuh"
#include "ssd_kernels.cuh"
#include "ssd_scan.cuh"
#include "ssd_scan_hb.cuh"
#include "ssd_selftest.cuh"
#include "ssd_state_hb.cuh"
#include "ssd_state.cuh"
#include "ssd_tc.cuh"

namespace {

using ssd::kTcN;

constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 64;  // device ordinals with per-device set-up state
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Plan {
  int64_t b, T, H, P, N, GB, GC;
  int Q, nc;
  bool bf16, softplus, tc;
  size_t cs_off, S_off, Hin_off, total;
  // tensor-core path: sequence segments of the state pass (1: none) and the
  // workspace of their hand-off (segment final states, decay products).  The
  // first `whole` items run unsplit; the hand-off covers the (b, h) rows
  // seg_bh0 .. seg_bh0 + seg_rows - 1 of the split ones
  int nseg = 1, cps = 0;
  int64_t whole = 0, seg_bh0 = 0, seg_rows = 0;
  size_t Fseg_off = 0, Lseg_off = 0, Dc_off = 0;
  // 256-token chunks, 64-wide heads, one (B, C) group: the chunk-state kernel
  // records per (b, chunk, head) whether the chunk's decay allows the
  // head-pair form (one byte each), and chunk_scan_hb computes the heads two
  // per MMA or, flagged, one by one
  bool hb = false;
  size_t flags_off = 0;
  // the same shapes: chunk states two heads per MMA (chunk_state_hb), after
  // dt_decay_kernel has written the per-token log2 decays [b, H, T] (u_off)
  bool state_hb = false;
  size_t u_off = 0;
  // the one-pass kernel (chunk_fused_hb) for the same shapes and for 128-token
  // chunks of 128-wide heads: items of fused_hp heads (2: two 64-wide heads
  // of one (B, C) group; 1: one 128-wide head), fused_spc 128-token stages
  // per chunk; with its prepass when items are split (nseg > 1; whole, cps,
  // seg_bh0, seg_rows, Fseg_off, Lseg_off as above) and the flagged-head pass
  // after it; Hin, flags and u then hold the flagged (chunk, head) units only
  bool fused = false;
  int fused_hp = 2, fused_spc = 2;
};

int num_sms();
int scan_pairs_per_cta(const Plan &pl, int num_sms);
// chunk_scan_hb pays a per-CTA set-up (C B^T, mask, C into tensor memory)
// and a pipeline fill; below this many head pairs per CTA the per-head
// kernel is faster (e.g. 4096-token windows of one sequence: 5 pairs)
constexpr int kHbMinPairs = 10;

// Segments of the tensor-core state pass.  Its CTAs walk their chunks one after
// another, two per SM; when the (batch, head, slice) items leave SM slots idle
// the sequence is split so that every slot works on a segment of at least four
// chunks.
// chunk_state_hb: one CTA per SM, one per (batch, head pair).  With more items
// than SMs, the items of a last, partly filled wave are split instead (the
// full waves' items run whole), into segments of at least two chunks, so that
// the last wave takes a fraction of an item's time: e.g. 8 x 2048 tokens x 40
// head pairs on 148 SMs = two full waves + 24 items, split in four.
void plan_segments(Plan *pl) {
  const int64_t items = pl->state_hb ? pl->b * ((pl->H + 1) / 2) : pl->b * pl->H * (pl->P / 64);
  const int64_t slots = (pl->state_hb ? 1 : 2) * static_cast<int64_t>(num_sms());
  int64_t nseg = 1, whole = 0;
  if (items < slots) {
    nseg = std::min<int64_t>(slots / items, pl->nc / 4);
  } else if (pl->state_hb && items % slots) {
    whole = items / slots * slots;
    nseg = std::min<int64_t>(slots / (items - whole), pl->nc / 2);
  }
  nseg = std::max<int64_t>(nseg, 1);
  pl->cps = static_cast<int>((pl->nc + nseg - 1) / nseg);
  pl->nseg = (pl->nc + pl->cps - 1) / pl->cps;
  pl->whole = pl->nseg > 1 ? whole : items;
  // the split items' (b, h) rows: from the first split item's first head on
  if (pl->state_hb) {
    const int64_t npairs = (pl->H + 1) / 2;
    pl->seg_bh0 = pl->whole / npairs * pl->H + 2 * (pl->whole % npairs);
  } else {
    pl->seg_bh0 = 0;
  }
  pl->seg_rows = pl->b * pl->H - pl->seg_bh0;
}

// Segments of the one-pass kernel: one CTA per SM, one per item (batch row,
// head pair or 128-wide head).  With more items than SMs the items of a last,
// partly filled wave are split (the full waves' items run whole); with fewer,
// every item is, when at least two segments fit; a split item's nseg segments
// of cps chunks start from the states the prepass computes.  E.g. 8 x 40 head
// pairs on 148 SMs: two full waves + 24 items in four segments of two chunks;
// 4 x 32 heads: one wave of 128 whole items.
void plan_fused(Plan *pl) {
  const int64_t ipb = (pl->H + pl->fused_hp - 1) / pl->fused_hp, items = pl->b * ipb;
  const int64_t slots = num_sms();
  int64_t nseg = 1, whole = items;
  if (items < slots) {
    nseg = std::min<int64_t>(slots / items, pl->nc);
    whole = 0;
  } else if (items % slots) {
    whole = items / slots * slots;
    nseg = std::min<int64_t>(slots / (items - whole), pl->nc);
  }
  if (nseg <= 1) {
    nseg = 1;
    whole = items;
  }
  pl->cps = static_cast<int>((pl->nc + nseg - 1) / nseg);
  pl->nseg = (pl->nc + pl->cps - 1) / pl->cps;
  pl->whole = pl->nseg > 1 ? whole : items;
  pl->seg_bh0 = pl->whole / ipb * pl->H + pl->fused_hp * (pl->whole % ipb);
  pl->seg_rows = pl->b * pl->H - pl->seg_bh0;
}

bool valid_dim(int64_t v) { return v >= 1 && v <= (int64_t(1) << 31) - 1; }

// Shared shape checks of both calls.  Returns SSD_OK or the error to report.
ssd_status check_dims(const ssd_dims *d) {
  if (!d) return SSD_ERR_INVALID_ARG;
  if (!valid_dim(d->batch) || !valid_dim(d->seqlen) || !valid_dim(d->nheads) ||
      !valid_dim(d->headdim) || !valid_dim(d->dstate) || !valid_dim(d->ngroups_b) ||
      !valid_dim(d->ngroups_c))
    return SSD_ERR_INVALID_ARG;
  if (d->io_dtype != SSD_F32 && d->io_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
  if (d->dt_softplus != 0 && d->dt_softplus != 1) return SSD_ERR_INVALID_ARG;
  if (d->nheads % d->ngroups_b || d->nheads % d->ngroups_c) return SSD_ERR_INVALID_ARG;
  if (d->headdim % 16 || d->dstate % 16 || d->headdim > 256 || d->dstate > 256)
    return SSD_ERR_UNSUPPORTED;
  return SSD_OK;
}

ssd_status make_plan(const ssd_dims *d, int32_t chunk, Plan *pl) {
  ssd_status st = check_dims(d);
  if (st != SSD_OK) return st;
  if (chunk != 64 && chunk != 128 && chunk != 256) return SSD_ERR_UNSUPPORTED;
  pl->b = d->batch;
  pl->T = d->seqlen;
  pl->H = d->nheads;
  pl->P = d->headdim;
  pl->N = d->dstate;
  pl->GB = d->ngroups_b;
  pl->GC = d->ngroups_c;
  pl->Q = chunk;
  pl->nc = static_cast<int>((d->seqlen + chunk - 1) / chunk);
  pl->bf16 = d->io_dtype == SSD_BF16;
  pl->softplus = d->dt_softplus != 0;
  pl->tc = pl->bf16 && pl->N == kTcN &&
           ((pl->Q == 256 && pl->P == 64) || (pl->Q == 128 && (pl->P == 64 || pl->P == 128)));
  // grid limits: gridDim.y / gridDim.z <= 65535
  if (pl->nc * ((pl->Q + 31) / 32) > 65535 || pl->b > 65535 || pl->H > 65535)
    return SSD_ERR_UNSUPPORTED;
  if (pl->b * pl->nc * pl->H > (int64_t(1) << 31) - 1) return SSD_ERR_UNSUPPORTED;
  const size_t states = static_cast<size_t>(pl->b) * pl->nc * pl->H * pl->N * pl->P;
  if (pl->tc) {
    // tensor-core path: the chunk initial states (bf16) go through HBM, plus,
    // for a segmented state pass, each segment's final state and decays
    pl->cs_off = pl->S_off = 0;
    pl->Hin_off = 0;
    pl->total = align_up(states * 2);
    const bool hb_shape = pl->Q == 256 && pl->P == 64 && pl->GB == 1 && pl->GC == 1;
    // The one-pass kernel when the (batch row, head pair) items fill at least
    // one wave of the SMs; with fewer (a long sequence over few heads) every
    // item would be split, and the two-pass kernels, whose chunk scan runs
    // over all chunks in parallel, are faster.  SSD_FUSED=1 / =0 forces one
    // or the other, as does a forced chunk-scan form (SSD_CHUNK_SCAN) the
    // two-pass kernels (for tests and comparisons; the results agree within
    // the tolerance).
    // 128-token chunks of 128-wide heads (any groups) take it, one head per
    // item, as soon as the items fill half the SMs.
    const char *fz = std::getenv("SSD_FUSED");
    const char *force = std::getenv("SSD_CHUNK_SCAN");
    const bool wide_shape = pl->Q == 128 && pl->P == 128;
    pl->fused_hp = hb_shape ? 2 : 1;
    pl->fused_spc = pl->Q / 128;
    const int64_t items = pl->b * ((pl->H + pl->fused_hp - 1) / pl->fused_hp);
    const bool fill = hb_shape ? items >= num_sms() : 2 * items >= num_sms();
    pl->fused = (hb_shape || wide_shape) && !(force && *force) &&
                (fz && *fz ? std::strcmp(fz, "0") != 0 : fill);
    pl->state_hb = hb_shape && !pl->fused;
    if (pl->fused) plan_fused(pl);
    else plan_segments(pl);
    if (pl->nseg > 1) {
      if (pl->b * pl->nseg > 65535 || pl->seg_rows > 65535) return SSD_ERR_UNSUPPORTED;
      const size_t bh = static_cast<size_t>(pl->seg_rows);
      pl->Fseg_off = pl->total;
      pl->Lseg_off = pl->Fseg_off + align_up(bh * pl->nseg * pl->N * pl->P * sizeof(float));
      pl->Dc_off = pl->Lseg_off + align_up(bh * pl->nseg * sizeof(float));
      pl->total = pl->Dc_off + align_up(bh * pl->nc * sizeof(float));
    }
    if (pl->fused) {
      pl->flags_off = pl->total;
      pl->total += align_up(static_cast<size_t>(pl->b) * pl->nc * pl->H);
      pl->u_off = pl->total;
      pl->total += align_up(static_cast<size_t>(pl->b) * pl->H * pl->T * sizeof(float));
    } else if (hb_shape) {  // the flags are reserved for every such shape
      pl->flags_off = pl->total;
      pl->total += align_up(static_cast<size_t>(pl->b) * pl->nc * pl->H);
      // SSD_CHUNK_SCAN=pair / =head forces the choice (the same result either
      // way, within the tolerance; for tests and tuning)
      if (force && std::strcmp(force, "pair") == 0) pl->hb = true;
      else if (force && std::strcmp(force, "head") == 0) pl->hb = false;
      else pl->hb = scan_pairs_per_cta(*pl, num_sms()) >= kHbMinPairs;
      pl->u_off = pl->total;
      pl->total += align_up(static_cast<size_t>(pl->b) * pl->H * pl->T * sizeof(float));
    }
  } else {
    pl->cs_off = 0;
    pl->S_off = align_up(static_cast<size_t>(pl->b) * pl->H * pl->nc * pl->Q * sizeof(float));
    pl->Hin_off = pl->S_off + align_up(states * sizeof(float));
    pl->total = pl->Hin_off + align_up(states * sizeof(float));
  }
  return SSD_OK;
}

// ---------------------------------------------------------------------------
// TMA descriptors (driver entry point fetched through the runtime; no libcuda
// link needed).
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// bf16 tensor of rank r (dims innermost first, strides in bytes of dims 1..r-1),
// box `box`, 128-byte swizzle, zero fill outside the tensor.
bool encode_bf16(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims,
                 const cuuint64_t *strides, const cuuint32_t *box) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [b, T, G, W] bf16 tensor, tiles of [Q rows][64] at (w0, g, t0, b).
bool encode_btgw(CUtensorMap *m, const void *base, int64_t b, int64_t T, int64_t G, int64_t W,
                 int Q) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(G),
                              static_cast<cuuint64_t>(T), static_cast<cuuint64_t>(b)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(W * 2), static_cast<cuuint64_t>(G * W * 2),
                                 static_cast<cuuint64_t>(T * G * W * 2)};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(Q), 1};
  return encode_bf16(m, base, 4, dims, strides, box);
}

// Kernel attributes live in each device's context: the dynamic shared-memory
// limit of a kernel is raised once per (kernel, device), with that device
// current, before its first launch there.
template <auto Kernel>
bool ensure_smem(int bytes) {
  static std::mutex mu;
  static bool done[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (!done[dev]) {
    if (cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
      return false;
    done[dev] = true;
  }
  return true;
}

ssd_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

void record(void *const *events, int i, cudaStream_t s) {
  if (events && events[i]) cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s);
}

// Programmatic dependent launch (the device side is grid_dep_wait /
// grid_dep_trigger): the kernels after dt_decay_kernel on the head-pair path
// may start while the one before them finishes, so that their set-up (barrier
// and tensor-memory set-up, input loads, the chunk scan's C B^T) overlaps its
// tail.  Off for a call that records per-stage events (the stages would
// overlap) and when SSD_PDL=0.
bool pdl_on(void *const *events) {
  if (events) return false;
  const char *e = std::getenv("SSD_PDL");
  return !(e && std::strcmp(e, "0") == 0);
}

template <typename... KArgs, typename... Args>
ssd_status launch_dependent(bool pdl, void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...) != cudaSuccess) {
    cudaGetLastError();  // clear the recorded launch error
    return SSD_ERR_CUDA;
  }
  return launch_status();
}

// ---------------------------------------------------------------------------
// Stage launchers
// ---------------------------------------------------------------------------
ssd_status launch_cumsum(const Plan &pl, const float *dt, const float *A, float *cs,
                         cudaStream_t s) {
  dim3 grid(pl.nc, static_cast<unsigned>(pl.b), static_cast<unsigned>((pl.H + 31) / 32));
  switch (pl.Q) {
    case 64: ssd::dt_cumsum_kernel<64><<<grid, 256, 0, s>>>(dt, A, cs, pl.T, pl.H, pl.nc, pl.softplus); break;
    case 128: ssd::dt_cumsum_kernel<128><<<grid, 256, 0, s>>>(dt, A, cs, pl.T, pl.H, pl.nc, pl.softplus); break;
    default: ssd::dt_cumsum_kernel<256><<<grid, 256, 0, s>>>(dt, A, cs, pl.T, pl.H, pl.nc, pl.softplus); break;
  }
  return launch_status();
}

template <typename HT>
ssd_status launch_passing(const Plan &pl, const float *S, const float *cs, const float *h0,
                          HT *Hin, float *h_final, cudaStream_t s) {
  const int NP = static_cast<int>(pl.N * pl.P);
  dim3 grid((NP / 4 + 255) / 256, static_cast<unsigned>(pl.H), static_cast<unsigned>(pl.b));
  ssd::state_passing_kernel<HT><<<grid, 256, 0, s>>>(S, cs, h0, Hin, h_final, static_cast<int>(pl.H),
                                                     pl.nc, pl.Q, NP);
  return launch_status();
}

template <typename IO>
ssd_status launch_state_simt(const Plan &pl, const void *x, const void *B, const float *cs,
                             float *S, cudaStream_t s) {
  const int64_t tiles = ((pl.N + 63) / 64) * ((pl.P + 63) / 64) * pl.nc;
  dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(pl.H), static_cast<unsigned>(pl.b));
  ssd::chunk_state_simt<IO><<<grid, 256, 0, s>>>(
      static_cast<const IO *>(x), static_cast<const IO *>(B), cs, S, pl.T, static_cast<int>(pl.H),
      static_cast<int>(pl.GB), static_cast<int>(pl.N), static_cast<int>(pl.P), pl.Q, pl.nc);
  return launch_status();
}

template <typename IO, typename HT>
ssd_status launch_scan_simt(const Plan &pl, const void *x, const void *B, const void *C,
                            const float *cs, const HT *Hin, const float *D, void *y,
                            cudaStream_t s) {
  const int smem = ssd::scan_simt_smem_floats(pl.Q, static_cast<int>(pl.N)) * 4;
  auto k = ssd::chunk_scan_simt<IO, HT>;
  if (!ensure_smem<ssd::chunk_scan_simt<IO, HT>>(ssd::scan_simt_smem_floats(256, 256) * 4)) return SSD_ERR_CUDA;
  const int64_t blocks = ((pl.Q + 31) / 32) * ((pl.P + 63) / 64) * pl.nc;
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(pl.H), static_cast<unsigned>(pl.b));
  k<<<grid, 256, smem, s>>>(static_cast<const IO *>(x), static_cast<const IO *>(B),
                            static_cast<const IO *>(C), cs, Hin, D, static_cast<IO *>(y), pl.T,
                            static_cast<int>(pl.H), static_cast<int>(pl.GB),
                            static_cast<int>(pl.GC), static_cast<int>(pl.N),
                            static_cast<int>(pl.P), pl.Q, pl.nc);
  return launch_status();
}

int num_sms() {
  static std::mutex mu;
  static int n[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lock(mu);
  if (n[dev] <= 0 &&
      (cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
       n[dev] <= 0))
    n[dev] = 148;
  return n[dev];
}

template <int Q>
ssd_status launch_state_pass(const Plan &pl, const CUtensorMap &mB, const CUtensorMap &mX,
                             const float *dt, const float *A, const float *u, const float *h0,
                             __nv_bfloat16 *Hin,
                             float *h_final, float *Fseg, float *Lseg, float *Dc,
                             uint8_t *flags, void *const *events, int ev, cudaStream_t s) {
  if (pl.state_hb) {
    // two heads per MMA; mB / mX are the 128-row tile maps here
    auto k = ssd::chunk_state_hb;
    if (!ensure_smem<ssd::chunk_state_hb>(ssd::StateHB::kBytes)) return SSD_ERR_CUDA;
    const int64_t items = pl.b * ((pl.H + 1) / 2);
    const int64_t ctas = pl.whole + (items - pl.whole) * (pl.nseg > 1 ? pl.nseg : 1);
    const ssd_status st = launch_dependent(
        pdl_on(events), k, dim3(static_cast<unsigned>(ctas)), dim3(ssd::kShThreads),
        ssd::StateHB::kBytes, s, mB, mX, u, h0, Hin, h_final, pl.T, static_cast<int>(pl.H), pl.nc,
        static_cast<int>(pl.whole), pl.nseg, pl.cps, pl.seg_bh0, Fseg, Lseg, Dc, flags);
    if (st != SSD_OK) return st;
  } else {
    using L = ssd::StatePass<Q>;
    auto k = ssd::chunk_state_pass_tc<Q>;
    if (!ensure_smem<ssd::chunk_state_pass_tc<Q>>(L::kBytes)) return SSD_ERR_CUDA;
    dim3 grid(static_cast<unsigned>(pl.P / L::PS), static_cast<unsigned>(pl.H),
              static_cast<unsigned>(pl.b * pl.nseg));
    k<<<grid, L::kThreads, L::kBytes, s>>>(mB, mX, dt, A, h0, Hin, h_final, pl.T,
                                           static_cast<int>(pl.H), static_cast<int>(pl.GB), pl.nc,
                                           static_cast<int>(pl.P), pl.softplus, pl.nseg, pl.cps,
                                           Fseg, Lseg, Dc);
  }
  if (launch_status() != SSD_OK || pl.nseg == 1) return launch_status();
  record(events, ev + 1, s);
  const int NP = static_cast<int>(pl.N * pl.P);
  dim3 g2(static_cast<unsigned>((NP / 4 + 255) / 256), static_cast<unsigned>(pl.seg_rows));
  return launch_dependent(pl.state_hb && pdl_on(events), ssd::state_fixup_kernel, g2, dim3(256),
                          0, s, Fseg, Lseg, Dc, Hin, h_final, static_cast<int>(pl.H), pl.nc,
                          pl.cps, pl.nseg, NP, pl.seg_bh0);
}

// One instance of multistep_kernel: KT bounds K (and k_prev in verify mode);
// the shared memory is sized for those bounds.
template <typename IO, int KT, int NC = 0, bool KX = false, bool VF = false>
ssd_status launch_ms(dim3 grid, const ssd_dims *d, int KP, const void *xp, const float *dtp,
                     const void *Bp, const int32_t *j, const void *x, const float *dt,
                     const float *A, const void *B, const void *C, const float *D,
                     const float *h_cache, void *y, float *h_j, float *h_K, float *h_next,
                     int PS, cudaStream_t s) {
  auto k = ssd::multistep_kernel<IO, KT, KT, NC, KX, VF>;
  const int64_t smem = ssd::ms_smem_bytes(KT, KT, static_cast<int>(d->dstate), PS, VF,
                                          static_cast<int>(sizeof(IO)));
  if (smem > 227 * 1024) return SSD_ERR_UNSUPPORTED;
  if (!ensure_smem<ssd::multistep_kernel<IO, KT, KT, NC, KX, VF>>(227 * 1024)) return SSD_ERR_CUDA;
  k<<<grid, ssd::kMsThreads, static_cast<size_t>(smem), s>>>(
      static_cast<const IO *>(x), dt, A, static_cast<const IO *>(B), static_cast<const IO *>(C),
      D, h_cache, j, static_cast<IO *>(y), h_j, h_K, static_cast<int>(d->seqlen),
      static_cast<int>(d->nheads), static_cast<int>(d->ngroups_b), static_cast<int>(d->ngroups_c),
      static_cast<int>(d->dstate), static_cast<int>(d->headdim), PS, d->dt_softplus,
      static_cast<const IO *>(xp), dtp, static_cast<const IO *>(Bp), h_next, KP,
      static_cast<int>(d->batch * d->nheads));
  return launch_status();
}

// The instance for a shape: the decode shape of the Mamba-2 layers (bf16,
// N = 128, K = 8, k_prev <= 8) with N and K fixed at compile time; a verify
// call of fewer new tokens at N = 128 (the draft model's step, K = 1) with N
// fixed; else a generic one.
template <bool VF>
ssd_status dispatch_ms(dim3 grid, const ssd_dims *d, int KP, const void *xp, const float *dtp,
                       const void *Bp, const int32_t *j, const void *x, const float *dt,
                       const float *A, const void *B, const void *C, const float *D,
                       const float *h_cache, void *y, float *h_j, float *h_K, float *h_next,
                       int PS, cudaStream_t s) {
  const bool bf16 = d->io_dtype == SSD_BF16;
  const bool small = d->seqlen <= 8 && (!VF || KP <= 8);
#define SSD_MS_ARGS grid, d, KP, xp, dtp, Bp, j, x, dt, A, B, C, D, h_cache, y, h_j, h_K, h_next, PS, s
  if (bf16 && small && d->seqlen == 8 && d->dstate == 128)
    return launch_ms<__nv_bfloat16, 8, 128, true, VF>(SSD_MS_ARGS);
  if (VF && bf16 && small && d->dstate == 128)  // the draft model's short steps
    return launch_ms<__nv_bfloat16, 8, 128, false, VF>(SSD_MS_ARGS);
  if (bf16)
    return small ? launch_ms<__nv_bfloat16, 8, 0, false, VF>(SSD_MS_ARGS)
                 : launch_ms<__nv_bfloat16, 16, 0, false, VF>(SSD_MS_ARGS);
  return small ? launch_ms<float, 8, 0, false, VF>(SSD_MS_ARGS)
               : launch_ms<float, 16, 0, false, VF>(SSD_MS_ARGS);
#undef SSD_MS_ARGS
}

// Heads per CTA of chunk_scan_hl: trades the per-group C B^T product (paid
// once per CTA) against wave quantisation over the SMs.
int scan_heads_per_cta(const Plan &pl, int num_sms) {
  const bool shared = pl.GB == 1 && pl.GC == 1;
  const double t_head = 1.0, t_group = shared ? 1.5 : 0.0;
  int best = 1;
  double best_cost = 1e300;
  for (int hp = 1; hp <= 16 && hp <= pl.H; ++hp) {
    const int64_t ctas = ((pl.H + hp - 1) / hp) * pl.nc * pl.b;
    const double waves = static_cast<double>((ctas + num_sms - 1) / num_sms);
    const double groups = shared ? 1.0 : static_cast<double>(hp);
    const double cost = waves * (hp * t_head + groups * (shared ? t_group : 0.5));
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = hp;
    }
  }
  return best;
}

template <int Q, int P>
ssd_status launch_scan_hl(const Plan &pl, const CUtensorMap &mC32, const CUtensorMap &mB,
                          const CUtensorMap &mX, const CUtensorMap &mH, const CUtensorMap &mY,
                          const float *dt, const float *A, const float *D, cudaStream_t s) {
  using L = ssd::ScanHL<Q, P>;
  auto k = ssd::chunk_scan_hl<Q, P>;
  if (!ensure_smem<ssd::chunk_scan_hl<Q, P>>(L::kBytes)) return SSD_ERR_CUDA;
  const int hpc = scan_heads_per_cta(pl, num_sms());
  dim3 grid(static_cast<unsigned>((pl.H + hpc - 1) / hpc), pl.nc, static_cast<unsigned>(pl.b));
  k<<<grid, L::kThreads, L::kBytes, s>>>(mC32, mB, mX, mH, mY, dt, A, D, pl.T,
                                         static_cast<int>(pl.H), static_cast<int>(pl.GB),
                                         static_cast<int>(pl.GC), pl.nc, hpc, pl.softplus);
  return launch_status();
}

// Head pairs per CTA of chunk_scan_hb: the per-CTA C B^T product and mask
// (~1.75 pairs of work) against wave quantisation.
int scan_pairs_per_cta(const Plan &pl, int num_sms) {
  const int64_t pairs = (pl.H + 1) / 2;
  int best = 1;
  double best_cost = 1e300;
  for (int pp = 1; pp <= std::min<int64_t>(pairs, ssd::kHbMaxPairs); ++pp) {
    const int64_t ctas = ((pairs + pp - 1) / pp) * pl.nc * pl.b;
    const double waves = static_cast<double>((ctas + num_sms - 1) / num_sms);
    const double cost = waves * (pp + 1.75);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = pp;
    }
  }
  return best;
}

// Head sets of the flagged-head items of chunk_scan_hb's launch: each item
// scans every kFlaggedSets-th head of its (batch, chunk) for the few the
// chunk-state kernel flagged (at most ScanHL<256, 64>::kMaxFlaggedHeads).
constexpr int kFlaggedSets = 4;

ssd_status launch_scan_hb(const Plan &pl, const CUtensorMap &mC32, const CUtensorMap &mB,
                          const CUtensorMap &mX, const CUtensorMap &mH, const CUtensorMap &mY,
                          const CUtensorMap &mY128,
                          const float *dt, const float *A, const float *D, const float *u,
                          const uint8_t *flags, bool pdl, cudaStream_t s) {
  auto k = ssd::chunk_scan_hb;
  if (!ensure_smem<ssd::chunk_scan_hb>(ssd::kHbLaunchBytes)) return SSD_ERR_CUDA;
  const int pp = scan_pairs_per_cta(pl, num_sms());
  const int64_t pairs = (pl.H + 1) / 2;
  const int hb_ranges = static_cast<int>((pairs + pp - 1) / pp);
  const int64_t kmax = ssd::ScanHL<256, 64>::kMaxFlaggedHeads;
  const int flagged_sets =
      static_cast<int>(std::max<int64_t>(kFlaggedSets, (pl.H + kmax - 1) / kmax));
  const int64_t blocks = (static_cast<int64_t>(hb_ranges) + flagged_sets) * pl.nc * pl.b;
  if (blocks > (int64_t(1) << 31) - 1) return SSD_ERR_UNSUPPORTED;
  return launch_dependent(pdl, k, dim3(static_cast<unsigned>(blocks)), dim3(ssd::kHbThreads),
                          ssd::kHbLaunchBytes, s, mC32, mB, mX, mH, mY, mY128, dt, A, D, u, flags,
                          pl.T,
                          static_cast<int>(pl.b), static_cast<int>(pl.H), pl.nc, pp, hb_ranges,
                          flagged_sets, pl.softplus);
}

// The one-pass path: [prepass of split items] -> chunk_fused_hb -> the
// flagged (chunk, head) units by the per-head body (chunk_scan_hb's flagged
// items alone).  Each kernel after the first is a programmatic dependent of
// the one before (pdl); the first waits for everything before it.
template <int HP, int SPC, int Q, int P>
ssd_status launch_fused_t(const Plan &pl, const void *x, const float *dt, const float *A,
                          const void *B, const void *C, const float *D, const float *h0, void *y,
                          float *h_final, uint8_t *ws, void *const *events, cudaStream_t s) {
  CUtensorMap mX, mB, mC, mY, mC32, mBQ, mXQ, mH, mYQ;
  const cuuint64_t hdims[3] = {static_cast<cuuint64_t>(pl.P), static_cast<cuuint64_t>(pl.N),
                               static_cast<cuuint64_t>(pl.b * pl.nc * pl.H)};
  const cuuint64_t hstr[2] = {static_cast<cuuint64_t>(pl.P * 2),
                              static_cast<cuuint64_t>(pl.N * pl.P * 2)};
  const cuuint32_t hbox[3] = {64, static_cast<cuuint32_t>(pl.N), 1};
  __nv_bfloat16 *Hin = reinterpret_cast<__nv_bfloat16 *>(ws + pl.Hin_off);
  if (!encode_btgw(&mX, x, pl.b, pl.T, pl.H, pl.P, 128) ||
      !encode_btgw(&mB, B, pl.b, pl.T, pl.GB, pl.N, 128) ||
      !encode_btgw(&mC, C, pl.b, pl.T, pl.GC, pl.N, 128) ||
      !encode_btgw(&mY, y, pl.b, pl.T, pl.H, pl.P, 128) ||
      !encode_btgw(&mC32, C, pl.b, pl.T, pl.GC, pl.N, 32) ||
      !encode_btgw(&mBQ, B, pl.b, pl.T, pl.GB, pl.N, pl.Q) ||
      !encode_btgw(&mXQ, x, pl.b, pl.T, pl.H, pl.P, pl.Q) ||
      !encode_btgw(&mYQ, y, pl.b, pl.T, pl.H, pl.P, pl.Q) ||
      !encode_bf16(&mH, Hin, 3, hdims, hstr, hbox))
    return SSD_ERR_CUDA;
  uint8_t *flags = ws + pl.flags_off;
  float *u = reinterpret_cast<float *>(ws + pl.u_off);
  float *Fseg = pl.nseg > 1 ? reinterpret_cast<float *>(ws + pl.Fseg_off) : nullptr;
  float *Lseg = pl.nseg > 1 ? reinterpret_cast<float *>(ws + pl.Lseg_off) : nullptr;
  const int64_t items = pl.b * ((pl.H + HP - 1) / HP);
  const int64_t split = items - pl.whole;
  const int H = static_cast<int>(pl.H), GB = static_cast<int>(pl.GB), GC = static_cast<int>(pl.GC);
  using L = ssd::FusedHB;
  if (!ensure_smem<ssd::chunk_fused_hb<true, HP, SPC>>(L::kBytes) ||
      !ensure_smem<ssd::chunk_fused_hb<false, HP, SPC>>(L::kBytes))
    return SSD_ERR_CUDA;
  int ev = 0;
  record(events, ev, s);
  ssd_status st;
  bool pdl = false;
  if (pl.nseg > 1) {
    const int64_t ctas = split * (pl.nseg - 1);
    st = launch_dependent(false, ssd::chunk_fused_hb<false, HP, SPC>,
                          dim3(static_cast<unsigned>(ctas)), dim3(ssd::kFuThreads), L::kBytes, s,
                          mX, mB, mC, mY, dt, A, D, h0, h_final, Hin, flags, u, pl.T, H, GB, GC,
                          pl.nc, pl.softplus ? 1 : 0, static_cast<int>(pl.whole), pl.nseg, pl.cps,
                          pl.seg_bh0, Fseg, Lseg, num_sms());
    if (st != SSD_OK) return st;
    record(events, ++ev, s);
    pdl = pdl_on(events);
  }
  const int64_t ctas = pl.whole + split * (pl.nseg > 1 ? pl.nseg : 0);
  st = launch_dependent(pdl, ssd::chunk_fused_hb<true, HP, SPC>, dim3(static_cast<unsigned>(ctas)),
                        dim3(ssd::kFuThreads), L::kBytes, s, mX, mB, mC, mY, dt, A, D, h0, h_final,
                        Hin, flags, u, pl.T, H, GB, GC, pl.nc, pl.softplus ? 1 : 0,
                        static_cast<int>(pl.whole), pl.nseg, pl.cps, pl.seg_bh0, Fseg, Lseg,
                        num_sms());
  if (st != SSD_OK) return st;
  record(events, ++ev, s);
  // the flagged (chunk, head) units, head by head (blocks that find none exit)
  using LH = ssd::ScanHL<Q, P>;
  if (!ensure_smem<ssd::chunk_scan_flagged<Q, P>>(LH::kBytes)) return SSD_ERR_CUDA;
  // head sets per (batch row, chunk): as many as still fit the launch in one
  // round of the SMs (its blocks take an SM each and nearly all of them only
  // read their flags), at least enough for kMaxFlaggedHeads heads a set
  const int64_t kmax = LH::kMaxFlaggedHeads;
  const int64_t fit = std::max<int64_t>(1, num_sms() / (static_cast<int64_t>(pl.nc) * pl.b));
  const int sets = static_cast<int>(
      std::max<int64_t>((pl.H + kmax - 1) / kmax, std::min<int64_t>(kFlaggedSets, fit)));
  const int64_t blocks = static_cast<int64_t>(sets) * pl.nc * pl.b;
  if (blocks > (int64_t(1) << 31) - 1) return SSD_ERR_UNSUPPORTED;
  st = launch_dependent(pdl_on(events), ssd::chunk_scan_flagged<Q, P>,
                        dim3(static_cast<unsigned>(blocks)), dim3(LH::kThreads), LH::kBytes, s,
                        mC32, mBQ, mXQ, mH, mYQ, dt, A, D, static_cast<const float *>(u),
                        static_cast<const uint8_t *>(flags), pl.T, H, GB, GC, pl.nc, sets,
                        pl.softplus ? 1 : 0);
  if (st != SSD_OK) return st;
  record(events, ++ev, s);
  return SSD_OK;
}

ssd_status launch_fused(const Plan &pl, const void *x, const float *dt, const float *A,
                        const void *B, const void *C, const float *D, const float *h0, void *y,
                        float *h_final, uint8_t *ws, void *const *events, cudaStream_t s) {
  if (pl.fused_hp == 2)
    return launch_fused_t<2, 2, 256, 64>(pl, x, dt, A, B, C, D, h0, y, h_final, ws, events, s);
  return launch_fused_t<1, 1, 128, 128>(pl, x, dt, A, B, C, D, h0, y, h_final, ws, events, s);
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Null, alignment and aliasing checks of a prefill call's buffers, as whole
// [b, T, ...] tensors of `d`; the workspace counts as an output of ws_used
// bytes.  Returns SSD_OK or SSD_ERR_INVALID_ARG; launches nothing.
ssd_status check_fwd_buffers(const ssd_dims *d, const void *x, const float *dt, const float *A,
                             const void *B, const void *C, const float *D, const float *h0,
                             const void *y, const float *h_final, const void *workspace,
                             size_t ws_used) {
  if (!x || !dt || !A || !B || !C || !y || !workspace) return SSD_ERR_INVALID_ARG;
  const void *ptrs[] = {x, dt, A, B, C, D, h0, y, h_final, workspace};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return SSD_ERR_INVALID_ARG;
  const size_t io = d->io_dtype == SSD_BF16 ? 2 : 4;
  const size_t bt = static_cast<size_t>(d->batch * d->seqlen);
  const size_t nx = bt * d->nheads * d->headdim * io;
  const size_t nB = bt * d->ngroups_b * d->dstate * io;
  const size_t nC = bt * d->ngroups_c * d->dstate * io;
  const size_t ndt = bt * d->nheads * 4;
  const size_t nst = static_cast<size_t>(d->batch * d->nheads * d->headdim * d->dstate) * 4;
  const size_t nh = static_cast<size_t>(d->nheads) * 4;
  struct Buf { const void *p; size_t n; };
  const Buf ins[] = {{x, nx}, {dt, ndt}, {A, nh}, {B, nB}, {C, nC}, {D, nh}, {h0, nst}};
  const Buf outs[] = {{y, nx}, {h_final, nst}, {workspace, ws_used}};
  for (const Buf &o : outs) {
    for (const Buf &i : ins)
      if (overlaps(o.p, o.n, i.p, i.n)) return SSD_ERR_INVALID_ARG;
  }
  if (overlaps(y, nx, h_final, nst) || overlaps(y, nx, workspace, ws_used) ||
      overlaps(h_final, nst, workspace, ws_used))
    return SSD_ERR_INVALID_ARG;
  return SSD_OK;
}

ssd_status fwd_impl(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                    const void *B, const void *C, const float *D, const float *h0, int32_t chunk,
                    void *y, float *h_final, void *workspace, size_t ws_bytes, void *const *events,
                    void *stream) {
  Plan pl;
  ssd_status st = make_plan(dims, chunk, &pl);
  if (st != SSD_OK) return st;
  if ((st = check_fwd_buffers(dims, x, dt, A, B, C, D, h0, y, h_final, workspace, pl.total)) !=
      SSD_OK)
    return st;
  if (ws_bytes < pl.total) return SSD_ERR_INVALID_ARG;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  float *cs = reinterpret_cast<float *>(ws + pl.cs_off);
  float *S = reinterpret_cast<float *>(ws + pl.S_off);
  void *Hin = ws + pl.Hin_off;

  if (pl.fused)
    return launch_fused(pl, x, dt, A, B, C, D, h0, y, h_final, ws, events,
                        static_cast<cudaStream_t>(stream));
  if (pl.tc) {
    CUtensorMap mX, mB, mC32, mH, mY;
    const cuuint64_t hdims[3] = {static_cast<cuuint64_t>(pl.P), static_cast<cuuint64_t>(pl.N),
                                 static_cast<cuuint64_t>(pl.b * pl.nc * pl.H)};
    const cuuint64_t hstr[2] = {static_cast<cuuint64_t>(pl.P * 2),
                                static_cast<cuuint64_t>(pl.N * pl.P * 2)};
    const cuuint32_t hbox[3] = {64, static_cast<cuuint32_t>(pl.N), 1};
    if (!encode_btgw(&mX, x, pl.b, pl.T, pl.H, pl.P, pl.Q) ||
        !encode_btgw(&mB, B, pl.b, pl.T, pl.GB, pl.N, pl.Q) ||
        !encode_btgw(&mC32, C, pl.b, pl.T, pl.GC, pl.N, 32) ||
        !encode_btgw(&mY, y, pl.b, pl.T, pl.H, pl.P, pl.Q) ||
        !encode_bf16(&mH, Hin, 3, hdims, hstr, hbox))
      return SSD_ERR_CUDA;
    // chunk_state_hb reads B and x in 128-token halves
    CUtensorMap mB128, mX128, mY128;
    // chunk_scan_hb stores y in 128-row tiles
    if (pl.hb && !encode_btgw(&mY128, y, pl.b, pl.T, pl.H, pl.P, 128)) return SSD_ERR_CUDA;
    if (pl.state_hb && (!encode_btgw(&mX128, x, pl.b, pl.T, pl.H, pl.P, 128) ||
                        !encode_btgw(&mB128, B, pl.b, pl.T, pl.GB, pl.N, 128)))
      return SSD_ERR_CUDA;
    const CUtensorMap &mBs = pl.state_hb ? mB128 : mB, &mXs = pl.state_hb ? mX128 : mX;
    int ev = 0;  // events[i] just before stage i
    record(events, ev, s);
    float *u = nullptr;
    if (pl.state_hb) {
      u = reinterpret_cast<float *>(ws + pl.u_off);
      dim3 g((pl.T + 31) / 32, static_cast<unsigned>((pl.H + 31) / 32), static_cast<unsigned>(pl.b));
      ssd::dt_decay_kernel<<<g, 256, 0, s>>>(dt, A, u, pl.T, static_cast<int>(pl.H), pl.softplus);
      if ((st = launch_status()) != SSD_OK) return st;
      record(events, ++ev, s);
    }
    float *Fseg = pl.nseg > 1 ? reinterpret_cast<float *>(ws + pl.Fseg_off) : nullptr;
    float *Lseg = pl.nseg > 1 ? reinterpret_cast<float *>(ws + pl.Lseg_off) : nullptr;
    float *Dc = pl.nseg > 1 ? reinterpret_cast<float *>(ws + pl.Dc_off) : nullptr;
    uint8_t *flags = pl.hb ? ws + pl.flags_off : nullptr;
    st = pl.Q == 256 ? launch_state_pass<256>(pl, mBs, mXs, dt, A, u, h0, static_cast<__nv_bfloat16 *>(Hin), h_final, Fseg, Lseg, Dc, flags, events, ev, s)
                     : launch_state_pass<128>(pl, mBs, mXs, dt, A, u, h0, static_cast<__nv_bfloat16 *>(Hin), h_final, Fseg, Lseg, Dc, flags, events, ev, s);
    if (st != SSD_OK) return st;
    const int se = ev + (pl.nseg > 1 ? 2 : 1);  // events index after the state stages
    record(events, se, s);
    if (pl.hb)
      st = launch_scan_hb(pl, mC32, mB, mX, mH, mY, mY128, dt, A, D, u, flags, pdl_on(events), s);
    else if (pl.Q == 256) st = launch_scan_hl<256, 64>(pl, mC32, mB, mX, mH, mY, dt, A, D, s);
    else if (pl.P == 64) st = launch_scan_hl<128, 64>(pl, mC32, mB, mX, mH, mY, dt, A, D, s);
    else st = launch_scan_hl<128, 128>(pl, mC32, mB, mX, mH, mY, dt, A, D, s);
    if (st != SSD_OK) return st;
    record(events, se + 1, s);
    return SSD_OK;
  }

  float *Hf = static_cast<float *>(Hin);
  record(events, 0, s);
  if ((st = launch_cumsum(pl, dt, A, cs, s)) != SSD_OK) return st;
  record(events, 1, s);
  st = pl.bf16 ? launch_state_simt<__nv_bfloat16>(pl, x, B, cs, S, s)
               : launch_state_simt<float>(pl, x, B, cs, S, s);
  if (st != SSD_OK) return st;
  record(events, 2, s);
  if ((st = launch_passing(pl, S, cs, h0, Hf, h_final, s)) != SSD_OK) return st;
  record(events, 3, s);
  st = pl.bf16 ? launch_scan_simt<__nv_bfloat16, float>(pl, x, B, C, cs, Hf, D, y, s)
               : launch_scan_simt<float, float>(pl, x, B, C, cs, Hf, D, y, s);
  if (st != SSD_OK) return st;
  record(events, 4, s);
  return SSD_OK;
}

int num_stages(const Plan &pl) {
  if (pl.fused) return pl.nseg > 1 ? 3 : 2;
  return pl.tc ? (pl.nseg > 1 ? 3 : 2) + (pl.state_hb ? 1 : 0) : 4;
}
const char *const kStageNamesSimt[] = {"dt_cumsum", "chunk_state_simt", "state_passing",
                                       "chunk_scan_simt"};

}  // namespace

// ---------------------------------------------------------------------------
// Allocation-free prefill: the scratch of ssd_fwd_noalloc lives in this
// static device array (SSD_NOALLOC_SCRATCH_BYTES), looked up once per device.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mutex;
void *g_noalloc_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name only stands in for the symbol, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
ssd_status noalloc_scratch(void **addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return SSD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SSD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SSD_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *addr = g_noalloc_addr[dev];
  return SSD_OK;
}

}  // namespace

extern "C" {

size_t ssd_fwd_workspace_size(const ssd_dims *dims, int32_t chunk) {
  Plan pl;
  return make_plan(dims, chunk, &pl) == SSD_OK ? pl.total : 0;
}

int32_t ssd_fwd_num_stages(const ssd_dims *dims, int32_t chunk) {
  Plan pl;
  if (make_plan(dims, chunk, &pl) != SSD_OK) return 0;
  return num_stages(pl);
}

const char *ssd_fwd_stage_name(const ssd_dims *dims, int32_t chunk, int32_t i) {
  Plan pl;
  if (make_plan(dims, chunk, &pl) != SSD_OK || i < 0 || i >= num_stages(pl)) return nullptr;
  if (!pl.tc) return kStageNamesSimt[i];
  if (pl.fused) {
    if (pl.nseg > 1 && i-- == 0) return "chunk_fused_prepass";
    return i == 0 ? "chunk_fused_hb" : "chunk_scan_flagged";
  }
  if (pl.state_hb && i-- == 0) return "dt_decay";
  if (i == 0) return pl.state_hb ? "chunk_state_hb" : "chunk_state_pass_tc";
  if (i == 1 && pl.nseg > 1) return "state_fixup";
  return pl.hb ? "chunk_scan_hb" : "chunk_scan_hl";
}

ssd_status ssd_fwd(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                   const void *B, const void *C, const float *D, const float *h0, int32_t chunk,
                   void *y, float *h_final, void *workspace, size_t workspace_bytes,
                   void *stream) {
  return fwd_impl(dims, x, dt, A, B, C, D, h0, chunk, y, h_final, workspace, workspace_bytes,
                  nullptr, stream);
}

ssd_status ssd_fwd_profiled(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                            const void *B, const void *C, const float *D, const float *h0,
                            int32_t chunk, void *y, float *h_final, void *workspace,
                            size_t workspace_bytes, void *const *events, void *stream) {
  if (!events) return SSD_ERR_INVALID_ARG;
  return fwd_impl(dims, x, dt, A, B, C, D, h0, chunk, y, h_final, workspace, workspace_bytes,
                  events, stream);
}

ssd_status ssd_fwd_noalloc(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                           const void *B, const void *C, const float *D, const float *h0,
                           int32_t chunk, void *y, float *h_final, void *stream) {
  Plan pl;
  ssd_status st = make_plan(dims, chunk, &pl);
  if (st != SSD_OK) return st;
  if (pl.total > SSD_NOALLOC_SCRATCH_BYTES) return SSD_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != SSD_OK) return st;
  return fwd_impl(dims, x, dt, A, B, C, D, h0, chunk, y, h_final, scratch,
                  SSD_NOALLOC_SCRATCH_BYTES, nullptr, stream);
}

// ---------------------------------------------------------------------------
// Sequential prefill: windows of at most `window` tokens chained through the
// state.  Workspace: [ssd_fwd workspace of one window][two carried states]
// and, for batch > 1, staging copies of one window of x, dt, B, C and y.
// ---------------------------------------------------------------------------
namespace {

struct SeqPlan {
  ssd_dims wd;  // dims of a full window
  size_t fwd_bytes, carry_off, carry_bytes, stage_off, total;
  size_t row_x, row_dt, row_b, row_c;  // bytes of one token of each tensor
  // windows are staged (copied) in the workspace: all tensors for batch > 1;
  // for batch 1 only dt, and only when a window's offset t0 H 4 bytes would
  // leave it off the 16-byte boundary the kernels need (H not a multiple of 4
  // and a window length that does not restore it)
  bool stage_all, stage_dt;
};

ssd_status make_seq_plan(const ssd_dims *dims, int32_t chunk, int64_t window, SeqPlan *sp) {
  ssd_status st = check_dims(dims);
  if (st != SSD_OK) return st;
  if (window < 1) return SSD_ERR_INVALID_ARG;
  sp->wd = *dims;
  sp->wd.seqlen = std::min<int64_t>(window, dims->seqlen);
  Plan pl;
  if ((st = make_plan(&sp->wd, chunk, &pl)) != SSD_OK) return st;
  const size_t io = dims->io_dtype == SSD_BF16 ? 2 : 4;
  sp->row_x = static_cast<size_t>(dims->nheads * dims->headdim) * io;
  sp->row_dt = static_cast<size_t>(dims->nheads) * 4;
  sp->row_b = static_cast<size_t>(dims->ngroups_b * dims->dstate) * io;
  sp->row_c = static_cast<size_t>(dims->ngroups_c * dims->dstate) * io;
  sp->fwd_bytes = pl.total;
  sp->carry_off = sp->fwd_bytes;
  sp->carry_bytes = align_up(static_cast<size_t>(dims->batch * dims->nheads * dims->dstate *
                                                 dims->headdim) * 4);
  sp->stage_off = sp->carry_off + 2 * sp->carry_bytes;
  sp->total = sp->stage_off;
  sp->stage_all = dims->batch > 1;
  sp->stage_dt = !sp->stage_all && sp->wd.seqlen < dims->seqlen &&
                 (static_cast<size_t>(sp->wd.seqlen) * sp->row_dt) % 16 != 0;
  const size_t rows = static_cast<size_t>(dims->batch * sp->wd.seqlen);
  if (sp->stage_all) {
    sp->total += align_up(rows * sp->row_x) * 2 + align_up(rows * sp->row_dt) +
                 align_up(rows * sp->row_b) + align_up(rows * sp->row_c);
  } else if (sp->stage_dt) {
    sp->total += align_up(rows * sp->row_dt);
  }
  return SSD_OK;
}

// Copies tokens [t0, t0 + len) of a [b, T, row] tensor to or from a [b, len, row] one.
bool copy_window(void *dst, size_t dpitch_tokens, const void *src, size_t spitch_tokens,
                 size_t row, int64_t b, int64_t len, cudaStream_t s) {
  return cudaMemcpy2DAsync(dst, dpitch_tokens * row, src, spitch_tokens * row,
                           static_cast<size_t>(len) * row, static_cast<size_t>(b),
                           cudaMemcpyDeviceToDevice, s) == cudaSuccess;
}

}  // namespace

size_t ssd_fwd_sequential_workspace_size(const ssd_dims *dims, int32_t chunk, int64_t window) {
  SeqPlan sp;
  return make_seq_plan(dims, chunk, window, &sp) == SSD_OK ? sp.total : 0;
}

ssd_status ssd_fwd_sequential(const ssd_dims *dims, const void *x, const float *dt,
                              const float *A, const void *B, const void *C, const float *D,
                              const float *h0, int32_t chunk, int64_t window, void *y,
                              float *h_final, void *workspace, size_t workspace_bytes,
                              void *stream) {
  SeqPlan sp;
  ssd_status st = make_seq_plan(dims, chunk, window, &sp);
  if (st != SSD_OK) return st;
  // every argument check before the first window is enqueued: the whole
  // tensors' pointers, alignment and aliasing, and the workspace size (each
  // window's own ssd_fwd checks then see only aligned, disjoint windows)
  if ((st = check_fwd_buffers(dims, x, dt, A, B, C, D, h0, y, h_final, workspace, sp.total)) !=
      SSD_OK)
    return st;
  if (workspace_bytes < sp.total) return SSD_ERR_INVALID_ARG;
  const int64_t b = dims->batch, T = dims->seqlen, W = sp.wd.seqlen;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  float *carry[2] = {reinterpret_cast<float *>(ws + sp.carry_off),
                     reinterpret_cast<float *>(ws + sp.carry_off + sp.carry_bytes)};
  uint8_t *stage = ws + sp.stage_off;
  const size_t rows = static_cast<size_t>(b * W);
  uint8_t *sx = stage, *sy = sx + align_up(rows * sp.row_x);
  uint8_t *sdt = sp.stage_all ? sy + align_up(rows * sp.row_x) : stage;
  uint8_t *sB = sdt + align_up(rows * sp.row_dt);
  uint8_t *sC = sB + align_up(rows * sp.row_b);
  const uint8_t *px = static_cast<const uint8_t *>(x), *pdt = reinterpret_cast<const uint8_t *>(dt),
                *pB = static_cast<const uint8_t *>(B), *pC = static_cast<const uint8_t *>(C);
  uint8_t *py = static_cast<uint8_t *>(y);
  int w = 0;
  for (int64_t t0 = 0; t0 < T; t0 += W, ++w) {
    const int64_t len = std::min(W, T - t0);
    ssd_dims d = sp.wd;
    d.seqlen = len;
    const float *hin = w == 0 ? h0 : carry[(w - 1) & 1];
    float *hout = t0 + len >= T ? h_final : carry[w & 1];
    const void *wx, *wdt, *wB, *wC;
    void *wy;
    if (!sp.stage_all) {  // a window of a single sequence is contiguous
      wx = px + t0 * sp.row_x;
      wdt = pdt + t0 * sp.row_dt;
      wB = pB + t0 * sp.row_b;
      wC = pC + t0 * sp.row_c;
      wy = py + t0 * sp.row_x;
      if (sp.stage_dt && !aligned16(wdt)) {
        if (cudaMemcpyAsync(sdt, wdt, static_cast<size_t>(len) * sp.row_dt,
                            cudaMemcpyDeviceToDevice, s) != cudaSuccess)
          return SSD_ERR_CUDA;
        wdt = sdt;
      }
    } else {
      if (!copy_window(sx, len, px + t0 * sp.row_x, T, sp.row_x, b, len, s) ||
          !copy_window(sdt, len, pdt + t0 * sp.row_dt, T, sp.row_dt, b, len, s) ||
          !copy_window(sB, len, pB + t0 * sp.row_b, T, sp.row_b, b, len, s) ||
          !copy_window(sC, len, pC + t0 * sp.row_c, T, sp.row_c, b, len, s))
        return SSD_ERR_CUDA;
      wx = sx; wdt = sdt; wB = sB; wC = sC; wy = sy;
    }
    st = fwd_impl(&d, wx, static_cast<const float *>(wdt), A, wB, wC, D, hin, chunk, wy, hout, ws,
                  sp.fwd_bytes, nullptr, stream);
    if (st != SSD_OK) return st;
    if (sp.stage_all && !copy_window(py + t0 * sp.row_x, T, sy, len, sp.row_x, b, len, s))
      return SSD_ERR_CUDA;
  }
  return SSD_OK;
}

ssd_status ssd_multistep(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                         const void *B, const void *C, const float *D, const float *h_cache,
                         const int32_t *j, void *y, float *h_j, float *h_K, void *stream) {
  ssd_status st = check_dims(dims);
  if (st != SSD_OK) return st;
  const int64_t b = dims->batch, K = dims->seqlen, H = dims->nheads, P = dims->headdim,
                N = dims->dstate, GB = dims->ngroups_b, GC = dims->ngroups_c;
  if (K > 16) return SSD_ERR_UNSUPPORTED;
  if (b > 65535 || H > 65535) return SSD_ERR_UNSUPPORTED;
  if (!x || !dt || !A || !B || !C || !h_cache || !j || !y || !h_j || !h_K)
    return SSD_ERR_INVALID_ARG;
  const void *ptrs[] = {x, dt, A, B, C, D, h_cache, j, y, h_j, h_K};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return SSD_ERR_INVALID_ARG;
  const bool bf16 = dims->io_dtype == SSD_BF16;
  const size_t io = bf16 ? 2 : 4;
  const size_t nx = static_cast<size_t>(b * K * H * P) * io;
  const size_t nst = static_cast<size_t>(b * H * N * P) * 4;
  struct Buf { const void *p; size_t n; };
  const Buf ins[] = {{x, nx},
                     {dt, static_cast<size_t>(b * K * H) * 4},
                     {A, static_cast<size_t>(H) * 4},
                     {B, static_cast<size_t>(b * K * GB * N) * io},
                     {C, static_cast<size_t>(b * K * GC * N) * io},
                     {D, static_cast<size_t>(H) * 4},
                     {h_cache, nst},
                     {j, static_cast<size_t>(b) * 4}};
  const Buf outs[] = {{y, nx}, {h_j, nst}, {h_K, nst}};
  for (const Buf &o : outs)
    for (const Buf &i : ins)
      if (overlaps(o.p, o.n, i.p, i.n)) return SSD_ERR_INVALID_ARG;
  if (overlaps(y, nx, h_j, nst) || overlaps(y, nx, h_K, nst) || overlaps(h_j, nst, h_K, nst))
    return SSD_ERR_INVALID_ARG;

  // column slice per block: the largest of 128, 64, 32, 16 that divides P
  const int PS = P % 128 == 0 ? 128 : P % 64 == 0 ? 64 : P % 32 == 0 ? 32 : 16;
  const int R = ssd::kMsThreads / (PS / 4);
  // raw rows of B move in 16-byte granules
  if (N % R || (N * (dims->io_dtype == SSD_BF16 ? 2 : 4)) % 16) return SSD_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // (b, h) items dealt out SM by SM (see multistep_kernel)
  const int64_t nsm_ = num_sms();
  if ((H * b + nsm_ - 1) / nsm_ > 65535) return SSD_ERR_UNSUPPORTED;
  dim3 grid(static_cast<unsigned>(nsm_), static_cast<unsigned>((H * b + nsm_ - 1) / nsm_),
            static_cast<unsigned>(P / PS));
  return dispatch_ms<false>(grid, dims, 0, nullptr, nullptr, nullptr, j, x, dt, A, B, C, D, h_cache,
                            y, h_j, h_K, nullptr, PS, s);
}

ssd_status ssd_verify(const ssd_dims *dims, int32_t k_prev, const void *x_prev,
                      const float *dt_prev, const void *B_prev, const int32_t *j_prev,
                      const void *x, const float *dt, const float *A, const void *B, const void *C,
                      const float *D, const float *h_cache, void *y, float *h_next, void *stream) {
  ssd_status st = check_dims(dims);
  if (st != SSD_OK) return st;
  const int64_t b = dims->batch, K = dims->seqlen, H = dims->nheads, P = dims->headdim,
                N = dims->dstate, GB = dims->ngroups_b, GC = dims->ngroups_c, KP = k_prev;
  if (K > 16 || KP > 16) return SSD_ERR_UNSUPPORTED;
  if (KP < 1) return SSD_ERR_INVALID_ARG;
  if (b > 65535 || H > 65535) return SSD_ERR_UNSUPPORTED;
  if (!x_prev || !dt_prev || !B_prev || !j_prev || !x || !dt || !A || !B || !C || !h_cache ||
      !y || !h_next)
    return SSD_ERR_INVALID_ARG;
  const void *ptrs[] = {x_prev, dt_prev, B_prev, j_prev, x, dt, A, B, C, D, h_cache, y, h_next};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return SSD_ERR_INVALID_ARG;
  const bool bf16 = dims->io_dtype == SSD_BF16;
  const size_t io = bf16 ? 2 : 4;
  const size_t nx = static_cast<size_t>(b * K * H * P) * io;
  const size_t nst = static_cast<size_t>(b * H * N * P) * 4;
  const size_t ndt = static_cast<size_t>(b * K * H) * 4;
  const size_t nB = static_cast<size_t>(b * K * GB * N) * io;
  const size_t nxp = static_cast<size_t>(b * KP * H * P) * io;
  const size_t ndtp = static_cast<size_t>(b * KP * H) * 4;
  const size_t nBp = static_cast<size_t>(b * KP * GB * N) * io;
  struct Buf { const void *p; size_t n; };
  const Buf ins[] = {{x_prev, nxp}, {dt_prev, ndtp}, {B_prev, nBp}, {j_prev, static_cast<size_t>(b) * 4},
                     {x, nx}, {dt, ndt}, {A, static_cast<size_t>(H) * 4}, {B, nB},
                     {C, static_cast<size_t>(b * K * GC * N) * io}, {D, static_cast<size_t>(H) * 4},
                     {h_cache, nst}};
  const Buf outs[] = {{y, nx}, {h_next, nst}};
  for (const Buf &o : outs)
    for (const Buf &i : ins)
      if (overlaps(o.p, o.n, i.p, i.n)) return SSD_ERR_INVALID_ARG;
  if (overlaps(y, nx, h_next, nst)) return SSD_ERR_INVALID_ARG;

  const int PS = P % 128 == 0 ? 128 : P % 64 == 0 ? 64 : P % 32 == 0 ? 32 : 16;
  const int R = ssd::kMsThreads / (PS / 4);
  // raw rows of B move in 16-byte granules
  if (N % R || (N * (dims->io_dtype == SSD_BF16 ? 2 : 4)) % 16) return SSD_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 grid(static_cast<unsigned>(H), static_cast<unsigned>(b), static_cast<unsigned>(P / PS));
  return dispatch_ms<true>(grid, dims, static_cast<int>(KP), x_prev, dt_prev, B_prev, j_prev, x, dt,
                           A, B, C, D, h_cache, y, nullptr, nullptr, h_next, PS, s);
}

// ---------------------------------------------------------------------------
// Context parallelism: per-segment decay, and the correction of a segment's
// outputs and final state once the states of the segments before it are known.
// Workspace: the running log2 decays a [b, H, T] (within 128-token tiles) and the
// tiles' totals [b, H, ceil(T / 128)], H_in [b, H, N, P] float32,
// then H_in rounded to bf16 in the tensor-core operand image (b H tiles of N P
// bf16).
// ---------------------------------------------------------------------------
namespace {

struct CpPlan {
  int64_t b, T, H, P, N, GC, ntiles;
  size_t pre_off, decay_bytes, hin_off, op_off, total;
};

ssd_status make_cp_plan(const ssd_dims *d, CpPlan *cp) {
  ssd_status st = check_dims(d);
  if (st != SSD_OK) return st;
  cp->b = d->batch;
  cp->T = d->seqlen;
  cp->H = d->nheads;
  cp->P = d->headdim;
  cp->N = d->dstate;
  cp->GC = d->ngroups_c;
  if (cp->b * cp->H > (int64_t(1) << 31) - 1 || cp->b > 65535) return SSD_ERR_UNSUPPORTED;
  cp->ntiles = (cp->T + ssd::kCpTile - 1) / ssd::kCpTile;
  cp->pre_off = align_up(static_cast<size_t>(cp->b * cp->H * cp->T) * 4);
  cp->decay_bytes = cp->pre_off + align_up(static_cast<size_t>(cp->b * cp->H * cp->ntiles) * 4);
  cp->hin_off = cp->decay_bytes;
  cp->op_off = cp->hin_off + align_up(static_cast<size_t>(cp->b * cp->H * cp->N * cp->P) * 4);
  cp->total = cp->op_off + align_up(static_cast<size_t>(cp->b * cp->H * cp->N * cp->P) * 2);
  return SSD_OK;
}

// a[b, h, t] = running log2 decay from the start of t's 128-token tile
// (inclusive) and pre[b, h, k] = the decay over the tiles before tile k (the
// running decay from the segment's start is their sum); the segment's total
// decay into decay[b H] when given.
ssd_status cp_running_decay(const CpPlan &cp, const float *dt, const float *A, int softplus,
                            float *a, float *pre, float *decay, cudaStream_t s) {
  dim3 g(static_cast<unsigned>(cp.ntiles), static_cast<unsigned>((cp.H + 31) / 32),
         static_cast<unsigned>(cp.b));
  if (cp.ntiles > 2147483647ll || g.y > 65535) return SSD_ERR_UNSUPPORTED;
  ssd::cp_tile_decay_kernel<<<g, 256, 0, s>>>(dt, A, a, pre, cp.T, static_cast<int>(cp.H),
                                              static_cast<int>(cp.ntiles), softplus);
  ssd_status st = launch_status();
  if (st != SSD_OK) return st;
  const int64_t rows = cp.b * cp.H;
  ssd::cp_tile_prefix_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, s>>>(
      pre, static_cast<int>(cp.ntiles), rows, decay);
  return launch_status();
}

// Heads per work unit of cp_correct_tc: a divisor of the heads per C group,
// the largest that still gives each persistent CTA eight units or more (each
// unit loads one C tile; more units even out the CTAs' shares).
int cp_heads_per_unit(const CpPlan &cp) {
  const int64_t per_group = cp.H / cp.GC, tiles = (cp.T + 127) / 128;
  for (int64_t hpc = per_group; hpc > 1; --hpc)
    if (per_group % hpc == 0 && tiles * cp.b * (cp.H / hpc) >= 8 * num_sms())
      return static_cast<int>(hpc);
  return 1;
}

ssd_status launch_cp_correct_tc(const CpPlan &cp, const void *C, void *y, const uint8_t *hin_op,
                                const float *a, const float *pre, cudaStream_t s) {
  const int P = static_cast<int>(cp.P);
  CUtensorMap mC, mYl, mYs;
  if (!encode_btgw(&mC, C, cp.b, cp.T, cp.GC, cp.N, 128) ||
      !encode_btgw(&mYl, y, cp.b, cp.T, cp.H, P, 128) ||
      !encode_btgw(&mYs, y, cp.b, cp.T, cp.H, P, 32))
    return SSD_ERR_CUDA;
  const int hpc = cp_heads_per_unit(cp);
  const int64_t units = cp.ntiles * cp.b * (cp.H / hpc);
  if (cp.T > 2147483647ll - 128) return SSD_ERR_UNSUPPORTED;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(units, num_sms()));
  const int nt = static_cast<int>(cp.ntiles), H = static_cast<int>(cp.H),
            GC = static_cast<int>(cp.GC);
  if (P == 64) {
    using L = ssd::CpTc<64>;
    if (!ensure_smem<ssd::cp_correct_tc<64>>(L::kBytes)) return SSD_ERR_CUDA;
    ssd::cp_correct_tc<64><<<grid, L::kThreads, L::kBytes, s>>>(mC, mYl, mYs, hin_op, a, pre, nt,
                                                                cp.T, H, GC, hpc, units);
  } else {
    using L = ssd::CpTc<128>;
    if (!ensure_smem<ssd::cp_correct_tc<128>>(L::kBytes)) return SSD_ERR_CUDA;
    ssd::cp_correct_tc<128><<<grid, L::kThreads, L::kBytes, s>>>(mC, mYl, mYs, hin_op, a, pre, nt,
                                                                 cp.T, H, GC, hpc, units);
  }
  return launch_status();
}

}  // namespace

size_t ssd_cp_workspace_size(const ssd_dims *dims) {
  CpPlan cp;
  return make_cp_plan(dims, &cp) == SSD_OK ? cp.total : 0;
}

ssd_status ssd_cp_segment_decay(const ssd_dims *dims, const float *dt, const float *A,
                                float *decay, void *workspace, size_t workspace_bytes,
                                void *stream) {
  CpPlan cp;
  ssd_status st = make_cp_plan(dims, &cp);
  if (st != SSD_OK) return st;
  if (!dt || !A || !decay || !workspace) return SSD_ERR_INVALID_ARG;
  const void *ptrs[] = {dt, A, decay, workspace};
  for (const void *p : ptrs)
    if (!aligned16(p)) return SSD_ERR_INVALID_ARG;
  if (workspace_bytes < cp.decay_bytes) return SSD_ERR_INVALID_ARG;
  const size_t ndt = static_cast<size_t>(cp.b * cp.T * cp.H) * 4, nh = cp.H * 4,
               nd = static_cast<size_t>(cp.b * cp.H) * 4;
  if (overlaps(decay, nd, dt, ndt) || overlaps(decay, nd, A, nh) ||
      overlaps(decay, nd, workspace, cp.decay_bytes) ||
      overlaps(workspace, cp.decay_bytes, dt, ndt) || overlaps(workspace, cp.decay_bytes, A, nh))
    return SSD_ERR_INVALID_ARG;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  return cp_running_decay(cp, dt, A, dims->dt_softplus, reinterpret_cast<float *>(ws),
                          reinterpret_cast<float *>(ws + cp.pre_off), decay,
                          static_cast<cudaStream_t>(stream));
}

ssd_status ssd_cp_correct(const ssd_dims *dims, int32_t nranks, int32_t rank,
                          const float *decays, const float *finals, const float *dt,
                          const float *A, const void *C, void *y, float *h_final,
                          void *workspace, size_t workspace_bytes, void *stream) {
  CpPlan cp;
  ssd_status st = make_cp_plan(dims, &cp);
  if (st != SSD_OK) return st;
  if (nranks < 1 || rank < 0 || rank >= nranks) return SSD_ERR_INVALID_ARG;
  if (!decays || !finals || !dt || !A || !C || !y || !workspace) return SSD_ERR_INVALID_ARG;
  const void *ptrs[] = {decays, finals, dt, A, C, y, h_final, workspace};
  for (const void *p : ptrs)
    if (p && !aligned16(p)) return SSD_ERR_INVALID_ARG;
  if (workspace_bytes < cp.total) return SSD_ERR_INVALID_ARG;
  const size_t io = dims->io_dtype == SSD_BF16 ? 2 : 4;
  const size_t BH = static_cast<size_t>(cp.b * cp.H), NP = static_cast<size_t>(cp.N * cp.P);
  struct Buf { const void *p; size_t n; };
  const Buf ins[] = {{decays, nranks * BH * 4}, {finals, nranks * BH * NP * 4},
                     {dt, static_cast<size_t>(cp.b * cp.T * cp.H) * 4}, {A, static_cast<size_t>(cp.H) * 4},
                     {C, static_cast<size_t>(cp.b * cp.T * cp.GC * cp.N) * io}};
  const Buf outs[] = {{y, static_cast<size_t>(cp.b * cp.T * cp.H * cp.P) * io},
                      {h_final, BH * NP * 4}, {workspace, cp.total}};
  for (const Buf &o : outs)
    for (const Buf &i : ins)
      if (overlaps(o.p, o.n, i.p, i.n)) return SSD_ERR_INVALID_ARG;
  if (overlaps(outs[0].p, outs[0].n, h_final, outs[1].n) ||
      overlaps(outs[0].p, outs[0].n, workspace, cp.total) ||
      overlaps(h_final, outs[1].n, workspace, cp.total))
    return SSD_ERR_INVALID_ARG;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  float *a = reinterpret_cast<float *>(ws);
  float *pre = reinterpret_cast<float *>(ws + cp.pre_off);
  float *hin = reinterpret_cast<float *>(ws + cp.hin_off);
  uint8_t *hin_op = ws + cp.op_off;
  const bool tc = dims->io_dtype == SSD_BF16 && cp.N == kTcN && (cp.P == 64 || cp.P == 128);
  const int64_t n4 = static_cast<int64_t>(BH * NP / 4);
  const unsigned blocks = static_cast<unsigned>((n4 + 255) / 256);
  // H_in of this rank (float32 for the CUDA-core update, the bf16 operand
  // image for the tensor-core one) and its true final state (rank 0: its own
  // final state)
  ssd::cp_combine_kernel<<<blocks, 256, 0, s>>>(
      decays, finals, rank, static_cast<int64_t>(BH), static_cast<int>(NP),
      static_cast<int>(cp.P), rank > 0 && !tc ? hin : nullptr, rank > 0 && tc ? hin_op : nullptr,
      h_final);
  if ((st = launch_status()) != SSD_OK) return st;
  if (rank == 0) return SSD_OK;  // the first segment started from the true h0
  if ((st = cp_running_decay(cp, dt, A, dims->dt_softplus, a, pre, nullptr, s)) != SSD_OK)
    return st;
  if (tc)
    return launch_cp_correct_tc(cp, C, y, hin_op, a, pre, s);
  const int PS = cp.P % 64 == 0 ? 64 : cp.P % 32 == 0 ? 32 : 16;
  const int smem = static_cast<int>((32 * cp.N + cp.N * PS) * 4);
  dim3 grid(static_cast<unsigned>((cp.T + 31) / 32), static_cast<unsigned>(cp.P / PS),
            static_cast<unsigned>(BH));
  if (grid.y > 65535 || BH > 65535) return SSD_ERR_UNSUPPORTED;
  if (dims->io_dtype == SSD_BF16) {
    if (!ensure_smem<ssd::cp_correct_simt<__nv_bfloat16>>((32 * 256 + 256 * 64) * 4))
      return SSD_ERR_CUDA;
    ssd::cp_correct_simt<__nv_bfloat16><<<grid, 256, smem, s>>>(
        static_cast<const __nv_bfloat16 *>(C), hin, a, pre, static_cast<int>(cp.ntiles),
        static_cast<__nv_bfloat16 *>(y), cp.T,
        static_cast<int>(cp.H), static_cast<int>(cp.GC), static_cast<int>(cp.N),
        static_cast<int>(cp.P), PS);
  } else {
    if (!ensure_smem<ssd::cp_correct_simt<float>>((32 * 256 + 256 * 64) * 4)) return SSD_ERR_CUDA;
    ssd::cp_correct_simt<float><<<grid, 256, smem, s>>>(
        static_cast<const float *>(C), hin, a, pre, static_cast<int>(cp.ntiles),
        static_cast<float *>(y), cp.T,
        static_cast<int>(cp.H), static_cast<int>(cp.GC), static_cast<int>(cp.N),
        static_cast<int>(cp.P), PS);
  }
  return launch_status();
}

ssd_status ssd_check_device_error(void *stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SSD_ERR_CUDA;
  int code = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&code, ssd::g_device_error, sizeof(int)) != cudaSuccess ||
      cudaMemcpyToSymbol(ssd::g_device_error, &zero, sizeof(int)) != cudaSuccess)
    return SSD_ERR_CUDA;
  if (code == ssd::kDevTimeout) return SSD_ERR_TIMEOUT;
  if (code == ssd::kDevBadJ) return SSD_ERR_INVALID_ARG;
  return SSD_OK;
}

ssd_status ssd_selftest_timeout(int64_t limit_ns, void *stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000) return SSD_ERR_INVALID_ARG;
  ssd::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t>(limit_ns));
  return launch_status();
}

const char *ssd_status_string(ssd_status status) {
  switch (status) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID_ARG: return "invalid argument";
    case SSD_ERR_UNSUPPORTED: return "unsupported shape or chunk length";
    case SSD_ERR_CUDA: return "CUDA error";
    case SSD_ERR_TIMEOUT: return "a kernel's bounded wait timed out";
  }
  return "unknown status";
}

int32_t ssd_version(void) { return SSD_VERSION; }

}  // extern "C"
