/*
 * ssd.h -- C ABI of libssd: the Mamba-2 SSD (state-space duality) layer and
 * the K-token multi-step verification decode, on one NVIDIA B300 (sm_103a).
 *
 * The operation.  For every batch row b and head h the layer carries a state
 * h of shape N x P and runs the selective recurrence with a scalar decay per
 * head (Mamba-2's SSD restriction of the SSM, cloud.tencent page "Mamba 2 ...
 * SSD", sections "核心创新——SSD" and "SSD算法"):
 *
 *     dt_t = softplus(dt_raw_t)         (if dims.dt_softplus; else dt_raw_t)
 *     h_t  = exp(dt_t * A_h) * h_{t-1} + B_t x_t^T
 *     y_t  = C_t^T h_t + D_h * x_t
 *
 * ssd_fwd evaluates it with the chunked block decomposition of that page
 * (section "SSD算法" and "深入解析分块与状态传递机制"): Q x Q diagonal blocks in
 * quadratic, attention-like form; the final state of every chunk from a zero
 * initial state; a short scan that passes states across chunks; then each
 * chunk's output from its true initial state.  ssd_multistep is the
 * MultiStep verification of speculative decoding ("Mamba in the Llama",
 * csdn page, section "推测解码"): K draft tokens advanced from a cached state,
 * returning the K outputs, the state at the last accepted position j and the
 * state after all K.
 *
 * Conventions shared by every call.
 *   - Pointers are DEVICE pointers unless stated otherwise; every tensor is
 *     contiguous and row-major, 16-byte aligned (the kernels stage tiles with
 *     the Tensor Memory Accelerator, which needs that alignment).
 *   - x, y        [batch, T, H, P]   io dtype (float32 or bfloat16)
 *     dt          [batch, T, H]      float32 (raw dt; see dt_softplus)
 *     B           [batch, T, G_B, N] io dtype
 *     C           [batch, T, G_C, N] io dtype
 *     A, D        [H]                float32 (A_h < 0 decays; D may be NULL = 0)
 *     states      [batch, H, N, P]   float32, P fastest
 *     Head h reads group h / (H / G) of B and C.
 *   - The caller owns every buffer, including the workspace.  The library
 *     never allocates, frees or synchronises; all work is enqueued on
 *     `stream` (a cudaStream_t, NULL = legacy default stream).
 *   - Inputs are read-only.  Outputs must not alias inputs or each other.
 *   - Argument errors are detected on the host before anything is launched.
 *   - Results: y is rounded to nearest even into the io dtype; states stay
 *     float32.
 */
#ifndef LIBSSD_SSD_H
#define LIBSSD_SSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SSD_VERSION 10000 /* major * 10000 + minor * 100 + patch */

typedef enum ssd_status {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, aliasing, short workspace */
    SSD_ERR_UNSUPPORTED = 2, /* a shape or chunk outside the supported envelope */
    SSD_ERR_CUDA = 3,        /* a CUDA launch or runtime call failed */
    SSD_ERR_TIMEOUT = 4      /* a kernel's bounded wait ran out (see ssd_check_device_error) */
} ssd_status;

typedef enum ssd_dtype { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

/* Problem description shared by ssd_fwd and ssd_multistep.
 *   batch, seqlen (T; K for ssd_multistep), nheads (H), headdim (P),
 *   dstate (N), ngroups_b (G_B), ngroups_c (G_C): sizes, all >= 1.
 *   P and N: multiples of 16, at most 256.  H % G_B == 0, H % G_C == 0.
 *   io_dtype: SSD_F32 or SSD_BF16 -- the dtype of x, B, C and y.
 *   dt_softplus: 1 = apply softplus (z > 20 -> z) to dt; 0 = dt is used as given. */
typedef struct ssd_dims {
    int64_t batch;
    int64_t seqlen;
    int64_t nheads;
    int64_t headdim;
    int64_t dstate;
    int64_t ngroups_b;
    int64_t ngroups_c;
    int32_t io_dtype;
    int32_t dt_softplus;
} ssd_dims;

/* Bytes of device workspace ssd_fwd needs for these dims and chunk length
 * (chunk in {64, 128, 256}).  Returns 0 for arguments ssd_fwd would reject.
 * The workspace holds the chunk initial states [b, nc, H, N, P]
 * (nc = ceil(T / Q); bf16 on the tensor-core path, float32 otherwise) and the
 * other intermediates of the kernels chosen for these dims. */
size_t ssd_fwd_workspace_size(const ssd_dims *dims, int32_t chunk);

/* Chunked SSD prefill (cloud.tencent Mamba-2 page, section "SSD算法").
 *   h0:       initial state [b, H, N, P] or NULL (zero state).
 *   chunk:    Q, the block size of the decomposition: 64, 128 or 256.  The
 *             result does not depend on it beyond rounding; it sets the
 *             schedule.  The last chunk may be short (any T >= 1).
 *   y:        output [b, T, H, P], io dtype.
 *   h_final:  output state after token T [b, H, N, P], or NULL.
 *   workspace/workspace_bytes: device scratch of at least
 *             ssd_fwd_workspace_size() bytes; contents need no initialisation
 *             and are garbage afterwards.
 * Returns SSD_OK once every kernel is enqueued on `stream`.
 * With 256-token chunks, 64-wide heads and one (B, C) group the chunk outputs
 * can be computed two heads per MMA in a scaled form (chunk_scan_hb) or head
 * by head (chunk_scan_hl); the call picks by the work per CTA.  The
 * environment variable SSD_CHUNK_SCAN=pair or =head, read on every call,
 * forces one of the two (results agree within the stated tolerance).  On
 * that path the kernels after the first are launched as programmatic
 * dependents, so that each one's set-up overlaps the end of the one before;
 * SSD_PDL=0 (read on every call) launches them one after another instead
 * (bit-identical results). */
ssd_status ssd_fwd(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                   const void *B, const void *C, const float *D, const float *h0, int32_t chunk,
                   void *y, float *h_final, void *workspace, size_t workspace_bytes,
                   void *stream);

/* Number of kernels ssd_fwd launches for these arguments (its stages), or 0
 * for arguments it would reject. */
int32_t ssd_fwd_num_stages(const ssd_dims *dims, int32_t chunk);

/* Name of stage i of ssd_fwd for these arguments ("dt_cumsum",
 * "chunk_state", "state_passing", "chunk_scan", ...), or NULL. */
const char *ssd_fwd_stage_name(const ssd_dims *dims, int32_t chunk, int32_t i);

/* ssd_fwd, additionally recording events[i] (a cudaEvent_t, host array of
 * ssd_fwd_num_stages() + 1 entries) on `stream` just before stage i and
 * events[num_stages] after the last stage, so a caller can time each kernel
 * on the stream it runs on.  Same arguments and results as ssd_fwd. */
ssd_status ssd_fwd_profiled(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                            const void *B, const void *C, const float *D, const float *h0,
                            int32_t chunk, void *y, float *h_final, void *workspace,
                            size_t workspace_bytes, void *const *events, void *stream);

/* Sequential ("chunked-prompt") prefill (the Falcon Mamba 7B release page,
 * "Mamba 再次挑戰霸主 Transformer", on parallel versus sequential prefill:
 * processing the prompt in pieces with the recurrent state carried between
 * them keeps memory independent of the prompt length, which is what lets an
 * SSM take prompts of any length).  The sequence is processed in windows of at most `window`
 * tokens; each window is one ssd_fwd whose h0 is the previous window's final
 * state (the first window's is h0).  The result equals one ssd_fwd over the
 * whole sequence up to rounding, in device memory that does not grow with T.
 *   window:   tokens per window, >= 1; a multiple of chunk keeps every window
 *             on the chunk grid.
 *   workspace/workspace_bytes: at least ssd_fwd_sequential_workspace_size()
 *             bytes -- one window's ssd_fwd workspace, two carried float32
 *             states and, for batch > 1, a staging copy of one window of x,
 *             dt, B, C and y (windows of a batched [b, T, ...] tensor are
 *             not contiguous; they are gathered and scattered with
 *             asynchronous 2-D copies on `stream`).
 * Other arguments and results as ssd_fwd.  Every step is enqueued on
 * `stream`, so the call can be captured in a CUDA graph. */
size_t ssd_fwd_sequential_workspace_size(const ssd_dims *dims, int32_t chunk, int64_t window);
ssd_status ssd_fwd_sequential(const ssd_dims *dims, const void *x, const float *dt,
                              const float *A, const void *B, const void *C, const float *D,
                              const float *h0, int32_t chunk, int64_t window, void *y,
                              float *h_final, void *workspace, size_t workspace_bytes,
                              void *stream);

/* K-token multi-step verification decode ("Mamba in the Llama", section
 * "推测解码": MultiStep returns the K outputs, the state at the last verified
 * position j and the state at K; FirstConflict then keeps h_j, which equals
 * h_K when all K drafts are accepted).
 *   dims.seqlen = K, 1 <= K <= 16.
 *   x [b, K, H, P], dt [b, K, H], B [b, K, G_B, N], C [b, K, G_C, N].
 *   h_cache:  cached state [b, H, N, P] (float32) to advance from.
 *   j:        DEVICE int32 [b], accepted-token count per batch row, 0..K.
 *             h_j is the state after the first j tokens of this call
 *             (j = 0 gives h_cache back).  Values outside 0..K make the
 *             kernel write h_j for no position; the host cannot check them.
 *   y [b, K, H, P] (io dtype), h_j and h_K [b, H, N, P] (float32): outputs.
 *   h_j and h_K may not alias h_cache or each other. */
ssd_status ssd_multistep(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                         const void *B, const void *C, const float *D, const float *h_cache,
                         const int32_t *j, void *y, float *h_j, float *h_K, void *stream);

/* Fused verification step with recompute ("Mamba in the Llama", section
 * "硬件特定优化": for the verifier, one kernel first recomputes the previous
 * steps from the cache, then decodes the new drafts, then caches; for a Mamba
 * draft model, recompute, decode and cache are likewise one kernel).  The
 * cache holds the state before the PREVIOUS call's k_prev drafts, of which
 * j_prev[b] were accepted; this call advances it through those j_prev[b]
 * tokens -- the state every accepted prefix ends in -- stores that as the
 * next cache, and decodes the K new tokens from it.  Per call each state is
 * read once and written once (ssd_multistep writes two states).
 *   Verifier: k_prev = K = the draft length.  Chaining ssd_verify(prev = the
 *             drafts of call s-1, j_prev = their accepted count) reproduces a
 *             ssd_multistep chain that continues from h_j bit for bit.
 *   Draft model: the first draft step of a round is ssd_verify with the
 *             previous round's k_prev drafts and K = 1 new token; the rest of
 *             the round are ssd_multistep calls with K = 1.
 *   dims.seqlen = K, the new tokens (1..16); k_prev: 1..16.
 *   x_prev [b, k_prev, H, P], dt_prev [b, k_prev, H], B_prev [b, k_prev, G_B, N]:
 *             the previous drafts (their C is not needed).
 *   j_prev:   DEVICE int32 [b], 0..k_prev.  A value outside that records
 *             SSD_ERR_INVALID_ARG in the device error word (see
 *             ssd_check_device_error) and leaves that batch row's y and
 *             h_next unwritten.
 *   x, dt, B, C, D: the new tokens, as in ssd_multistep.
 *   h_cache:  [b, H, N, P] float32, the state before the previous drafts.
 *   y [b, K, H, P] (io dtype), h_next [b, H, N, P] (float32): outputs; they
 *             may not alias any input or each other. */
ssd_status ssd_verify(const ssd_dims *dims, int32_t k_prev, const void *x_prev,
                      const float *dt_prev, const void *B_prev, const int32_t *j_prev,
                      const void *x, const float *dt, const float *A, const void *B, const void *C,
                      const float *D, const float *h_cache, void *y, float *h_next, void *stream);

/* Context parallelism over the sequence (Mamba-2 page, section "序列并行的两种形式",
 * context parallelism: each GPU computes the outputs and the final state of
 * its own segment of the sequence, then the states are passed from GPU to
 * GPU).  Rank r of nranks holds tokens [t_r, t_{r+1}) of every sequence:
 *   1. ssd_fwd on the segment, with h0 on rank 0 and NULL (zero) elsewhere:
 *      y (local) and F_r = the segment's final state (h_final);
 *   2. ssd_cp_segment_decay: Lambda_r[b, h], the segment's total decay (the
 *      product over its tokens of exp(dt_t A_h));
 *   3. the caller gathers every rank's Lambda and F (e.g. an all-gather),
 *      rank-ordered, into decays [nranks, b, H] and finals [nranks, b, H, N, P];
 *   4. ssd_cp_correct: the true state entering segment r,
 *         H_in(0) = 0,  H_in(r'+1) = Lambda_r' H_in(r') + F_r'
 *      (the scan over ranks; F_0 already includes h0), then
 *         y_t += exp(cs_t) C_t^T H_in(r)   for every token t of the segment,
 *         h_final = Lambda_r H_in(r) + F_r,
 *      with cs_t the running sum of dt A from the segment's start to t
 *      (inclusive).  The concatenated y and the last rank's h_final then
 *      equal one ssd_fwd over the whole sequence up to rounding.
 * dims describe this rank's segment (seqlen = its length).  Workspace: at
 * least ssd_cp_workspace_size(dims) bytes, no initialisation needed.  All
 * work is enqueued on `stream`; nothing is allocated or synchronised. */
size_t ssd_cp_workspace_size(const ssd_dims *dims);

/* decay [b, H] float32 (output): the segment's total decay Lambda.  dt, A as
 * in ssd_fwd (dims.dt_softplus applies). */
ssd_status ssd_cp_segment_decay(const ssd_dims *dims, const float *dt, const float *A,
                                float *decay, void *workspace, size_t workspace_bytes,
                                void *stream);

/* nranks >= 1, 0 <= rank < nranks.  decays [nranks, b, H] and finals
 * [nranks, b, H, N, P] (float32, rank-ordered; entries of ranks after `rank`
 * are not read).  dt, A, C: this segment's, as in ssd_fwd.  y: this segment's
 * ssd_fwd output, updated in place (rank 0: unchanged).  h_final (output,
 * [b, H, N, P], may be NULL): the segment's true final state.  y and h_final
 * may not alias an input, the workspace or each other. */
ssd_status ssd_cp_correct(const ssd_dims *dims, int32_t nranks, int32_t rank,
                          const float *decays, const float *finals, const float *dt,
                          const float *A, const void *C, void *y, float *h_final,
                          void *workspace, size_t workspace_bytes, void *stream);

/* Allocation-free variant of ssd_fwd.  The pages have no counterpart: this
 * entry point exists for callers that cannot call cudaMalloc at the point
 * where they run the layer -- code working under a fixed device-memory plan
 * that forbids allocation after start-up, code inside a framework whose
 * caching allocator already owns the device memory (a raw cudaMalloc there
 * sits outside its accounting, or fails once the pool holds everything), and
 * latency-critical paths where cudaMalloc's implicit device synchronisation
 * is not acceptable.
 * Same arguments and results as ssd_fwd, without the workspace: the scratch
 * lives in a static device array of SSD_NOALLOC_SCRATCH_BYTES bytes inside
 * this library, which every GPU that loads the library holds until the
 * process exits.  Shapes whose ssd_fwd_workspace_size() exceeds that return
 * SSD_ERR_UNSUPPORTED before anything is launched.  The call allocates and
 * frees nothing itself, but the array's 64 MiB are claimed on a device when
 * the library's device code is loaded there -- under CUDA's lazy module
 * loading, at the first libssd call on that device, which may be this one;
 * if the device is full by then, that call returns SSD_ERR_CUDA.  Make one
 * warm-up call per device at start-up, before a memory plan or a caching
 * allocator takes the rest of the device.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address once and keeps it for the life of the process,
 *     so a device reset (cudaDeviceReset) is unsupported after that call.
 *   - All calls on a device share the one array and it keeps the previous
 *     call's contents; nothing in it needs to start at zero (every byte the
 *     kernels read is written earlier in the same call).  Calls that overlap
 *     on the GPU (different streams, or different host threads) race on the
 *     array: serialise them. */
#define SSD_NOALLOC_SCRATCH_BYTES (64ull << 20)
ssd_status ssd_fwd_noalloc(const ssd_dims *dims, const void *x, const float *dt, const float *A,
                           const void *B, const void *C, const float *D, const float *h0,
                           int32_t chunk, void *y, float *h_final, void *stream);

/* Synchronises `stream`, then reads and clears the library's device error
 * word: SSD_OK, or SSD_ERR_TIMEOUT if a kernel gave up a bounded wait since
 * the last check (its outputs are then invalid).  Diagnostic call; the only
 * entry point that synchronises. */
ssd_status ssd_check_device_error(void *stream);

/* Diagnostic of the bounded-wait path.  Every wait inside the library's
 * kernels gives up after a time limit, records SSD_ERR_TIMEOUT in the device
 * error word and lets the kernel finish (freeing its tensor memory) instead of
 * hanging or trapping.  This call launches one small kernel whose only work is
 * such a wait, on a barrier nothing completes, with the limit limit_ns
 * (1000 .. 1e9 ns, else SSD_ERR_INVALID_ARG) instead of the kernels' 2 s; the
 * next ssd_check_device_error(stream) then reports SSD_ERR_TIMEOUT and clears
 * it.  The context stays usable.  Not part of the layer (the pages have no
 * counterpart): it lets a caller check the failure path without a GPU fault. */
ssd_status ssd_selftest_timeout(int64_t limit_ns, void *stream);

/* Static, never-NULL description of a status code. */
const char *ssd_status_string(ssd_status status);

/* SSD_VERSION of the built library. */
int32_t ssd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBSSD_SSD_H */
