/*
 * sa.h -- C ABI of the banded + global sparse attention library (forward).
 *
 * The operation (one attention head, query row i, key row j, positions 0..N-1):
 *
 *   S_i = { j : |i-j| <= floor(w/2)*d  and  (i-j) mod d == 0 }  U  G ,
 *         and S_i = {0..N-1} when i is in G,
 *   out[i] = sum_{j in S_i} softmax_j(scale * <q_i, k_j>) v_j .
 *
 * w is the window, d the head's dilation, G the set of global positions.
 * Sources:
 *  - Ultralytics glossary "Longformer", section "How the Longformer attention
 *    works": a sliding window of w/2 positions on each side, a dilated window
 *    with gaps of d between attended positions at the same cost, and global
 *    tokens that attend to every position and are attended by every position.
 *    The section's mask-count example fixes "within w/2" as the inclusive test
 *    |i-j| <= w//2.
 *  - "GMAT: Global Memory Augmentation for Transformers", sections
 *    "Global-Memory Augmented Transformers" (sparse attention as an additive
 *    {0,-inf} mask on Q K^T) and "Global Memory" (M memory tokens prefixed to
 *    the sequence, dense in both directions).  GMAT memory is global_idx =
 *    0..M-1 over the concatenated [memory; main] sequence: that mask is
 *    identical to GMAT's main-sequence band plus dense memory rows/columns.
 *  - "Unlimiformer", section 2.3, Eq. (1): softmax(Q K^T / sqrt(d_k)) V; the
 *    caller passes scale (normally 1/sqrt(D)).
 *
 * Conventions for every entry point:
 *  - Tensors are device pointers, contiguous [B, H, N, D] with D fastest,
 *    16-byte aligned; the caller owns them.  q, k, v, out share one dtype.
 *    (sa_forward_host alone takes host buffers, and is synchronous.)
 *  - Host arrays (dilation, global_idx) are read during the call only; the
 *    caller may free them on return.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream); the call returns once it is enqueued.  Launch failures return
 *    SA_ERR_CUDA.  A kernel that detects a stalled wait records it in a
 *    per-device error word that sa_sync_status() reports as SA_ERR_TIMEOUT.
 *  - Validation happens before anything is launched; on any non-OK status
 *    nothing was enqueued and sa_last_error() describes the problem.
 *  - Thread safety: calls may come from several host threads and streams.
 *  - Device scratch comes from one stream-ordered pool per device, created on
 *    the first call there.  The environment variable SA_POOL_MAX_BYTES
 *    (decimal bytes, read at that moment) caps the pool; a call whose scratch
 *    does not fit returns SA_ERR_NO_MEMORY before any of its kernels is
 *    launched.
 *  - Stream capture: a call may be captured into a CUDA graph once a call of
 *    the same problem (B, H, N, D, window, dilation, global set, pattern) has
 *    run on the device outside capture -- that call builds and uploads the
 *    schedule.  A first call under capture returns SA_ERR_INVALID_ARG with
 *    nothing captured.  The schedule of a captured call is kept for the life
 *    of the process (the graph may replay at any time); its scratch is taken
 *    and returned by the graph's own stream-ordered allocation nodes.
 *    Profiling (sa_profile_begin) records no events for captured calls.
 */
#ifndef SA_H_
#define SA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *sa_stream_t; /* same type as cudaStream_t */

typedef enum {
  SA_OK = 0,
  SA_ERR_INVALID_ARG = 1, /* null pointer, bad size, index out of range      */
  SA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. D not 64/128)   */
  SA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed            */
  SA_ERR_TIMEOUT = 4,     /* a kernel gave up on a stalled wait              */
  SA_ERR_NO_MEMORY = 5    /* device scratch could not be allocated           */
} sa_status;

/*
 * Input / output element type and the precision of the products:
 *  SA_BF16  bf16 in memory; bf16 x bf16 products on the tensor cores, fp32
 *           accumulation and softmax, bf16 output.
 *  SA_FP32  fp32 in memory; fp32 arithmetic throughout on the CUDA cores,
 *           fp32 output.
 *  SA_TF32  fp32 in memory; the two products on the tensor cores in tf32 (the
 *           inputs' lowest 13 mantissa bits do not take part), fp32
 *           accumulation, softmax and output.  D = 64 only.  For scales near
 *           1/sqrt(D) the error is a fraction of bf16's; a scale several
 *           times larger sharpens the softmax until tf32 scores no longer meet
 *           fp32 accuracy -- use SA_FP32 there.
 */
typedef enum { SA_BF16 = 0, SA_FP32 = 1, SA_TF32 = 2 } sa_dtype;

/*
 * Precision of the P V product on the bf16 tensor-core path.  The softmax
 * weights P are computed in fp32; the tensor cores multiply bf16 operands.
 *  SA_PV_SINGLE  P is rounded to one bf16 value (8 significant bits).  The
 *                rounding errors of a row's weights average out over many
 *                comparable keys; on a row whose softmax rests on a few keys
 *                they do not, and the output error can exceed the library's
 *                tolerance |err| <= 2e-3 + 1e-2 |ref| where |ref| is small.
 *  SA_PV_SPLIT   P = P_hi + P_lo, two bf16 values (16 significant bits); the
 *                P V product runs over both (1.5x the tensor-core work of
 *                SA_PV_SINGLE).  The tolerance holds for every row.
 *  SA_PV_AUTO    (default) SA_PV_SPLIT when some non-global row sees fewer
 *                than 128 keys (a narrow window, a short chunk) or when
 *                |scale| sqrt(D) > 1.25 (scores sharper than the usual
 *                1/sqrt(D) scaling of unit-variance q and k), else
 *                SA_PV_SINGLE.  The choice looks at shapes and the scale
 *                only: inputs whose norms make the softmax sharp at the usual
 *                scale need SA_PV_SPLIT set explicitly.
 * SA_FP32 and SA_TF32 keep P in fp32 / tf32 and are not affected.
 */
typedef enum { SA_PV_AUTO = 0, SA_PV_SINGLE = 1, SA_PV_SPLIT = 2 } sa_pv_mode;

/*
 * sa_set_pv_mode -- process-wide choice for the calls enqueued after it
 * returns (an atomic setting; calls already enqueued are not affected).
 * SA_ERR_INVALID_ARG for an unknown mode.  sa_get_pv_mode returns the setting.
 */
sa_status sa_set_pv_mode(sa_pv_mode mode);
sa_pv_mode sa_get_pv_mode(void);

/*
 * sa_uses_split_p -- 1 if a bf16 call with these shapes and scale would split
 * P under the current setting, else 0 (chunk = 0 for the band pattern, else
 * the chunk length and n_memory of sa_forward_chunked).  Host only.
 */
int sa_uses_split_p(int N, int D, int window, const int32_t *dilation, int H,
                    const int32_t *global_idx, int n_global, int chunk, int n_memory,
                    float scale);

/* Largest number of distinct global positions accepted. */
#define SA_MAX_GLOBALS 256

/*
 * sa_forward -- out = banded + global sparse attention of (q, k, v).
 *
 *  q, k, v   device, [B,H,N,D] in `dtype`; read only.
 *  out       device, [B,H,N,D] in `dtype`; fully written.
 *  B, H, N   >= 1.   D: 64 or 128 (else SA_ERR_UNSUPPORTED).
 *  window    w >= 0; half-width floor(w/2).
 *  dilation  host, H entries >= 1 (per head), or NULL for all 1.
 *  global_idx host, n_global entries in [0, N); duplicates are merged (a set).
 *            May be NULL when n_global == 0.  At most SA_MAX_GLOBALS distinct.
 *  scale     multiplier of q.k before the softmax (finite).
 *  dtype     SA_BF16, SA_FP32 or SA_TF32 (see sa_dtype; SA_TF32 with D other
 *            than 64 is SA_ERR_UNSUPPORTED).
 *  stream    cudaStream_t on which all work is enqueued.
 *
 * Device scratch (gathered global rows, split-K partials) comes from a
 * library-owned stream-ordered pool; exhaustion returns SA_ERR_NO_MEMORY.
 */
sa_status sa_forward(const void *q, const void *k, const void *v, void *out, int B,
                     int H, int N, int D, int window, const int32_t *dilation,
                     const int32_t *global_idx, int n_global, float scale,
                     sa_dtype dtype, sa_stream_t stream);

/*
 * sa_forward_lse -- sa_forward, and also the natural-log log-sum-exp of each
 * row's masked scores: lse[b,h,i] = log(sum_{j in S_i} exp(scale*<q_i,k_j>)).
 *  lse   device, [B,H,N] float32, or NULL (then identical to sa_forward).
 */
sa_status sa_forward_lse(const void *q, const void *k, const void *v, void *out,
                         float *lse, int B, int H, int N, int D, int window,
                         const int32_t *dilation, const int32_t *global_idx,
                         int n_global, float scale, sa_dtype dtype,
                         sa_stream_t stream);

/*
 * sa_forward_global_proj -- sa_forward_lse with separate projections for the
 * global attention (Ultralytics glossary "Longformer", section "How the
 * Longformer attention works": the global attention has query, key and value
 * projections of its own).  A global row i scores scale * <q_global_i,
 * k_global_j> over every key j and averages v_global; every other row uses
 * q, k, v for its band keys and its global keys alike, exactly as
 * sa_forward_lse.  The mask, and so sa_count_pairs, is that of sa_forward.
 *
 *  q_global, k_global, v_global  device, [B,H,N,D] in `dtype`, 16-byte
 *            aligned, non-null; read only.  Only the global rows of q_global
 *            are read; k_global and v_global are read in full when
 *            n_global > 0 and not at all otherwise.
 *  Other arguments, errors and stream semantics: as sa_forward_lse.
 */
sa_status sa_forward_global_proj(const void *q, const void *k, const void *v,
                                 const void *q_global, const void *k_global,
                                 const void *v_global, void *out, float *lse, int B, int H,
                                 int N, int D, int window, const int32_t *dilation,
                                 const int32_t *global_idx, int n_global, float scale,
                                 sa_dtype dtype, sa_stream_t stream);

/*
 * sa_forward_host -- sa_forward_lse on host buffers: the inputs are copied to
 * the current device, the attention runs there, and out (and lse) are copied
 * back; the call returns when they are written (synchronous).
 *
 * Every (b, h) slice is a problem of its own (its band, its global rows and
 * its output involve that slice only), so the call cuts the slices into
 * groups of consecutive heads and pipelines them over two sets of device
 * buffers on three streams of its own: group g+1's inputs are copied in while
 * group g is computed and group g-1's output is copied out.
 *
 *  q, k, v   host, [B,H,N,D] in `dtype`, contiguous; read only.  Page-locked
 *            memory (cudaHostAlloc, cudaHostRegister) lets the copies run
 *            asynchronously and overlap the computation; pageable memory
 *            gives the same result with the copies serialised on the host.
 *  out       host, [B,H,N,D] in `dtype`; fully written.
 *  lse       host, [B,H,N] float32, or NULL.
 *  heads_per_group  slices per group: 0 lets the library choose (about sixteen
 *            groups of at least 32 MiB of inputs each); a value below H splits
 *            each batch element's heads into groups of that many; H or more
 *            takes floor(heads_per_group / H) whole batch elements per group.
 *  Other arguments: as sa_forward (no alignment rule for the host buffers).
 *
 * Device memory: two buffer sets of one group's q, k, v, out (and lse) from
 * the library's stream-ordered pool, plus each group's sa_forward scratch;
 * SA_ERR_NO_MEMORY if they cannot be had.  Every argument is checked before
 * any copy.  On any status, everything the call enqueued has finished when it
 * returns.  Like sa_sync_status, it reports (and clears) the device error
 * word at the end: SA_ERR_TIMEOUT if a kernel gave up on a stalled wait.
 */
sa_status sa_forward_host(const void *q, const void *k, const void *v, void *out, float *lse,
                          int B, int H, int N, int D, int window, const int32_t *dilation,
                          const int32_t *global_idx, int n_global, float scale, sa_dtype dtype,
                          int heads_per_group);

/*
 * sa_count_pairs -- exact number of (i, j) pairs in the mask, |S_i| summed
 * over i, per head (per_head[H], may be NULL) and over all heads of one batch
 * element (*total, may be NULL).  Host only, integer arithmetic, no GPU use.
 * Same arguments and validation as sa_forward.  The in-mask FLOP count of a
 * call is 4 * D * B * total (2D for q.k and 2D for p*v per pair).
 * This is the count of the mask-count example in the Ultralytics glossary
 * "Longformer", section "How the Longformer attention works" (window 512,
 * global token 0): 461,054 / 988,414 / 2,043,134 scored pairs at
 * N = 1024 / 2048 / 4096, which the section prints rounded as 0.5M / 1.0M /
 * 2.0M against full attention's N^2.
 */
sa_status sa_count_pairs(int N, int window, const int32_t *dilation, int H,
                         const int32_t *global_idx, int n_global, int64_t *per_head,
                         int64_t *total);

/*
 * sa_forward_chunked -- GMAT chunked self-attention with a global memory
 * ("GMAT: Global Memory Augmentation for Transformers", subsection "Chunked
 * self-attention", with the memory of section "Global Memory").  The sequence
 * of N positions is [memory; main]: positions [0, n_memory) are memory tokens,
 * which score every position and are scored by every position; the main
 * positions are cut into contiguous chunks of `chunk` positions starting at
 * n_memory (the last chunk may be shorter), and a main position scores the
 * main positions of its own chunk plus the memory.  With n_memory = 0 each
 * chunk is plain attention over `chunk` positions; with chunk >= N - n_memory
 * it is plain attention over the whole sequence.
 *
 *  q, k, v, out, lse, B, H, N, D, scale, dtype, stream: as sa_forward_lse
 *    (device pointers, contiguous [B, H, N, D], 16-byte aligned; lse may be
 *    NULL; output dtype = input dtype).
 *  n_memory  0 <= n_memory <= N, at most SA_MAX_GLOBALS (else
 *            SA_ERR_UNSUPPORTED).
 *  chunk     >= 1.
 *  Errors: SA_ERR_INVALID_ARG / SA_ERR_UNSUPPORTED before any launch, as for
 *  sa_forward.  Asynchronous on `stream`.
 */
sa_status sa_forward_chunked(const void *q, const void *k, const void *v, void *out, float *lse,
                             int B, int H, int N, int D, int n_memory, int chunk, float scale,
                             sa_dtype dtype, sa_stream_t stream);

/*
 * sa_count_pairs_chunked -- exact number of in-mask (i, j) pairs of one head of
 * sa_forward_chunked: n_memory * N for the memory rows plus, per chunk of
 * length c, c * (n_memory + c).  Host only.  Same validation as
 * sa_forward_chunked; per_head must be non-null.
 */
sa_status sa_count_pairs_chunked(int N, int n_memory, int chunk, int64_t *per_head);

/*
 * sa_forward_gather -- attention over per-query key lists ("Unlimiformer:
 * Long-Range Transformers with Unlimited Length Input", section 2.2
 * "Retrieval-augmented Cross-Attention": each head retrieves the top-k keys of
 * a query and attends only to them; section 2.3 Eq. (1): standard dot-product
 * attention over that set).  The retrieval (a kNN index) is the caller's; this
 * call takes its result.  Row i of head (b, h):
 *   out[b,h,i] = sum_t softmax_t(scale * <q[b,h,i], k[b,h,idx_t]>) v[b,h,idx_t]
 * over the valid entries idx_t = idx[b,h,i,t], t < K.
 *
 *  q         device, [B,H,Nq,D] in `dtype`; read only.
 *  k, v      device, [B,H,Nk,D] in `dtype`; read only.
 *  idx       device, int32 [B,H,Nq,K]; read only.  An entry outside [0, Nk)
 *            (e.g. -1) is padding and is skipped, so lists may be ragged; an
 *            index listed twice counts twice (retrieval output has no repeats).
 *            May be NULL when K == 0.
 *  out       device, [B,H,Nq,D] in `dtype`; fully written.  A row with no valid
 *            entry gets zeros.
 *  lse       device, float32 [B,H,Nq], or NULL: natural-log log-sum-exp of the
 *            row's scores (-inf for a row with no valid entry).
 *  B, H, Nq, Nk >= 1; K >= 0; D: 64 or 128 (else SA_ERR_UNSUPPORTED).
 *  scale     finite.  dtype: SA_BF16 or SA_FP32 (fp32 arithmetic either way).
 *  q, k, v, out 16-byte aligned; idx, lse 4-byte aligned.
 *  Errors: SA_ERR_INVALID_ARG / SA_ERR_UNSUPPORTED before any launch;
 *  SA_ERR_CUDA if the launch fails.  Asynchronous on `stream`; allocates no
 *  device memory.  Timed as stage 1 by sa_profile_begin/end.
 */
sa_status sa_forward_gather(const void *q, const void *k, const void *v, const int32_t *idx,
                            void *out, float *lse, int B, int H, int Nq, int Nk, int D, int K,
                            float scale, sa_dtype dtype, sa_stream_t stream);

/*
 * sa_check_stalled_wait -- exercises the failure detection of the kernels
 * without a GPU fault: enqueues on `stream` one small kernel that waits on a
 * barrier nothing will ever arrive on, through the same bounded wait the
 * attention kernels use, but giving up after `limit_us` microseconds (1 ..
 * 2,000,000) instead of two seconds.  It then sets the device error word and
 * returns, leaving the context usable: the next sa_sync_status(stream) returns
 * SA_ERR_TIMEOUT (and clears the word).  SA_ERR_INVALID_ARG for a limit out of
 * range; SA_ERR_CUDA if the launch fails.
 */
sa_status sa_check_stalled_wait(uint32_t limit_us, sa_stream_t stream);

/* Thread-local description of the last non-OK status on this host thread. */
const char *sa_last_error(void);

/*
 * sa_sync_status -- waits for `stream`, then reports (and clears) the current
 * device's error word: SA_ERR_TIMEOUT if a kernel gave up on a stalled wait,
 * SA_ERR_CUDA if the stream reported an error, else SA_OK.
 */
sa_status sa_sync_status(sa_stream_t stream);

/*
 * Per-stage timing.  Between sa_profile_begin() and sa_profile_end(), every
 * sa_forward* call records CUDA events around each of its kernel launches on
 * its own stream.  sa_profile_end() waits for those events and returns, per
 * stage, the number of launches and their summed device time in milliseconds.
 * Stages: 0 gather of global rows, 1 band tiles (with the global-row split-K
 * work when it runs in the same launch, as on the tensor cores with at most
 * 16 residue classes; or the list attention of sa_forward_gather),
 * 2 global-row split-K pass as a launch of its own, 3 merge of partial
 * softmax statistics.  Process-wide; not for concurrent use from several
 * threads.  Each launch is also an NVTX range ("sa.band", "sa.merge", ...).
 */
#define SA_NUM_STAGES 4
typedef struct {
  int64_t launches[SA_NUM_STAGES];
  double ms[SA_NUM_STAGES];
} sa_profile;

sa_status sa_profile_begin(void);
sa_status sa_profile_end(sa_profile *out);

/*
 * sa_forward_noalloc -- sa_forward_lse without any device memory allocation.
 *
 * No passage of the source pages corresponds to this call: it exists for
 * callers that must not allocate device memory while they run attention --
 * a host application that owns the whole device memory budget (for example
 * through its own pool), an allocator-free plug-in or runtime, or code that
 * runs where allocation is not allowed.  sa_forward takes its scratch (the
 * band-tile work list, the gathered global rows, the split-K partial softmax
 * statistics) from a library-owned pool and caches schedules in cudaMalloc'ed
 * buffers; this call takes all of it from one static device array of
 * SA_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that
 * loads the library holds until the process exits.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 *  Arguments, layouts, ownership and validation are those of sa_forward_lse
 *  (lse may be NULL).  The arithmetic runs on the CUDA cores in fp32 for every
 *  input type (bf16 in and out for SA_BF16; SA_TF32 runs as SA_FP32), so results agree with
 *  sa_forward_lse within the library's stated tolerance, not bit for bit.
 *
 *  Size limit: a problem whose scratch does not fit the array even after the
 *  global-row pass is split into fewer key chunks is rejected with
 *  SA_ERR_UNSUPPORTED and a message giving the bytes it needs; nothing is
 *  launched.  (One 131072-long sequence with 16 heads, D = 128 and 64
 *  globals fits.)
 *
 *  Set-up: the first call on each device looks up the device address of the
 *  static array (with that device current), and so does the first call after
 *  the device's CUDA context has been replaced (a device reset invalidates
 *  the address; the library notices the new context and looks it up again).
 *  Make that first call before any stream capture begins.
 *
 *  Work lists: the band-tile and global-row work lists are written into the
 *  array by a small kernel on `stream` from values passed as kernel
 *  parameters; no host buffer is copied and the call does not wait for the
 *  stream.
 *
 *  Sharing: every call uses the same array, which keeps what the last call
 *  left there.  Each call writes every scratch byte it later reads, so nothing
 *  needs clearing between calls, but calls whose work overlaps on the GPU
 *  (different streams, or different host threads) race on the array: order
 *  them on one stream or synchronise between them.
 */
#define SA_NOALLOC_SCRATCH_BYTES (8u << 20)
sa_status sa_forward_noalloc(const void *q, const void *k, const void *v, void *out,
                             float *lse, int B, int H, int N, int D, int window,
                             const int32_t *dilation, const int32_t *global_idx,
                             int n_global, float scale, sa_dtype dtype,
                             sa_stream_t stream);

/* Library version string. */
const char *sa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SA_H_ */
