/*
 * gc.h -- C ABI of the GB300 error-feedback gradient-compression library
 * (libgc.so, hand-written sm_103a CUDA).
 *
 * The method (page titles and sections it follows):
 *  - mbrenndoerfer.com "Gradient Compression", Top-K Sparsification:
 *      g^_t = TopK(g_t + e_{t-1}),   e_t = (g_t + e_{t-1}) - g^_t,
 *    with a sparse wire format of one fp32 value plus one int32 index per
 *    kept entry; 1-bit SGD, Q(g) = sign(g) * ||g||_1 / d with a per-layer
 *    scalar; QSGD, Q_s(g) = ||g|| * sgn(g) * xi(g, s) with stochastic
 *    rounding; the union of per-worker sparse vectors on the receiver.
 *  - inferensys.com "Gradient Compression" (zh glossary): Random-k with a
 *    per-iteration random mask; the Top-k + 8-bit pipeline; all-gather of
 *    sparse indices and values.
 *  - inferensys.com "Gradient Compression" (genomic glossary) and
 *    "Gradient Sparsification": per-layer selection, 8-bit quantization,
 *    stochastic rounding, DGC momentum correction and momentum factor masking.
 *
 * Data model.  A gradient is a flat fp32 "arena"; tensor t (a layer)
 * occupies elements [off[t], off[t+1]) and is compressed independently.
 * n_t = off[t+1] - off[t] must satisfy 1 <= n_t <= 2^31 - 1.  Sparse
 * payloads list, per tensor, k_t entries in ascending TENSOR-LOCAL int32
 * index order, tensor t's entries at [koff[t], koff[t+1]) with koff the
 * prefix sum of k.  Sign bits are packed LSB-first, 32 per uint32 word, each
 * tensor starting on a new word (word offset = sum of ceil(n_t'/32) over
 * t' < t), pad bits zero.
 *
 * Order of selection.  Top-k keeps the k_t elements of largest |x|; equal
 * magnitudes (and +0 / -0) go to the lower index.  Random-k keeps the k_t
 * smallest Philox keys, ties to the lower index.
 *
 * Random numbers.  Philox4x32-10 (Salmon et al., SC'11).  Element i of the
 * arena, call (seed, iter) and purpose p (1 int8 rounding, 2 QSGD, 3
 * random-k) uses word (i mod 4) of the block with counter
 * (lo32(i/4), hi32(i/4), lo32(iter), p) and key (lo32(seed), hi32(seed)).
 * Stochastic rounding rounds |x| up iff r * 2^-32 < frac(|x|).
 *
 * Arithmetic.  IEEE fp32, round to nearest even, one rounding per written
 * operation (no fused multiply-add, no flush to zero).  Results are
 * bit-identical from run to run; per-tensor norms are reduced in a fixed
 * order.
 *
 * Conventions for every entry point.
 *  - Pointers named "device" point to device memory owned by the caller;
 *    the library never allocates, frees or retains them.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work and return; nothing synchronises except
 *    gc_get_device_status.
 *  - A layout is passed twice: `dev` (its arrays in device memory, read by
 *    the kernels) and `host` (the same values in host memory, used for
 *    validation and launch sizing).  They must hold identical values; a
 *    mismatch in the totals is detected on the device and reported by
 *    gc_get_device_status as GC_DIAG_LAYOUT_MISMATCH, and all kernels of
 *    that call then do nothing.
 *  - `workspace` is caller-owned device scratch of at least
 *    gc_workspace_size() bytes for that operation and layout, 256-byte
 *    aligned.  It may be reused between calls but not shared by calls that
 *    run concurrently.
 *  - Buffers must not alias each other, except where stated.
 *  - g, e, u, v, out must be 16-byte aligned.
 *  - Argument errors are returned before anything is enqueued.  No C++
 *    exception crosses this interface.
 *
 * Buckets.  A layout may describe tensors t0 .. t1-1 of a larger arena: off
 * and koff are then that arena's own offsets of those tensors (off[0] and
 * koff[0] need not be 0), so the arena's own layout arrays serve:
 * {t1 - t0, off + t0, k + t0, koff + t0}, on the host and on the device.  Per-element arrays (g, e, u, v, out, dense int8 /
 * QSGD codes) and per-entry arrays (idx, val, q) are passed as the WHOLE
 * arena's arrays and are read and written at those offsets only; per-tensor
 * arrays (k, scale, mean_abs, thresholds, norms, counts, residual
 * descriptors) and sign-bit words are passed offset to the bucket's first
 * tensor (its word offset is the sum of ceil(n / 32), or of ceil(k / 32) for
 * the kept-value bits, over the arena's earlier tensors).  Random numbers
 * are drawn at arena indices, so compressing an arena bucket by bucket, in
 * any order or concurrently on several streams (each call with its own
 * workspace), gives exactly the whole-arena call's outputs: a training loop
 * can compress each bucket as soon as backward has produced its gradients.
 */
#ifndef GC_H_
#define GC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gc_status {
  GC_OK = 0,
  GC_ERR_INVALID_ARG = 1, /* null pointer where one is required, bad flag or mode */
  GC_ERR_LAYOUT = 2,      /* off[0] or koff[0] negative, off not increasing, n_t >= 2^31,
                             k_t > n_t, koff[t+1] - koff[t] != k_t */
  GC_ERR_WORKSPACE = 3,   /* workspace NULL, misaligned or smaller than gc_workspace_size */
  GC_ERR_ALIGNMENT = 4,   /* a data pointer is not 16-byte aligned */
  GC_ERR_CUDA = 5,        /* a CUDA launch or copy failed (cudaGetLastError) */
  GC_ERR_DEVICE = 6       /* gc_get_device_status found an error word set on the device */
} gc_status;

/* Flags of the sparse compressors. */
#define GC_EF 0x1u          /* error feedback: acc = g + e, residual written back to e */
#define GC_INT8 0x2u        /* Top-k only: kept values sent as int8 codes + one fp32 scale per tensor */
#define GC_RANDK 0x4u       /* random-k selection instead of Top-k */
#define GC_UNBIASED 0x8u    /* random-k only, without GC_EF: send g * (n/k), no residual */
#define GC_NO_MASK 0x10u    /* momentum only: keep u on the selected set (no factor masking) */
#define GC_LAZY 0x20u       /* set by gc_ef_topk_compress_lazy; not accepted elsewhere */
#define GC_FORCE_EXACT 0x100u /* select with full passes over the tensor instead of the
                                 sampled candidate threshold (same results; for testing) */
#define GC_MULTI_KERNEL 0x200u /* Top-k: run the multi-kernel pipeline even where the one-launch
                                  path would (same results; for testing and comparison) */

/* Operations, for gc_workspace_size. */
typedef enum gc_op {
  GC_OP_TOPK = 0,       /* gc_ef_topk_compress (Top-k and random-k) */
  GC_OP_MOMENTUM = 1,   /* gc_ef_topk_compress_momentum */
  GC_OP_SIGN = 2,       /* gc_sign_compress */
  GC_OP_QUANTIZE = 3,   /* gc_quantize_stochastic */
  GC_OP_DECOMPRESS = 4  /* gc_sparse_decompress_accumulate, gc_dense_decompress_accumulate */
} gc_op;

/* Dense quantizer modes. */
#define GC_Q_INT8 0 /* s = max|acc| / 127, code = sgn * min(127, SR(|acc| / s)) */
#define GC_Q_QSGD 1 /* N = ||acc||_2, code = sgn * min(s, SR(|acc| * s / N)) */

/* Dense payload kinds for gc_dense_decompress_accumulate. */
#define GC_DENSE_SIGN 0
#define GC_DENSE_INT8 1
#define GC_DENSE_QSGD 2

typedef struct gc_layout {
  int32_t num_tensors;  /* T >= 1 */
  const int64_t* off;   /* [T+1] element offsets, strictly increasing; off[0] = 0 for a whole
                           arena, > 0 for a bucket (see Buckets above) */
  const int64_t* k;     /* [T] kept entries per tensor, 0 <= k_t <= n_t; may be NULL for dense ops */
  const int64_t* koff;  /* [T+1] koff[t+1] = koff[t] + k_t; koff[0] = 0 for a whole arena, the
                           arena's own koff of the first tensor for a bucket; may be NULL for
                           dense ops */
} gc_layout;

/* Diagnostics of the last call that used a workspace. */
typedef struct gc_diag {
  uint32_t error_bits;       /* GC_DIAG_* bits */
  uint32_t exact_tensors;    /* tensors selected by full passes (fallback or GC_FORCE_EXACT) */
  uint32_t overflow_tensors; /* tensors whose candidate list overflowed (then selected exactly) */
  uint32_t one_launch;       /* 1 if the call ran as one cooperative launch (see GC_MULTI_KERNEL) */
} gc_diag;

#define GC_DIAG_LAYOUT_MISMATCH 0x1u /* dev and host layouts disagree; the call did nothing */
#define GC_DIAG_SELECT 0x2u          /* internal selection inconsistency (should never be set) */
#define GC_DIAG_INDEX_RANGE 0x4u     /* decompress met a payload index >= n_t; entry skipped */
#define GC_DIAG_BAD_THRESHOLD 0x8u   /* a threshold or clipping norm was negative or NaN */
#define GC_DIAG_INDEX_ORDER 0x10u    /* decompress met a worker's indices not ascending within a
                                        tensor; see gc_sparse_decompress_accumulate */
#define GC_DIAG_TIMEOUT 0x20u        /* a grid-wide wait of the one-launch path ran out (about a
                                        second); that call's outputs are incomplete */

/* CUDA-graph capture.  gc_ef_topk_compress_dev_iter and
 * gc_quantize_stochastic_dev_iter are gc_ef_topk_compress and
 * gc_quantize_stochastic with the iteration counter in device memory: the
 * kernels read *iter_dev where the other entry points take `iter`, and the
 * call ends by adding 1 to *iter_dev.  A call captured once into a graph
 * therefore replays as successive steps (fresh random-k keys and stochastic
 * rounding draws), with results bit-identical to calling the plain entry
 * point with iter = 0, 1, 2, ... from the counter's starting value.  The
 * calls enqueue only kernels and memsets on `stream` (no allocation, no
 * synchronization), so they can be captured.
 *   iter_dev: device uint64, 8-byte aligned; nothing else may write it
 *             while the call runs.  Other arguments as the plain entry. */
/* Bytes of workspace that operation `op` needs for layout `host` and
 * `flags`.  *bytes is set on GC_OK. */
gc_status gc_workspace_size(const gc_layout* host, int32_t op, uint32_t flags, size_t* bytes);

/* EF Top-k (or random-k) compression of a whole arena (mbrenndoerfer.com
 * "Gradient Compression", Top-K Sparsification equations; inferensys.com
 * zh glossary, Random-k and Top-k + 8-bit).
 *   acc = g + e        (GC_EF; without it acc = g and e may be NULL)
 *   S_t = the k_t kept elements of tensor t (Top-k by |acc|, or random-k)
 *   payload: idx[koff[t] + j] = local index of the j-th kept element
 *            (ascending); val = acc there, or with GC_INT8 q = int8 code,
 *            scale[t] = max|acc_t| / 127, and val (optional) = q * scale[t];
 *            GC_RANDK|GC_UNBIASED: val = g * (float)(n_t / k_t), no EF
 *   residual (GC_EF): e = acc off S, +0 on S, or acc - q * scale with GC_INT8.
 * g: device fp32[N] (read only).  e: device fp32[N] in/out.  idx: device
 * int32[sum k].  val: device fp32[sum k] (required without GC_INT8,
 * optional with it).  q: device int8[sum k] and scale: device fp32[T],
 * both required iff GC_INT8.  seed, iter: Philox key and counter words.
 * GC_INT8 cannot be combined with GC_RANDK.
 * Launches.  Top-k on an arena of at most 2^22 elements in at most 1024
 * tensors runs as one cooperative launch (all CTAs resident) whose phases
 * meet at three or four grid-wide barriers; every wait there is bounded and sets
 * GC_DIAG_TIMEOUT if it runs out.  gc_diag.one_launch reports it.  Other
 * arenas, random-k, GC_FORCE_EXACT and GC_MULTI_KERNEL use the multi-kernel
 * pipeline (14 kernels chained as programmatic dependent launches: each
 * waits for the previous one's completion before touching memory).  Both
 * give identical results. */
gc_status gc_ef_topk_compress(const gc_layout* dev, const gc_layout* host, const float* g, float* e,
                              int32_t* idx, float* val, int8_t* q, float* scale, uint64_t seed,
                              uint64_t iter, uint32_t flags, void* workspace, size_t ws_bytes,
                              void* stream);
gc_status gc_ef_topk_compress_dev_iter(const gc_layout* dev, const gc_layout* host, const float* g,
                                       float* e, int32_t* idx, float* val, int8_t* q, float* scale,
                                       uint64_t seed, uint64_t* iter_dev, uint32_t flags,
                                       void* workspace, size_t ws_bytes, void* stream);

/* EF Top-k with DGC local gradient clipping (genomic glossary "Gradient
 * Compression", DGC: local gradient clipping normalizes the gradient's
 * magnitude before compression; zh glossary: clipping before quantization
 * controls the range).  Per tensor: N = ||g_t||_2 (fp64 sum in a fixed
 * order), g' = (C / N) * g when N > C (C / N rounded to fp32), else g; then
 * gc_ef_topk_compress(GC_EF | flags) on g'.
 *   max_norm: device fp32[T], C >= 0 (negative or NaN: no clipping, and
 *             GC_DIAG_BAD_THRESHOLD is set).
 *   norm:     device fp32[T] out: N (within 1e-6 relative of an fp64 sum).
 * flags: GC_EF (required), GC_INT8, GC_FORCE_EXACT.  Reads g twice (norm,
 * then the streaming pass). */
gc_status gc_ef_topk_compress_clipped(const gc_layout* dev, const gc_layout* host, const float* g,
                                      float* e, const float* max_norm, float* norm, int32_t* idx,
                                      float* val, int8_t* q, float* scale, uint64_t seed,
                                      uint64_t iter, uint32_t flags, void* workspace,
                                      size_t ws_bytes, void* stream);

/* Threshold sparsification with EF (genomic glossary "Gradient
 * Compression": gradients below a fixed or adaptive magnitude threshold are
 * dropped; "Gradient Sparsification": the threshold adapts to each
 * iteration's distribution).  Tensor t keeps every element with
 * |acc| >= tau[t], at most k_t of them (the largest, in the Top-k order);
 * payload, int8 option and residual as gc_ef_topk_compress.
 *   tau:   device fp32[T], >= 0 (the caller adapts it between calls if it
 *          wants an adaptive threshold); a negative or NaN entry keeps
 *          nothing and sets GC_DIAG_BAD_THRESHOLD.
 *   count: device int64[T] out: entries kept; tensor t's payload is
 *          [koff[t], koff[t] + count[t]) of the k_t slots, the rest untouched.
 * flags: GC_EF, GC_INT8, GC_FORCE_EXACT.  Workspace: gc_workspace_size(
 * GC_OP_TOPK, flags) is sufficient. */
gc_status gc_ef_threshold_compress(const gc_layout* dev, const gc_layout* host, const float* g,
                                   float* e, const float* tau, int64_t* count, int32_t* idx,
                                   float* val, int8_t* q, float* scale, uint64_t seed,
                                   uint64_t iter, uint32_t flags, void* workspace, size_t ws_bytes,
                                   void* stream);

/* Density (fraction of elements kept) of a warm-up schedule ("Gradient
 * Sparsification", warm-up: sparsity introduced gradually over the first
 * iterations by a linear, exponential or step schedule): from rho_start at
 * step 0 to rho_final at step >= warmup_steps.
 *   kind 0 linear: rho_start + (rho_final - rho_start) * f
 *   kind 1 exponential: rho_start * (rho_final / rho_start)^f
 *   kind 2 step: kind 1 evaluated at f rounded down to a multiple of 1/stages
 * with f = step / warmup_steps.  Host only; k_t = min(n_t, ceil(density * n_t)). */
double gc_warmup_density(int64_t step, int64_t warmup_steps, double rho_start, double rho_final,
                         int32_t kind, int32_t stages);

/* gc_ef_topk_compress with timing hooks: `events` is a host array of
 * `n_events` (0..32) cudaEvent_t handles created by the caller, recorded on
 * `stream`.  With n_events <= 5 they mark the phases of the call: [0] start,
 * [1] before the streaming pass over g and e, [2] after it, [3] after the
 * k-th key search, [4] after the payload write.  With n_events > 5, [0] marks
 * the start and [j] the end of the j-th operation the call enqueues (for
 * per-kernel timing).  NULL entries are skipped.  Results are identical to
 * gc_ef_topk_compress. */
gc_status gc_ef_topk_compress_profiled(const gc_layout* dev, const gc_layout* host, const float* g,
                                       float* e, int32_t* idx, float* val, int8_t* q, float* scale,
                                       uint64_t seed, uint64_t iter, uint32_t flags,
                                       void* workspace, size_t ws_bytes, void* stream,
                                       void* const* events, int32_t n_events);

/* Residual of one tensor kept in pending form by gc_ef_topk_compress_lazy
 * (device memory, caller-owned; all-zero = no pending selection). */
typedef struct gc_residual_desc {
  uint32_t flags;    /* bit 0: a selection is pending; bit 1: it was int8-quantized */
  uint32_t thr;      /* selection key of the k-th kept element: (bits(acc) << 1) */
  int32_t last_tie;  /* largest kept local index among elements whose key == thr */
  float scale;       /* int8 scale of that call */
  uint64_t seed;     /* Philox key of that call */
  uint64_t iter;     /* Philox counter word of that call */
} gc_residual_desc;

/* EF Top-k (+ int8) with the residual update deferred ("lazy" residual).
 * The pages' residual e_t = (g_t + e_{t-1}) - g^_t is not scattered into e
 * at the kept positions; instead e keeps acc everywhere and rd[t] records
 * which elements were kept (every element whose key exceeds thr, plus those
 * equal to thr up to last_tie) and, for int8, how their codes were drawn.
 * The next call's streaming pass recomputes the exact residual of each
 * element from (e, rd) in registers before adding g, which saves the k
 * random read-modify-writes of the eager update.  Payloads are bit-identical
 * to gc_ef_topk_compress(GC_EF | flags), and gc_ef_residual_materialize turns
 * (e, rd) into the plain residual (for checkpoints or switching to the eager
 * entry point).
 *   e:  device fp32[N], pending residual in/out (a plain residual when rd is
 *       all zero, e.g. before the first call).
 *   rd: device gc_residual_desc[T], in/out.
 * flags: GC_INT8 and GC_FORCE_EXACT are accepted; GC_EF is implied; the
 * layout must not change between calls sharing (e, rd). */
gc_status gc_ef_topk_compress_lazy(const gc_layout* dev, const gc_layout* host, const float* g,
                                   float* e, gc_residual_desc* rd, int32_t* idx, float* val,
                                   int8_t* q, float* scale, uint64_t seed, uint64_t iter,
                                   uint32_t flags, void* workspace, size_t ws_bytes, void* stream);

/* Applies the pending residual of gc_ef_topk_compress_lazy: e <- the exact
 * EF residual, rd <- all zero.  One pass over the tensors with a pending
 * selection; no workspace. */
gc_status gc_ef_residual_materialize(const gc_layout* dev, const gc_layout* host, float* e,
                                     gc_residual_desc* rd, void* stream);

/* Matrix layout for PowerSGD: matrix t is row-major rows[t] x cols[t] at
 * element offset start[t] of the gradient arena (matrices must not overlap;
 * vectors such as biases are left out and sent some other way). */
typedef struct gc_matrix_layout {
  int32_t num_tensors;  /* T >= 1 */
  const int64_t* start; /* [T] element offset of matrix t */
  const int64_t* rows;  /* [T] m_t >= 1 */
  const int64_t* cols;  /* [T] n_t >= 1 */
} gc_matrix_layout;

/* Workspace bytes for gc_powersgd_compress / _decompress_accumulate. */
gc_status gc_powersgd_workspace_size(const gc_matrix_layout* host, int32_t rank, size_t* bytes);

/* PowerSGD with error feedback (mbrenndoerfer.com "Gradient Compression",
 * PowerSGD section: G ~ P Q^T found by power iteration, error feedback on
 * G - P Q^T; chipfoundryservices.com glossary: rank-4 PowerSGD).  One
 * warm-started power-iteration step per call, per matrix:
 *   M = G + E;  P = M Q;  orthonormalize P's columns (modified
 *   Gram-Schmidt);  Q = M^T P;  E = M - P Q^T.
 * Sums over rows or columns are reduced in a fixed order (fp32 compensated
 * partials, fp64 across them); the elementwise steps are single fp32
 * roundings: s_ij = sum_k P_ik Q_jk accumulated in k order, E = M - s.
 *   rank: 1, 2 or 4.
 *   g: device fp32 arena (read);  e: device fp32 arena, residual in/out.
 *   q: device fp32[sum_t cols[t] * rank], row-major n_t x rank per matrix:
 *      in, the previous call's Q (warm start; any full-rank start the first
 *      time); out, this call's Q.
 *   p: device fp32[sum_t rows[t] * rank] out, orthonormal columns.
 *   p_raw: device fp32 like p, or NULL: receives P = M Q before
 *      orthonormalization.
 * Payload of a call: p and q ((m + n) * rank values per matrix). */
gc_status gc_powersgd_compress(const gc_matrix_layout* dev, const gc_matrix_layout* host,
                               int32_t rank, const float* g, float* e, float* q, float* p,
                               float* p_raw, void* workspace, size_t ws_bytes, void* stream);

/* gc_powersgd_compress with the residual kept pending: the step's last pass,
 * E = M - P Q^T, is not run; e keeps M, and the next call makes the residual
 * element by element (same fp32 operations, so results are bit-identical to
 * gc_powersgd_compress) before it adds g.  One pass over the matrices fewer
 * per call.
 *   e:      in: a plain residual (p_prev == NULL) or the previous call's M;
 *           out: this call's M.
 *   q:      in: the previous call's Q (warm start, and the Q of the pending
 *           residual); out: this call's Q.
 *   p_prev: the previous call's (orthonormal) p, or NULL; must not be p (keep
 *           two p buffers and alternate them).
 * gc_powersgd_residual_materialize(e, p, q) turns the pending form into the
 * plain residual (E = M - P Q^T with this call's p and q). */
gc_status gc_powersgd_compress_lazy(const gc_matrix_layout* dev, const gc_matrix_layout* host,
                                    int32_t rank, const float* g, float* e, float* q, float* p,
                                    const float* p_prev, float* p_raw, void* workspace,
                                    size_t ws_bytes, void* stream);
gc_status gc_powersgd_residual_materialize(const gc_matrix_layout* dev,
                                           const gc_matrix_layout* host, int32_t rank, float* e,
                                           const float* p, const float* q, void* workspace,
                                           size_t ws_bytes, void* stream);

/* Receiver of one PowerSGD payload: out += P Q^T per matrix, with the same
 * fp32 accumulation as the residual (call once per worker, in order). */
gc_status gc_powersgd_decompress_accumulate(const gc_matrix_layout* dev,
                                            const gc_matrix_layout* host, int32_t rank,
                                            const float* p, const float* q, float* out,
                                            void* workspace, size_t ws_bytes, void* stream);

/* Size of the scratch array built into libgc for gc_ef_topk_compress_noalloc. */
#define GC_NOALLOC_MAX_WORKSPACE_BYTES (32u << 20)

/* gc_ef_topk_compress without a caller-provided workspace.  The pages have
 * no counterpart: this is a library convenience.  It serves callers that
 * cannot allocate device memory at the point where they compress (their
 * memory manager owns the GPU's memory, or a cudaMalloc there would stall the
 * device).  Inputs, outputs and results are those of gc_ef_topk_compress; the
 * scratch is one array of GC_NOALLOC_MAX_WORKSPACE_BYTES inside the library,
 * held on every GPU that loads it until the process exits.
 *  - Layouts whose gc_workspace_size(GC_OP_TOPK, flags) exceeds that size are
 *    rejected with GC_ERR_WORKSPACE before anything is enqueued.
 *  - The first call on a device looks up the array's device address (once
 *    per device, with that device current); make that first call before any
 *    stream capture on the device.
 *  - All calls share the array: calls that overlap on the GPU (other streams,
 *    other threads) race on it and must be serialized by the caller.
 *  - It allocates and frees nothing. */
gc_status gc_ef_topk_compress_noalloc(const gc_layout* dev, const gc_layout* host, const float* g,
                                      float* e, int32_t* idx, float* val, int8_t* q, float* scale,
                                      uint64_t seed, uint64_t iter, uint32_t flags, void* stream);

/* Diagnostics of the last gc_ef_topk_compress_noalloc call on the current
 * device: waits for `stream`, then reads the diagnostic words at the head of
 * the built-in scratch (what gc_get_device_status reads from a caller's
 * workspace).  It reports, for instance, GC_DIAG_LAYOUT_MISMATCH when that
 * call's device and host layouts disagreed (its kernels then did nothing),
 * and the exact_tensors / overflow_tensors counts.  A later noalloc call on
 * any stream of the device overwrites them.  Returns GC_ERR_DEVICE if an error
 * bit is set; allocates nothing. */
gc_status gc_ef_topk_compress_noalloc_status(void* stream, gc_diag* out);

/* Quantizers of the kept values, for the *_quantized entry points. */
#define GC_KEPT_INT8 1 /* as GC_INT8: scale = max|kept| / 127, code = sgn * min(127, SR(|x| / scale)) */
#define GC_KEPT_QSGD 2 /* scale = N = ||kept||_2, code = sgn * min(s, SR((|x| * s) / N)) */
#define GC_KEPT_SIGN 3 /* scale = mu = mean |kept|, one bit per kept value (1 = sign bit clear) */

/* EF Top-k, then a quantizer applied to the kept values (zh glossary
 * "Gradient Compression": the Top-k + 8-bit pipeline, quantization after
 * sparsification; mbrenndoerfer.com "Gradient Compression": QSGD equation
 * Q_s(g) = ||g|| sgn(g) xi(g, s), 1-bit SGD equation sign(g) ||g||_1 / d with
 * one scalar).  The quantized vector of tensor t is its k_t kept values x_j
 * in ascending index order:
 *   GC_KEPT_QSGD: scale[t] = N = (float)sqrt(sum_j x_j^2), the sum in fp64 in
 *     a fixed order (within 1e-6 relative of any order); q[koff[t] + j] =
 *     sgn(x_j) * min(s, SR((|x_j| * s) / N)), stochastic rounding with the
 *     Philox word of purpose 2 at the element's arena index; decoded value
 *     sgn * ((|q| * N) / s).  N = 0 gives codes 0.
 *   GC_KEPT_SIGN: scale[t] = mu = (float)(sum_j |x_j| / k_t) (fp64 sum);
 *     bit j of tensor t's words is 1 iff x_j has a clear sign bit; tensor t's
 *     bits start at word sum_{t' < t} ceil(k_t' / 32), LSB first, pad bits 0;
 *     decoded value bit ? mu : -mu.
 *   GC_KEPT_INT8: gc_ef_topk_compress with GC_INT8.
 *   residual (GC_EF): e = acc off S, acc - decoded value on S.
 *   k_t = 0 gives scale[t] = 0.
 * idx: device int32[sum k].  val: device fp32[sum k] or NULL: the decoded
 * values.  q: device int8[sum k] (QSGD, INT8; else may be NULL).  bits:
 * device uint32[sum ceil(k_t/32)] (SIGN; else may be NULL), fully written.
 * scale: device fp32[T].  s_levels: 1..127 (QSGD).  flags: GC_EF,
 * GC_FORCE_EXACT.  Workspace: gc_workspace_size(GC_OP_TOPK). */
gc_status gc_ef_topk_compress_quantized(const gc_layout* dev, const gc_layout* host, const float* g,
                                        float* e, int32_t* idx, float* val, int8_t* q,
                                        uint32_t* bits, float* scale, int32_t kind,
                                        int32_t s_levels, uint64_t seed, uint64_t iter,
                                        uint32_t flags, void* workspace, size_t ws_bytes,
                                        void* stream);

/* gc_ef_topk_compress_momentum followed by the kept-value quantizer of
 * gc_ef_topk_compress_quantized, applied to the kept velocity v[S]; v[S]
 * keeps v - decoded value, u[S] = +0 unless GC_NO_MASK.  flags: GC_NO_MASK,
 * GC_FORCE_EXACT.  Workspace: gc_workspace_size(GC_OP_MOMENTUM). */
gc_status gc_ef_topk_compress_momentum_quantized(const gc_layout* dev, const gc_layout* host,
                                                 const float* g, float* u, float* v, float beta,
                                                 int32_t* idx, float* val, int8_t* q,
                                                 uint32_t* bits, float* scale, int32_t kind,
                                                 int32_t s_levels, uint64_t seed, uint64_t iter,
                                                 uint32_t flags, void* workspace, size_t ws_bytes,
                                                 void* stream);

/* DGC momentum correction + Top-k (inferensys.com "Gradient Sparsification",
 * momentum correction and momentum factor masking; genomic glossary, DGC):
 *   u = beta * u + g;  v = v + u;  S = Top-k of |v|;  payload v[S] (or int8);
 *   v[S] = +0 (int8: v - q * scale);  u[S] = +0 unless GC_NO_MASK.
 * u, v: device fp32[N] in/out.  Other arguments as gc_ef_topk_compress
 * (GC_EF, GC_RANDK, GC_UNBIASED are not accepted here). */
gc_status gc_ef_topk_compress_momentum(const gc_layout* dev, const gc_layout* host, const float* g,
                                       float* u, float* v, float beta, int32_t* idx, float* val,
                                       int8_t* q, float* scale, uint64_t seed, uint64_t iter,
                                       uint32_t flags, void* workspace, size_t ws_bytes,
                                       void* stream);

/* 1-bit sign compression with EF (mbrenndoerfer.com "Gradient Compression",
 * 1-bit SGD equation, per-layer scalar):
 *   acc = g + e (e may be NULL: no EF);  mean_abs[t] = (float)(sum|acc_t| / n_t);
 *   bit = 1 iff acc has a clear sign bit;  e = acc - (bit ? mean_abs : -mean_abs).
 * bits: device uint32[sum ceil(n_t/32)].  mean_abs: device fp32[T].  The
 * sum is reduced in a fixed order (relative error below 1e-6). */
gc_status gc_sign_compress(const gc_layout* dev, const gc_layout* host, const float* g, float* e,
                           uint32_t* bits, float* mean_abs, void* workspace, size_t ws_bytes,
                           void* stream);

/* Single-pass sign compression with the residual kept pending.  The bits
 * and mean_abs are those of gc_sign_compress with EF; e is left holding acc,
 * and the residual e = acc - (bit ? mean_abs : -mean_abs) is applied by the
 * next call (pass this call's mean_abs as its prev_mean_abs) in registers
 * before g is added, or by gc_sign_residual_materialize.  One pass over g
 * and e instead of two.
 *   e: device fp32[N]: on entry a plain residual (prev_mean_abs == NULL) or
 *      the previous call's acc; on exit this call's acc.
 *   prev_mean_abs: device fp32[T] of the previous call, or NULL. */
gc_status gc_sign_compress_lazy(const gc_layout* dev, const gc_layout* host, const float* g,
                                float* e, const float* prev_mean_abs, uint32_t* bits,
                                float* mean_abs, void* workspace, size_t ws_bytes, void* stream);

/* e <- e - (signbit(e) ? -mean_abs[t] : mean_abs[t]): turns the pending form
 * left by gc_sign_compress_lazy into the plain EF residual. */
gc_status gc_sign_residual_materialize(const gc_layout* dev, const gc_layout* host, float* e,
                                       const float* mean_abs, void* stream);

/* Dense stochastic quantization (genomic glossary: 8-bit quantization,
 * stochastic rounding, QSGD; mbrenndoerfer.com QSGD equation):
 *   mode GC_Q_INT8: scale[t] = max|acc_t| / 127, code = sgn * min(127, SR(|acc| / scale))
 *   mode GC_Q_QSGD: scale[t] = (float)||acc_t||_2, code = sgn * min(s, SR((|acc| * s) / N)),
 *                   decoded value sgn * ((|code| * N) / s);  1 <= s_levels <= 127.
 *   acc = g + e with EF (e != NULL), and then e = acc - decoded value.
 * codes: device int8[N].  scale: device fp32[T]. */
gc_status gc_quantize_stochastic(const gc_layout* dev, const gc_layout* host, const float* g,
                                 float* e, int8_t* codes, float* scale, int32_t mode,
                                 int32_t s_levels, uint64_t seed, uint64_t iter, void* workspace,
                                 size_t ws_bytes, void* stream);
gc_status gc_quantize_stochastic_dev_iter(const gc_layout* dev, const gc_layout* host, const float* g,
                                          float* e, int8_t* codes, float* scale, int32_t mode,
                                          int32_t s_levels, uint64_t seed, uint64_t* iter_dev,
                                          void* workspace, size_t ws_bytes, void* stream);

/* Receiver of W workers' sparse payloads (mbrenndoerfer.com: the union of
 * different sparse vectors; zh glossary: all-gather of indices and values):
 *   for w = 0..W-1 in order: out[off[t] + idx_w[j]] += value_w[j],
 *   value = val_w[j], or q_w[j] * scale_w[t] when val is NULL.
 * Each element's contributions are added in worker order (fp32, one rounding
 * each), so the result equals that sequential loop bit for bit.
 * idx, val, q, scale: HOST arrays of W device pointers (val NULL, or q and
 * scale NULL).  Each worker's indices of a tensor must be strictly
 * ascending, as every compressor of this library emits them.  An index
 * outside [0, n_t) is skipped and flagged (GC_DIAG_INDEX_RANGE); indices out
 * of order are flagged (GC_DIAG_INDEX_ORDER), and an entry of that worker
 * may then be skipped, so the sum is defined only for ascending payloads.
 * out: device fp32[N], caller-initialised, accumulated into; it must not
 * alias a payload.  Workspace: gc_workspace_size(GC_OP_DECOMPRESS) with the
 * layout's k and koff. */
gc_status gc_sparse_decompress_accumulate(const gc_layout* dev, const gc_layout* host, int32_t W,
                                          const int32_t* const* idx, const float* const* val,
                                          const int8_t* const* q, const float* const* scale,
                                          float* out, void* workspace, size_t ws_bytes,
                                          void* stream);

/* Receiver of W workers' payloads of gc_ef_topk_compress_quantized (or its
 * momentum form), as gc_sparse_decompress_accumulate with the value of entry
 * j of tensor t decoded as the sender's decoded value:
 *   GC_KEPT_INT8: q_w[j] * scale_w[t]
 *   GC_KEPT_QSGD: sgn(q) * ((|q| * scale_w[t]) / s_levels)  (+0 for q = 0)
 *   GC_KEPT_SIGN: bit (j - koff[t]) of tensor t's words of bits_w ? scale_w[t]
 *                 : -scale_w[t]  (words as in gc_ef_topk_compress_quantized)
 * idx, q, bits, scale: HOST arrays of W device pointers (q for INT8 / QSGD,
 * bits for SIGN; the other may be NULL). */
gc_status gc_sparse_decompress_accumulate_quantized(const gc_layout* dev, const gc_layout* host,
                                                    int32_t W, int32_t kind, int32_t s_levels,
                                                    const int32_t* const* idx,
                                                    const int8_t* const* q,
                                                    const uint32_t* const* bits,
                                                    const float* const* scale, float* out,
                                                    void* workspace, size_t ws_bytes, void* stream);

/* Receiver of W workers' dense payloads, out += decode(payload_w) in order
 * w = 0..W-1.  kind GC_DENSE_SIGN: data = uint32 bits (word layout above),
 * decode = bit ? scale[t] : -scale[t].  GC_DENSE_INT8: data = int8 codes,
 * decode = code * scale[t].  GC_DENSE_QSGD: decode = sgn * ((|code| * N) / s).
 * data, scale: HOST arrays of W device pointers. */
gc_status gc_dense_decompress_accumulate(const gc_layout* dev, const gc_layout* host, int32_t W,
                                         int32_t kind, int32_t s_levels, const void* const* data,
                                         const float* const* scale, float* out, void* workspace,
                                         size_t ws_bytes, void* stream);

/* Waits for `stream`, then reads the diagnostics that the last call using
 * `workspace` left there.  Returns GC_ERR_DEVICE if an error bit is set. */
gc_status gc_get_device_status(const void* workspace, size_t ws_bytes, void* stream, gc_diag* out);

/* Static description of a status code. */
const char* gc_status_string(gc_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t gc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GC_H_ */
