/*
 * lora_sgmv.h -- C ABI of the GB300 (sm_103a) multi-adapter LoRA delta library.
 *
 * The operation.  A batch of T tokens mixes tokens of N LoRA adapters that are
 * all resident in GPU memory; every token is served by its own adapter in one
 * pass over the batch (C-LoRA report, vivodigitale.it, "Come funziona
 * l'architettura": mixed-adapter decode batches, per-adapter work fused into one
 * launch per decode step).  Training packs many adapters of different rank on
 * one frozen base and runs their forward and backward together over the
 * concatenated LoRA tensors, tiled along the token or hidden dimension rather
 * than the small rank dimension, in four forward/backward cases (PLoRA
 * technical summary, gist.science, "2. LoRA Execution Engine", Kernelontwerp).
 * For token t routed to adapter i (rank r_i, scale s_i = alpha_i / r_i):
 *     shrink   h_t   = A_i x_t                      A_i: r_i x d_in
 *     expand   y_t  += s_i B_i h_t                  B_i: d_out x r_i
 *     dh       dh_t  = s_i B_i^T dy_t
 *     dB       dB_i  = s_i sum_{t in i} dy_t h_t^T
 *     dA       dA_i  = sum_{t in i} dh_t x_t^T
 *     dX       dx_t += A_i^T dh_t
 * (The pages print no formula; these are the standard LoRA algebra of the
 * method they describe.)  All products accumulate in fp32.
 *
 * Conventions shared by every entry point.
 *  - Ownership: the caller allocates and frees every buffer (inputs, outputs,
 *    segment storage, workspace) and every stream and event.  The library
 *    never allocates or frees device memory, creates streams and events only
 *    when asked to (lora_side_streams_create), keeps no mutable state between
 *    calls (the one exception is the fixed
 *    scratch array of lora_packed_bwd_noalloc, described there) and never
 *    synchronises, except lora_query_status.  Every call is stream-ordered on
 *    `stream`; calls on different streams share nothing but what the caller
 *    passes them.
 *  - Pointers marked "device" must be device (or managed) memory, 16-byte
 *    aligned.  bf16 tensors are passed as raw 16-bit words (IEEE bfloat16).
 *  - Errors found on the host (NULL pointer, size out of range, misalignment,
 *    workspace too small) are returned at once and nothing is launched.
 *    Errors found on the device (an adapter id outside [0, N), an
 *    inconsistent adapter table, a bounded wait that gave up) are written to
 *    the device status word of the lora_segments in use; the kernels skip the
 *    offending work and never trap.  Read it with lora_query_status.
 *  - Debug build (liblora_sgmv_debug.so, the same ABI; lora_debug_checks()
 *    returns 1 there): every index the kernels read from the routing
 *    metadata (tile and span entries and counts, perm, the slots derived from
 *    them) is checked before it addresses memory.  An index out of range sets
 *    LORA_ERR_INDEX and records where in status[1]; the access is redirected
 *    to an in-range index, the results are unspecified and nothing traps.
 *    The release build has no such checks (it trusts lora_build_segments).
 *  - Tokens whose id lies outside [0, N) belong to no adapter: their H / dH
 *    rows are not written and their y / dX rows are left unchanged.
 *  - y and dX accumulate (+=) and are rounded once to bf16 (nearest-even)
 *    after the fp32 sum; H, dH, dA and dB are fp32 and are overwritten.
 */
#ifndef LORA_SGMV_H
#define LORA_SGMV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LORA_SGMV_ABI_VERSION 2

/* Exported entry points (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define LORA_API __attribute__((visibility("default")))
#else
#define LORA_API
#endif

/* Largest supported adapter rank; sizes are checked against it. */
#define LORA_MAX_RANK 128
/* Token rows per work tile of the packed kernels. */
#define LORA_TILE_M 128
#define LORA_MAX_PROJECTIONS 8   /* projections of one lora_multi_fwd call */
/* Tokens per span (the work unit of the reductions over tokens, dA and dB). */
#define LORA_SPAN_TOKENS 1024

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef struct CUstream_st *lora_stream_t;

typedef enum lora_status {
    LORA_OK = 0,
    LORA_ERR_INVALID_ARG = 1,          /* NULL where a pointer is required, negative count */
    LORA_ERR_SHAPE = 2,                /* a size outside the supported range */
    LORA_ERR_ALIGNMENT = 3,            /* a pointer not 16-byte aligned */
    LORA_ERR_BAD_ADAPTER_ID = 4,       /* device: a token id outside [0, N) */
    LORA_ERR_WORKSPACE_TOO_SMALL = 5,  /* storage / workspace below the required bytes */
    LORA_ERR_UNSUPPORTED = 6,          /* no kernel for this device or configuration */
    LORA_ERR_TIMEOUT = 7,              /* device: a bounded wait gave up */
    LORA_ERR_BAD_TABLE = 8,            /* device: rank / row offset inconsistent */
    LORA_ERR_BAD_SEGMENTS = 9,         /* device: segment offsets not monotone or not ending at T */
    LORA_ERR_CUDA = 10,                /* a CUDA runtime call failed */
    LORA_ERR_INDEX = 11                /* device, debug build only: an index read from the routing
                                          metadata was out of range (status[1] says where) */
} lora_status_t;

/*
 * The stacked adapter table: N adapters, all resident on the device.
 *   rank[i]      r_i, 1 <= r_i <= r_max <= LORA_MAX_RANK           (device int32 [N])
 *   row_off[i]   sum_{j<i} r_j; row_off[N] = sum_r                   (device int32 [N+1])
 *   scale[i]     s_i = alpha_i / r_i (fp32)                          (device float [N])
 *   A            bf16 [sum_r, d_in] row-major: A_i is rows row_off[i] .. row_off[i]+r_i-1
 *   B            bf16 [sum_r, d_out] row-major: B_i transposed and stacked like A,
 *                i.e. row row_off[i]+k holds column k of B_i (B_i[o, k] = B[row_off[i]+k, o]).
 *                Stored this way every weight operand of every kernel is a plain 2-D
 *                tile of A or B that one TMA tensor map can address.
 * The host fields (n_adapters, d_in, d_out, r_max, sum_r) size the launches;
 * the device arrays must agree with them (checked on the device: a mismatch
 * sets LORA_ERR_BAD_TABLE and the adapter is skipped).
 * d_in and d_out are multiples of 8 in [8, 1 << 20].
 */
typedef struct lora_adapter_table {
    int32_t n_adapters;
    int32_t d_in;
    int32_t d_out;
    int32_t r_max;
    int32_t sum_r;
    int32_t reserved;
    const int32_t *rank;
    const int32_t *row_off;
    const float *scale;
    const void *A;
    const void *B;
} lora_adapter_table;

/*
 * Routing metadata of one batch (built once, shared by every LoRA layer of a
 * step).  All pointers are device memory carved out of the caller's storage
 * by lora_build_segments; the struct itself is a plain host value.
 *   perm[T]          token indices grouped by adapter, ascending adapter id,
 *                    original order inside a group (stable); only the first
 *                    seg_start[N] entries are valid (tokens with a bad id are left out)
 *   seg_start[N+1]   start of adapter i's group in perm
 *   tiles[4*max_tiles]  work tiles {adapter, begin (index into perm), rows (1..LORA_TILE_M),
 *                    flags (bit 0: the rows are consecutive token indices)}, ordered by
 *                    adapter then begin; n_tiles[0] of them are valid
 *   spans[4*max_spans]  the same cut at LORA_SPAN_TOKENS tokens; n_spans[0] valid
 *   status[0]        device status word (an lora_status_t, LORA_OK when clean)
 *   status[1]        debug build only: where the first failed index check sits
 *                    (source file number << 16 | line; see lora_query_index_check), else 0
 */
typedef struct lora_segments {
    int32_t n_tokens;
    int32_t n_adapters;
    int32_t max_tiles;
    int32_t sorted;
    int32_t *perm;
    int32_t *seg_start;
    int32_t *tiles;
    int32_t *n_tiles;
    int32_t *status;
    int32_t *scratch;      /* builder-internal counters (histogram / scan) */
    int64_t scratch_words;
    int32_t max_spans;
    int32_t reserved;
    int32_t *spans;
    int32_t *n_spans;
} lora_segments;

/* ABI version of the loaded library (LORA_SGMV_ABI_VERSION). */
LORA_API int32_t lora_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
LORA_API const char *lora_status_string(lora_status_t status);

/* Bytes of device storage lora_build_segments needs for T tokens and N adapters
 * (0 when the sizes are out of range). */
LORA_API size_t lora_segments_bytes(int32_t n_tokens, int32_t n_adapters);

/*
 * Segment-metadata builder: group the batch's tokens by adapter (stable) and
 * cut every group into work tiles of at most LORA_TILE_M rows.
 *   ids          device int32 [T]: adapter of every token, any order; or NULL
 *   seg_offsets  device int32 [N+1]: tokens already grouped, adapter i owning
 *                tokens seg_offsets[i] .. seg_offsets[i+1]-1; or NULL
 *                (exactly one of ids / seg_offsets is given)
 *   n_tokens     T >= 0;  n_adapters  N in [1, 65536]
 *   storage      device, >= lora_segments_bytes(T, N) bytes, 16-byte aligned;
 *                it must stay allocated while `out` is in use
 *   out          host struct filled with pointers into storage
 * Resets the status word.  Ids outside [0, N) set LORA_ERR_BAD_ADAPTER_ID and
 * the tokens are left out; non-monotone offsets set LORA_ERR_BAD_SEGMENTS.
 */
LORA_API lora_status_t lora_build_segments(const int32_t *ids, const int32_t *seg_offsets,
                                  int32_t n_tokens, int32_t n_adapters,
                                  void *storage, size_t storage_bytes,
                                  lora_segments *out, lora_stream_t stream);

/* Bytes of device workspace lora_packed_fwd / lora_packed_bwd need for this
 * table and T tokens (0 when the sizes are out of range).  The workspace holds
 * the hand-off rows between the kernels, the counters from which the
 * persistent kernels claim their work items at run time (each zeroed inside
 * the call by the kernel that runs before its user), and for the backward the
 * ordered mode's tickets and case i's partial sums.  Nothing in it has to
 * start at zero; calls that overlap on the GPU need separate workspaces. */
LORA_API size_t lora_workspace_bytes(const lora_adapter_table *table, int32_t n_tokens);

/*
 * SGMV shrink (case i): H[t, 0:r_i] = A_i x_t, H[t, r_i:r_max] = 0.
 *   H  device fp32 [T, r_max] (out);  x  device bf16 [T, d_in] (in)
 * Rows of tokens with a bad id are not written.
 */
LORA_API lora_status_t lora_sgmv_shrink(float *H, const void *x, const lora_adapter_table *table,
                               const lora_segments *segs, lora_stream_t stream);

/*
 * SGMV expand (case ii): y[t, :] += s_i B_i H[t, 0:r_i].
 *   y  device bf16 [T, d_out] (in/out);  H  device fp32 [T, r_max] (in)
 */
LORA_API lora_status_t lora_sgmv_expand(void *y, const float *H, const lora_adapter_table *table,
                               const lora_segments *segs, lora_stream_t stream);

/*
 * Packed forward = shrink then expand over all adapters of the batch.
 *   y       device bf16 [T, d_out] (in/out, +=)
 *   H_save  device fp32 [T, r_max] (out) to keep H for the backward, or NULL
 *   x       device bf16 [T, d_in]
 *   ws      device workspace of >= lora_workspace_bytes(table, T) bytes (may be
 *           NULL when that is 0); it carries H from the shrink to the expand:
 *           as bf16 hi + lo (~16 significant bits), or, for batches of at most
 *           512 tokens, as fp32 partial sums over slices of d_in that the
 *           expand adds in a fixed order; contents need not be preserved after
 *           the call
 */
LORA_API lora_status_t lora_packed_fwd(void *y, float *H_save, const void *x,
                              const lora_adapter_table *table, const lora_segments *segs,
                              void *ws, size_t ws_bytes, lora_stream_t stream);

/*
 * Packed backward, the four cases: dh (case i), dX (case ii), dB (case iii),
 * dA (case iv).
 *   dX       device bf16 [T, d_in] (in/out, +=), or NULL to skip
 *   dA       device fp32 [sum_r, d_in] (out, overwritten; adapters with no
 *            token get zeros), or NULL to skip
 *   dB       device fp32 [sum_r, d_out], B's layout (row row_off[i]+k = column k of
 *            dB_i; out, overwritten), or NULL
 *   dY       device bf16 [T, d_out];  X  device bf16 [T, d_in] (the forward input)
 *   H_saved  device fp32 [T, r_max] from lora_packed_fwd, or NULL to recompute it
 *   ws       device workspace of >= lora_workspace_bytes(table, T) bytes; it carries
 *            bf16 copies of H and dH between the four cases (the dB, dA and dX
 *            products consume bf16 H / dH with fp32 accumulation)
 * Reproducibility: dX (and the forward's y and H) come out bit-identical from
 * run to run.  dA and dB are summed over spans of up to LORA_SPAN_TOKENS
 * tokens, each span's fp32 partial added into the zeroed output as it
 * finishes: for an adapter with at most two spans the result is still
 * bit-identical (two additions to zero commute exactly); with more, the
 * span partials may be added in a different order from run to run, so the
 * last bits of dA / dB can differ (every order is within the same rounding
 * of the exact sum).  lora_packed_bwd_ex with LORA_BWD_DETERMINISTIC fixes
 * the order.
 */
LORA_API lora_status_t lora_packed_bwd(void *dX, float *dA, float *dB, const void *dY, const void *X,
                              const float *H_saved, const lora_adapter_table *table,
                              const lora_segments *segs, void *ws, size_t ws_bytes,
                              lora_stream_t stream);

/*
 * lora_packed_bwd with its independent products side by side on two streams
 * the caller owns.  dB needs only dY and H, so it (with the bf16 copy of a
 * saved H) runs on side->stream[0] beside case i (dh) on `stream`; dA needs dh
 * and runs on side->stream[1] beside case ii (dX) on `stream`.  The tails of
 * one kernel's last wave then overlap the next kernel, which a single stream
 * cannot do.  Results are those of lora_packed_bwd, bit for bit.
 *   side  host struct: two distinct streams on the current device, neither of
 *         them `stream`, and four distinct events (cudaEvent_t, timing may be
 *         disabled), owned by the caller: made by lora_side_streams_create (or
 *         by the caller's own runtime calls) and released with
 *         lora_side_streams_destroy.  The call records
 *         the events and makes the streams wait on them (fork after the zeroing
 *         of dA / dB, join before it returns: on return, `stream` is ordered
 *         after everything the call enqueued on the side streams, also when a
 *         launch failed).  Work the caller enqueues on the side streams after
 *         the call is not ordered with it.  The streams and events may be
 *         reused by the next call; two calls in flight at once (from different
 *         host threads) must use different side streams and events.  Under
 *         stream capture of `stream` the side streams join the capture through
 *         the fork and leave it at the join.
 * Errors: those of lora_packed_bwd; LORA_ERR_INVALID_ARG when side is NULL,
 * a stream or event is NULL, the side streams coincide with each other or
 * with `stream`, or two events coincide.
 */
typedef struct lora_side_streams {
    lora_stream_t stream[2];
    void *event[4];
} lora_side_streams;

/* Create a lora_side_streams set on the current device: two new non-blocking
 * streams and four events with timing disabled, owned by the caller (these
 * two calls are the only ones that create or destroy CUDA objects).  On error
 * nothing is left allocated and *side is zeroed.  Errors: LORA_ERR_INVALID_ARG
 * (NULL), LORA_ERR_CUDA. */
LORA_API lora_status_t lora_side_streams_create(lora_side_streams *side);
/* Destroy a set made by lora_side_streams_create (NULL members are skipped;
 * work still queued on the streams completes first, as cudaStreamDestroy
 * guarantees) and zero *side. */
LORA_API lora_status_t lora_side_streams_destroy(lora_side_streams *side);

LORA_API lora_status_t lora_packed_bwd_concurrent(void *dX, float *dA, float *dB, const void *dY, const void *X,
                                                  const float *H_saved, const lora_adapter_table *table,
                                                  const lora_segments *segs, void *ws, size_t ws_bytes,
                                                  const lora_side_streams *side, lora_stream_t stream);

/*
 * The packed backward with options: lora_packed_bwd when side is NULL and
 * flags is 0, lora_packed_bwd_concurrent when side is given.
 *   side   NULL, or the caller's side streams and events (see
 *          lora_packed_bwd_concurrent)
 *   flags  0 or LORA_BWD_DETERMINISTIC: dA and dB come out bit-identical from
 *          run to run for every adapter.  The partial sum of each span of
 *          LORA_SPAN_TOKENS tokens is added into the output in span order (for
 *          adapters of more than two spans, a span's adds wait, within the
 *          launch and for a bounded time, until the previous span's adds are
 *          complete; a wait that gives up sets LORA_ERR_TIMEOUT on the device).
 *          Uses ticket counters at the end of the workspace, which
 *          lora_workspace_bytes includes, zeroed by the call.  The pages give no
 *          summation order; this mode fixes one.
 * Errors: those of lora_packed_bwd / lora_packed_bwd_concurrent;
 * LORA_ERR_INVALID_ARG for unknown flag bits.
 */
#define LORA_BWD_DETERMINISTIC 1u
LORA_API lora_status_t lora_packed_bwd_ex(void *dX, float *dA, float *dB, const void *dY, const void *X,
                                          const float *H_saved, const lora_adapter_table *table,
                                          const lora_segments *segs, void *ws, size_t ws_bytes,
                                          const lora_side_streams *side, uint32_t flags, lora_stream_t stream);

/*
 * Measurement variants of lora_packed_fwd / lora_packed_bwd: the same checks,
 * kernels and results, and in addition CUDA events are recorded on `stream`
 * around each kernel launch: events[2k] before and events[2k + 1] after the
 * k-th kernel, while 2k + 1 < n_events.  The pages have no counterpart; these
 * exist so a caller can time each kernel of the path on its own stream.
 *   events      n_events cudaEvent_t handles (as void *) created by the
 *               caller, or NULL when n_events is 0; they are only recorded
 *   n_recorded  out, may be NULL: events recorded (2 x kernels launched)
 * Kernel order.  Forward: case i (shrink), case ii (expand); a batch of at
 * most 512 tokens gets one pair around its two decode launches.  Backward:
 * [case i shrink, when H_saved is NULL], [the bf16 copy of H_saved, when
 * given and dB is requested], case iii (dB, if requested), case i (dh), case
 * iv (dA, if requested), case ii (dX, if requested).  The
 * zeroing of dA / dB precedes the first pair.  Like lora_packed_bwd, the
 * marked backward runs all of its kernels one after another on `stream`, so
 * that each pair brackets one kernel alone.
 * Errors: those of the unmarked call; LORA_ERR_INVALID_ARG when n_events < 0
 * or events is NULL with n_events > 0.
 */
LORA_API lora_status_t lora_packed_fwd_marked(void *y, float *H_save, const void *x,
                                              const lora_adapter_table *table, const lora_segments *segs,
                                              void *ws, size_t ws_bytes, lora_stream_t stream,
                                              void *const *events, int32_t n_events, int32_t *n_recorded);
LORA_API lora_status_t lora_packed_bwd_marked(void *dX, float *dA, float *dB, const void *dY, const void *X,
                                              const float *H_saved, const lora_adapter_table *table,
                                              const lora_segments *segs, void *ws, size_t ws_bytes,
                                              lora_stream_t stream, void *const *events, int32_t n_events,
                                              int32_t *n_recorded);

/*
 * One optimizer step for every adapter of the table, fused with the refresh
 * of the bf16 weights the forward reads.  Each tenant keeps FP32 master
 * weights, optimizer moments and gradient buffers beside its LoRA parameters
 * (C-LoRA report, "Come funziona l'architettura": the AdapterStore); the
 * pages name no optimizer, and the step is AdamW, adapter i with its own
 * learning rate lr[i] and step number t = step[i] (>= 1, the caller advances
 * it):
 *   w <- w - lr wd w;  m <- b1 m + (1 - b1) g;  v <- b2 v + (1 - b2) g^2
 *   w <- w - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
 * and the table's bf16 A / B rows are overwritten with round-to-nearest-even(w).
 *   wA, mA, vA  device fp32 [sum_r, d_in]   master A and its moments (in/out;
 *               the moments start at zero)
 *   wB, mB, vB  device fp32 [sum_r, d_out]  master B^T (stored like the table's
 *               B) and its moments (in/out)
 *   gA, gB      device fp32 gradients in the same layouts (dA, dB of
 *               lora_packed_bwd)
 *   lr          device fp32 [n_adapters]; step  device int32 [n_adapters]
 *   beta1, beta2 in [0, 1), eps >= 0, weight_decay >= 0
 * Writes the table's A and B (its bf16 weights).  Errors: LORA_ERR_INVALID_ARG
 * (null pointer, hyper-parameter out of range), LORA_ERR_ALIGNMENT (fp32
 * arrays need 16-byte, lr / step 4-byte alignment), the table checks of the
 * other calls.  The pages have no optimizer kernel of their own.
 */
LORA_API lora_status_t lora_adamw_step(const lora_adapter_table *table, float *wA, float *wB, const float *gA,
                                       const float *gB, float *mA, float *vA, float *mB, float *vB, const float *lr,
                                       const int32_t *step, float beta1, float beta2, float eps, float weight_decay,
                                       lora_stream_t stream);

/*
 * Packed forward of several projections that read the same input x (a layer's
 * q / k / v, or its gate / up), each with its own adapter table:
 *   for p < n_proj:  H_p[t] = A_{p,i} x_t,  y_p[t] += s_{p,i} B_{p,i} H_p[t]
 * Decode steps are launch-latency-sized, and the C-LoRA report's decode
 * kernel serves every adapter of the batch in one launch per step ("Come
 * funziona l'architettura"); here a batch of at most 512 tokens runs all the
 * projections in the same two launches (the shrink, then the expand as a
 * programmatic dependent), blockIdx.y selecting the projection.  Larger
 * batches run lora_packed_fwd's kernels projection after projection.
 *   n_proj    1 .. LORA_MAX_PROJECTIONS
 *   y         host array of n_proj device pointers, bf16 [T, d_out_p] (in/out, +=)
 *   H_save    host array of n_proj device pointers fp32 [T, r_max_p] (out;
 *             NULL entries skip), or NULL for none
 *   x         device bf16 [T, d_in], shared by every projection
 *   tables    host array of n_proj tables; all with the same d_in and
 *             n_adapters (= segs->n_adapters); ranks, scales, B, d_out free
 *   ws        device workspace of >= lora_multi_workspace_bytes(n_proj, tables, T)
 * Results per projection are those of lora_packed_fwd on that projection.
 * Errors: those of lora_packed_fwd; LORA_ERR_SHAPE when n_proj is out of range
 * or the tables disagree on d_in or n_adapters.
 */
LORA_API size_t lora_multi_workspace_bytes(int32_t n_proj, const lora_adapter_table *tables, int32_t n_tokens);
LORA_API lora_status_t lora_multi_fwd(int32_t n_proj, void *const *y, float *const *H_save, const void *x,
                                      const lora_adapter_table *tables, const lora_segments *segs, void *ws,
                                      size_t ws_bytes, lora_stream_t stream);

/*
 * A LoRA layer's forward in one persistent launch: the base projection with
 * the packed delta on the same fp32 accumulators,
 *   y_t = W x_t + s_i B_i (A_i x_t)          (token t of adapter i)
 * The frozen base weight W is shared by every adapter of the batch, which is
 * what packing amortises (PLoRA technical summary, "2. LoRA Execution
 * Engine": base-model computation shared across the packed adapters).
 *   y       device bf16 [T, d_out] (out, overwritten; rounded once from fp32)
 *   H_save  device fp32 [T, r_max] (out): h = A_i x_t, zero beyond r_i, for
 *           lora_packed_bwd; or NULL
 *   x       device bf16 [T, d_in];  W  device bf16 [d_out, d_in] row-major
 *           (a linear layer's weight)
 *   segs    built from seg_offsets (tokens grouped by adapter, the packed
 *           layout); a batch routed from unsorted ids gives LORA_ERR_UNSUPPORTED
 *   ws      device workspace of >= lora_fused_base_workspace_bytes(table, T)
 *           bytes: the bf16 s_i h hand-off rows and one ready counter per tile
 * The delta's h enters the expand as bf16 (s_i h rounded once); products
 * accumulate in fp32.  The kernel is a cooperative launch (one CTA per SM,
 * all resident).  Errors: those of lora_packed_fwd; LORA_ERR_TIMEOUT on the
 * device if a wait between CTAs gives up (it is bounded).
 */
LORA_API size_t lora_fused_base_workspace_bytes(const lora_adapter_table *table, int32_t n_tokens);
LORA_API lora_status_t lora_fused_base_fwd(void *y, float *H_save, const void *x, const void *W,
                                           const lora_adapter_table *table, const lora_segments *segs,
                                           void *ws, size_t ws_bytes, lora_stream_t stream);

/*
 * Packing planner (host only, no GPU work): group LoRA fine-tuning
 * configurations into packed jobs and place the jobs on a pool of GPUs
 * (PLoRA technical summary, "1. LoRA Packing Planner (Offline)": minimise the
 * completion time of a set of configurations on a fixed pool, a 0-1 knapsack
 * variant solved round by round, with a cost model for memory and throughput).
 * Cost model: a job step of the packed set S takes
 *     t(S) = step_overhead_s + sum_{c in S} tokens_per_step_c * w_c,
 *     w_c  = base_s_per_token + lora_s_per_token + lora_s_per_token_rank * rank_c
 * and the job runs max_{c in S} steps_c steps.  Each round makes the next job
 * from the configurations not yet placed: the set whose memory fits one GPU
 * (job_mem_bytes + sum of mem_bytes, counted in whole mem_unit_bytes units,
 * each configuration's size rounded up) and that trains the most tokens per
 * second, sum_c steps_c tokens_per_step_c / (max_c steps_c * t(S)), found
 * exactly (Dinkelbach iterations over 0-1 knapsacks).  A round's job may
 * then be cut into balanced parts where that ends the pool's work sooner: for
 * a cap D on a job's duration every job is cut into the fewest parts that each
 * end within D (configurations dealt, largest step cost first, to the part
 * with the least cost so far); the caps tried are the parts' own durations,
 * plus every job cut into single configurations, and the plan that ends
 * first is kept (the uncut plan on ties, then fewer jobs); then, while it
 * helps, one job at a time is cut into one part more or one fewer (the change
 * that ends the pool soonest, strictly sooner).  Jobs are placed
 * longest first, each on the GPU that frees first (lowest index on ties); a
 * job uses one GPU.  The plan never ends later than the uncut rounds' jobs
 * or than one configuration per job under the same placement.
 *   configs    n_configs entries (host); n_configs in [1, 4096]
 *   job_of     out, host int32 [n_configs]: the job of every configuration
 *              (jobs numbered in the order the rounds made them, the parts
 *              of a cut job one after another)
 *   jobs       out, host array with room for n_configs jobs
 *   n_jobs     out: jobs made;  makespan_s  out: predicted completion time
 * Work grows as n_configs^3 x budget units (per round, per choice of the
 * longest configuration, a knapsack pass per Dinkelbach iteration), plus
 * |S|^3 for cutting a job of |S| configurations: meant for search spaces of a
 * few hundred configurations and budgets of a few thousand units (120
 * configurations, 4200 units: ~0.1-0.3 s).
 * Errors: LORA_ERR_INVALID_ARG (NULL, negative cost terms, a zero-time step),
 * LORA_ERR_SHAPE (a configuration that does not fit one GPU alone, sizes out
 * of range, a memory budget of more than 2^20 units, n_configs x (budget
 * units + 1) above 2^28, host memory exhausted).
 */
typedef struct lora_plan_config {
    int32_t rank;             /* LoRA rank */
    int32_t tokens_per_step;  /* tokens of its batch in every training step */
    int64_t steps;            /* training steps it needs */
    int64_t mem_bytes;        /* device memory it adds to a job (adapter state, optimizer, activations) */
} lora_plan_config;

typedef struct lora_plan_cost {
    double step_overhead_s;        /* fixed time of one job step */
    double base_s_per_token;       /* frozen base model, forward + backward, per token */
    double lora_s_per_token;       /* LoRA path per token, rank-independent part */
    double lora_s_per_token_rank;  /* LoRA path per token and unit of rank */
    int64_t gpu_mem_bytes;         /* memory of one GPU */
    int64_t job_mem_bytes;         /* memory of every job besides its configurations */
    int64_t mem_unit_bytes;        /* granularity of the memory budget */
    int32_t n_gpus;                /* GPUs in the pool */
    int32_t reserved;
} lora_plan_cost;

typedef struct lora_plan_job {
    int32_t gpu;        /* GPU of the pool the job runs on */
    int32_t n_configs;  /* configurations packed into it */
    double start_s;     /* predicted start */
    double duration_s;  /* predicted duration: steps x step time */
    double step_s;      /* predicted time of one step */
} lora_plan_job;

LORA_API lora_status_t lora_plan_pack(const lora_plan_config *configs, int32_t n_configs,
                                      const lora_plan_cost *cost, int32_t *job_of, lora_plan_job *jobs,
                                      int32_t *n_jobs, double *makespan_s);

/*
 * Packed backward without a workspace, for callers that cannot allocate device
 * memory (no cudaMalloc, no allocator of their own to draw scratch from).  The
 * pages have no counterpart to this call; it exists only for such callers.
 * Same arguments and results as lora_packed_bwd minus ws / ws_bytes: the bf16
 * H / dH hand-off scratch lives in a fixed 8 MiB array inside the library's device
 * memory (held by every GPU that loads the library until exit), laid out as
 * lora_packed_bwd lays out its workspace: two bf16 hand-off copies of
 * T * 64 values when r_max <= 64, T * 128 otherwise (each rounded up to 256
 * bytes), then a few counters and, for batches of few tiles, fp32 partial
 * sums of case i; when all of it does not fit in 8 MiB
 * LORA_ERR_WORKSPACE_TOO_SMALL is returned and nothing runs.  Allocates
 * nothing.  All calls share the array: calls that overlap on the GPU race and
 * must be serialised by the caller.  The first call on a device resolves the
 * array's device address (cudaGetSymbolAddress) and caches it; make that first
 * call before capturing a stream.
 */
LORA_API lora_status_t lora_packed_bwd_noalloc(void *dX, float *dA, float *dB, const void *dY, const void *X,
                                               const float *H_saved, const lora_adapter_table *table,
                                               const lora_segments *segs, lora_stream_t stream);

/*
 * Diagnostic: runs the tensor-core kernels' bounded pipeline wait against a
 * barrier that nothing completes (one CTA, two warps) and lets it give up:
 * after about 2 s of SM clock (4e9 cycles) LORA_ERR_TIMEOUT is written to
 * *status (device int32, 4-byte aligned; a nonzero value already there is
 * kept) and the kernel returns.  Shows on a given GPU that a stalled pipeline
 * ends with a status instead of a hang, and that the context stays usable.
 * Stream-ordered; synchronise before reading *status.
 * Errors: LORA_ERR_INVALID_ARG (NULL), LORA_ERR_ALIGNMENT, LORA_ERR_CUDA.
 */
LORA_API lora_status_t lora_check_wait_timeout(int32_t *status, lora_stream_t stream);

/* 1 in the debug build (device-side index checks compiled in), else 0. */
LORA_API int32_t lora_debug_checks(void);

/* Synchronise `stream`, return the device status word of `segs` and store in
 * *where (host int32) status[1]: in the debug build, after LORA_ERR_INDEX,
 * the failed check's source file number << 16 | line (file numbers: 1
 * route.cu, 2 tc_rowproj.cu, 3 tc_colproj.cu, 4 tc_tokred.cu, 5 decode.cu,
 * 6 tc_base.cu, 7 dispatch.cu); else 0.  Errors: LORA_ERR_INVALID_ARG (NULL),
 * LORA_ERR_CUDA. */
LORA_API lora_status_t lora_query_index_check(const lora_segments *segs, lora_stream_t stream, int32_t *where);

/* Synchronise `stream` and return the device status word of `segs`. */
LORA_API lora_status_t lora_query_status(const lora_segments *segs, lora_stream_t stream);

/* Clear the device status word and the debug build's check site (stream-ordered). */
LORA_API lora_status_t lora_reset_status(const lora_segments *segs, lora_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* LORA_SGMV_H */
