/*
 * dvl.h -- C ABI of the GB300 draft-head argmax library (libdvl.so).
 *
 * The operation: a speculative-decoding draft head projects M hidden rows
 * h[M][K] against the rows of its LM head W[N][K] and keeps, per hidden row,
 * the best token -- logits = h . W^T, reduced on the device to an id and its
 * logit, so no logit tensor is ever written to memory.  N is either the full
 * vocabulary or a frequency-ranked shortlist of it, in which case a d2t map
 * turns a shortlist row index into a full-vocabulary id.
 *   - the projection and its shape ("Shortlist MTP", section "What I was
 *     testing": hidden width 2,560 against 248,320 rows; M is 1 for a draft
 *     step and 3 for an MTP2 verify step);
 *   - the shortlist and its on-device reduction ("Shortlist MTP", sections
 *     "What was actually happening" and "Re-running the comparison fairly":
 *     the shortlist projection and local argmax reduction);
 *   - the trim at load and the d2t map ("Masked MTP drafts": a ranks .txt
 *     next to the model, the head weight trimmed at load; EAGLE-3's d2t
 *     index mapping reused for a frequency-ranked subset);
 *   - the NVFP4 head ("Masked MTP drafts": the trimmed head requantized to
 *     NVFP4) and the FP8 head ("Masked MTP drafts", section "Update
 *     (November 2026)": a drafter's own FP8 head; "[DGX Spark]
 *     Qwen3.8-Flash-Next on two DGX Sparks", section "The costs: a 69%
 *     smaller KV pool and FP8 GDN weights": weights read as FP8 E4M3);
 *   - the ranks builder ("Shortlist MTP", section "Building the 16k
 *     shortlist"; "[DGX Spark] Qwen3.8-Flash-Next on two DGX Sparks",
 *     section "Build the draft vocabulary from your own text").
 *
 * Conventions for every entry point:
 *   - Memory: the caller owns every buffer.  "device" pointers are CUDA
 *     device memory on the current device; "host" pointers are ordinary host
 *     memory.  The GPU entry points never allocate, free or synchronize; they
 *     enqueue work on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and return.  Results are ready in stream order.
 *   - Errors: arguments are checked on the host before anything is enqueued;
 *     a bad argument returns a non-zero dvl_status and enqueues nothing.  A
 *     failed launch returns DVL_ERR_CUDA (the outputs are then undefined).
 *   - Threading: calls are thread-safe.  One workspace serves one stream at a
 *     time: two calls that may run concurrently on the GPU must not share a
 *     workspace.
 *   - Alignment: W, h, scales and the workspace start on 16-byte boundaries;
 *     d2t, ids and logits on 4-byte boundaries.
 */
#ifndef DVL_H
#define DVL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DVL_OK = 0,
    DVL_ERR_INVALID_ARG = 1,  /* NULL pointer, bad size, misalignment        */
    DVL_ERR_OUT_OF_RANGE = 2, /* an id outside [0, V) (host-checked ids; as a
                                 device-side bit: a d2t entry outside [0, V)) */
    DVL_ERR_UNSUPPORTED = 3,  /* a shape this build has no kernel for        */
    DVL_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required  */
    DVL_ERR_CUDA = 5,         /* a CUDA runtime call or a launch failed      */
    DVL_ERR_TIMEOUT = 6       /* device-side bit: a bounded wait gave up     */
} dvl_status;

typedef enum {
    DVL_BF16 = 0,  /* W: bfloat16 [N][K] row-major                          */
    DVL_NVFP4 = 1, /* W: E2M1 codes [N][K/2] (low nibble = even k), E4M3
                      scales [N][K/16] (one per 16 consecutive k of a row),
                      one fp32 tensor scale                                  */
    DVL_FP8 = 2    /* W: E4M3 codes [N][K], one fp32 tensor scale; no
                      per-block scales                                       */
} dvl_dtype;

/* Limits of this build. */
#define DVL_MAX_M 32        /* hidden rows per call                            */
#define DVL_MAX_TOPK 4      /* k of draft_topk                                 */
#define DVL_K_MULTIPLE 64   /* K must be a positive multiple of this           */
#define DVL_MAX_K 24576     /* largest hidden width                            */

/* dvl_head.flags: the caller promises that no work still pending on the
 * stream when the call is enqueued writes w, scales or d2t (true of weights
 * loaded long before; not of a head trim_head has just filled on the same
 * stream unless the caller synchronized since).  The kernel may then start
 * streaming the head before the preceding kernel on the stream has finished
 * (programmatic dependent launch); without the flag it reads nothing before
 * that kernel completes. */
#define DVL_HEAD_STATIC 1

/* A draft head as the kernels read it.  Every pointer is device memory. */
typedef struct dvl_head {
    int32_t dtype;        /* dvl_dtype                                         */
    int32_t N;            /* rows of W (>= 1)                                  */
    int32_t K;            /* hidden width (multiple of 64, <= DVL_MAX_K)       */
    int32_t flags;        /* DVL_HEAD_* bits; 0 when none applies              */
    int64_t V;            /* full vocabulary size: ids lie in [0, V)           */
    int64_t id_base;      /* with d2t == NULL, row n has full id id_base + n;
                             id_base + N <= V.  0 for a whole head; the first
                             id of a slice when a head is split by rows.       */
    const void *w;        /* bf16 [N][K], NVFP4 codes [N][K/2] or FP8 [N][K]   */
    const uint8_t *scales;/* NVFP4: E4M3 [N][K/16]; NULL for bf16 and FP8      */
    float global_scale;   /* NVFP4 / FP8 tensor scale; ignored for bf16        */
    int32_t reserved2;    /* must be 0                                         */
    const int32_t *d2t;   /* int32 [N]: full-vocabulary id of each row, each in
                             [0, V); NULL means the identity map shifted by
                             id_base.  The kernels read no memory through a
                             d2t entry; a returned id outside [0, V) is
                             returned as it is and reported as the
                             device-side status bit DVL_ERR_OUT_OF_RANGE (see
                             dvl_workspace_status)                           */
} dvl_head;

/* Human-readable name of a status code (static storage). */
const char *dvl_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int dvl_version(void);

/* The CUDA runtime's description of the error behind the calling thread's
 * most recent DVL_ERR_CUDA ("no error" if there was none).  Static storage. */
const char *dvl_last_error(void);

/* ---------------------------------------------------------------------- */
/* Workspace                                                              */
/* ---------------------------------------------------------------------- */

/* Bytes of device workspace one draft_argmax (k = 1) or draft_topk call
 * with M hidden rows needs.  Returns 0 for M or k outside their limits.
 * The workspace holds the cross-block reduction state: a ticket counter,
 * the per-row best keys and, for k > 1, one candidate list per thread block.
 * It is self-cleaning: every call leaves it as it found it. */
size_t dvl_workspace_bytes(int32_t M, int32_t k);

/* Zero a workspace before its first use (enqueued on `stream`).  Only
 * needed once; also restores a workspace whose last call did not complete.
 * ws: device, 16-byte aligned; bytes >= dvl_workspace_bytes(M, k) of every
 * call that will use it. */
dvl_status dvl_workspace_init(void *ws, size_t bytes, void *stream);

/* Device-side failures recorded in a workspace since it was last read: a
 * bitmask with bit (1 << s) set for each dvl_status s a kernel reported:
 *   DVL_ERR_TIMEOUT       a bounded wait of the tcgen05 kernel gave up; that
 *                         call's results are not valid;
 *   DVL_ERR_OUT_OF_RANGE  a draft call returned an id outside [0, V): a d2t
 *                         entry out of range won, and is returned as it is.
 * The status word is read after the work already enqueued on `stream` (this
 * synchronizes `stream`), then cleared on `stream`.
 *   ws:          a workspace from dvl_workspace_init.
 *   status_bits: HOST (out).
 * Errors: DVL_ERR_INVALID_ARG, DVL_ERR_CUDA. */
dvl_status dvl_workspace_status(void *ws, uint32_t *status_bits, void *stream);

/* ---------------------------------------------------------------------- */
/* The hot path                                                           */
/* ---------------------------------------------------------------------- */

/* Per hidden row m: the full-vocabulary id of the head row with the largest
 * logit sum_k W[n][k] * h[m][k], and that logit.  The dot products run in
 * fp32 on the device (products of bf16 values are exact; the order of the
 * additions is the kernel's).  Exactly equal logits go to the lowest full
 * id; a NaN logit ranks below every number (among NaN logits the lowest id
 * wins, reported with a NaN logit); -0 and +0 compare equal and +0 is
 * reported.  For NVFP4,
 * weight = e2m1(code) * e4m3(scale) * global_scale; for FP8,
 * weight = e4m3(code) * global_scale; the kernel applies global_scale to the
 * finished dot product.
 *   head:      the head (see dvl_head); host struct, device pointers.
 *   h:         device bf16 [M][K], row-major.
 *   M:         1 .. DVL_MAX_M.
 *   ids:       device int32 [M] (out).
 *   max_logit: device fp32 [M] (out).
 *   ws:        device workspace of at least dvl_workspace_bytes(M, 1)
 *              bytes, zeroed once by dvl_workspace_init.
 * Errors: DVL_ERR_INVALID_ARG (NULL, misaligned, N < 1, K not a multiple of
 * 64 or above DVL_MAX_K, M out of range, unknown flags, reserved2 non-zero, dtype
 * unknown, NVFP4 without scales, FP8 with scales, d2t == NULL with
 * id_base + N > V),
 * DVL_ERR_WORKSPACE, DVL_ERR_CUDA. */
dvl_status dvl_draft_argmax(const dvl_head *head, const void *h, int32_t M,
                            int32_t *ids, float *max_logit, void *ws,
                            size_t ws_bytes, void *stream);

/* Per hidden row m: the k best head rows by (logit desc, full id asc), as
 * full ids and logits, best first.  Same arithmetic, rules and errors as
 * dvl_draft_argmax; k = 1 gives exactly its result.  Rows are distinct; a
 * d2t that repeats an id can make an id appear twice.
 *   k:      1 .. DVL_MAX_TOPK, and k <= N.
 *   ids:    device int32 [M][k] (out).
 *   logits: device fp32 [M][k] (out).
 *   ws:     at least dvl_workspace_bytes(M, k) bytes. */
dvl_status dvl_draft_topk(const dvl_head *head, const void *h, int32_t M, int32_t k,
                          int32_t *ids, float *logits, void *ws, size_t ws_bytes,
                          void *stream);

/* Which kernels a dvl_draft_argmax (k = 1) or dvl_draft_topk call with this
 * head, M and k launches, for logs and tests; enqueues nothing.  *kernel is
 * a static string owned by the library:
 *   "bf16-cuda-cores"  CUDA-core kernel (one or two hidden rows, widths
 *                      other than 2,560 / 5,120, short heads);
 *   "bf16-mma"         register-path tensor cores (3 .. 8 hidden rows at
 *                      width 2,560 or 5,120, and argmax at 9 .. 16 rows at
 *                      2,560, on a 32-byte aligned head of at least 8 rows
 *                      per warp of the grid);
 *   "bf16-tcgen05"     5th-generation tensor cores (5 .. 32 hidden rows, when
 *                      the register-path kernel does not apply);
 *   "nvfp4-mma", "fp8-mma"  the low-bit heads.
 * *launches is the number of kernel launches of the call.  The choice
 * depends on the current device's SM count.
 * Errors: those of dvl_draft_topk's head and M / k checks, and
 * DVL_ERR_CUDA when the device cannot be queried. */
dvl_status dvl_draft_plan(const dvl_head *head, int32_t M, int32_t k, const char **kernel,
                          int32_t *launches);

/* dvl_draft_argmax for callers that cannot allocate device memory.  The
 * pages have no counterpart of this entry point.
 *
 * Who needs it: code running as a plugin inside an inference engine that
 * owns every device allocation (raw cudaMalloc is not available to it), and
 * latency-critical decode loops where a cudaMalloc would stall the pipeline
 * (it may synchronize the device).  Such a caller passes the head, h and the
 * outputs only; the reduction scratch lives in a fixed 512-byte array in the
 * library's own device memory (a static __device__ array: every GPU that
 * loads the library keeps it until the process exits).  This entry point
 * allocates nothing and frees nothing.
 *   Same arguments, arithmetic and results as dvl_draft_argmax, without
 *   ws / ws_bytes; the same argument errors.  M above DVL_MAX_M (32), the
 *   most the fixed scratch holds, returns DVL_ERR_INVALID_ARG before
 *   anything is enqueued.
 *   The first call in a CUDA context looks up the array's device address
 *   (cudaGetSymbolAddress, with that context's device current) and keeps it
 *   for that context; make that first call before any stream capture.
 *   Every call clears the scratch's reduction state (ticket and best keys)
 *   with memsets enqueued on `stream`, then runs the argmax on it.  The
 *   scratch's status word is not cleared: device-side failures (the bits of
 *   dvl_workspace_status) accumulate there until dvl_noalloc_status reads
 *   them.  All calls on a device share the one array: two calls that may
 *   run at the same time on the GPU (on different streams, or from
 *   different threads) race on it and may return wrong results.  Keep them
 *   in one stream order. */
dvl_status dvl_draft_argmax_noalloc(const dvl_head *head, const void *h, int32_t M,
                                    int32_t *ids, float *max_logit, void *stream);

/* The device-side failure bits that dvl_draft_argmax_noalloc calls on the
 * current device recorded since the last read (the bits and meaning of
 * dvl_workspace_status), read after the work already enqueued on `stream`
 * (this synchronizes `stream`) and then cleared on `stream`.  No
 * counterpart on the pages; allocates nothing.
 *   status_bits: HOST (out).
 * Errors: DVL_ERR_INVALID_ARG, DVL_ERR_CUDA. */
dvl_status dvl_noalloc_status(uint32_t *status_bits, void *stream);

/* Candidate scores through a head ("Masked MTP drafts", section "Update
 * (November 2026)": a drafter that carries no head of its own scores its
 * candidates through the target's LM head, bf16 or NVFP4, and the trim
 * stacks on top).  For m < M and j < c:
 *   logits[m][j] = sum_k W[ids[m][j] - id_base][k] * h[m][k]
 * with the head's dtype and arithmetic (fp32 accumulation; NVFP4 weights
 * e2m1 * e4m3, FP8 weights e4m3, with the tensor scale on the finished dot),
 * in any summation
 * order.  The head's rows are ids id_base .. id_base + N - 1: a full head
 * (id_base 0) or any contiguous slice of one.  An id outside them scores
 * NaN; the ids live on the device and are not checked on the host.
 *   head:   a head without d2t (d2t == NULL).
 *   h:      device bf16 [M][K], row-major, 16-byte aligned.
 *   M:      1 .. DVL_MAX_M.
 *   ids:    device int32 [M][c], row-major (the candidates of row m).
 *   c:      candidates per row, >= 1, with M * c < 2^31.
 *   logits: device fp32 [M][c] (out), row-major.
 * Nothing is allocated; no workspace.  The call is enqueued on `stream`.
 * Errors: DVL_ERR_INVALID_ARG (the head checks of dvl_draft_argmax, a head
 * with d2t, NULL or misaligned pointers, M or c out of range), DVL_ERR_CUDA. */
dvl_status dvl_score_ids(const dvl_head *head, const void *h, int32_t M,
                         const int32_t *ids, int32_t c, float *logits, void *stream);

/* ---------------------------------------------------------------------- */
/* Load time                                                              */
/* ---------------------------------------------------------------------- */

/* Trim a full head to the rows a ranks list names, in the list's order:
 * W_trim[i] = W_full[ranks[i]] (byte copy of the row, in any dtype; for NVFP4 the codes
 * and the scales), d2t[i] = ranks[i].  The ranks are checked on the host
 * before anything is enqueued; duplicates are accepted (padded lists exist)
 * and counted.
 *   full:      the full head: N == V, d2t == NULL, id_base == 0.
 *   ranks:     HOST int32 [n_ranks], each in [0, V).
 *   n_ranks:   >= 1.
 *   w_trim:    device, rows of the same format: bf16 [n][K] or codes [n][K/2].
 *   scales_trim: device E4M3 [n][K/16] for NVFP4; NULL for bf16.
 *   d2t:       device int32 [n_ranks] (out); the trimmed head's d2t.
 *   n_duplicates: HOST (out, may be NULL): entries that repeat an earlier id.
 * The ranks are copied to d2t with a host-to-device copy from pageable
 * memory, which returns once the source has been read.
 * Errors: DVL_ERR_INVALID_ARG, DVL_ERR_OUT_OF_RANGE (nothing enqueued),
 * DVL_ERR_CUDA. */
dvl_status dvl_trim_head(const dvl_head *full, const int32_t *ranks, int32_t n_ranks,
                         void *w_trim, uint8_t *scales_trim, int32_t *d2t,
                         int32_t *n_duplicates, void *stream);

/* Requantize a bf16 head to NVFP4 or FP8 at load ("Masked MTP drafts": the
 * trimmed head requantized to NVFP4 at no measured acceptance cost; the
 * pages give no recipe).  In fp32, each operation rounded once, in order:
 *   NVFP4: g = amax / (6 * 448); per 16 consecutive weights of a row
 *          s = RNE_e4m3(amax_b / (6 g)), code = RNE_e2m1(w / (s g)), all
 *          codes 0 when s is 0;
 *   FP8:   g = amax / 448; code = RNE_e4m3(w / g);
 * amax is the head's largest |w| (g = 1 for an all-zero head); RNE rounds
 * to the nearest value of the format, ties to even, saturating at its
 * largest finite value; a code's sign is its quotient's.  The weights must
 * be finite.
 *   src:    a bf16 head (only dtype, N, K and w are read).
 *   dtype:  DVL_NVFP4 or DVL_FP8.
 *   codes:  device, 16-byte aligned: NVFP4 [N][K/2] (low nibble = even k) or
 *           FP8 [N][K].
 *   scales: device, 16-byte aligned NVFP4 E4M3 [N][K/16]; NULL for FP8.
 *   global_scale: HOST float (out): g.
 *   ws:     a workspace from dvl_workspace_init (at least
 *           dvl_workspace_bytes(1, 1) bytes); left as it was found.
 * This load-time call synchronizes `stream` once, to read amax back.
 * Errors: DVL_ERR_INVALID_ARG, DVL_ERR_WORKSPACE, DVL_ERR_CUDA. */
dvl_status dvl_quantize_head(const dvl_head *src, int32_t dtype, void *codes, uint8_t *scales,
                             float *global_scale, void *ws, size_t ws_bytes, void *stream);

/* Learn escaped ids into spare rows of a trimmed head while serving ("Masked
 * MTP drafts", section "Update (November 2026)": a static trim can miss;
 * the server learns the escaped ids into spare head rows).  For i < n:
 *   W_trim[row0 + i] = W_full[ids[i]] (the row's bytes; NVFP4 codes and
 *   scales), d2t[row0 + i] = ids[i],
 * the same copy as dvl_trim_head, into rows row0 .. row0 + n - 1.  Allocate
 * the trimmed buffers with room for the rows they may learn; a head of
 * row0 + n rows over the same buffers then includes the learned ids.
 *   full:   the full head: N == V, d2t == NULL, id_base == 0.
 *   ids:    HOST int32 [n], each in [0, V), checked before anything is
 *           enqueued (DVL_ERR_OUT_OF_RANGE).
 *   n:      >= 1.   row0: >= 0, with row0 + n < 2^31.
 *   w_trim, scales_trim (NVFP4; NULL for bf16), d2t: the trimmed head's
 *           device buffers from their row 0 (not offset); the caller owns
 *           them and sizes them for rows up to row0 + n (not checkable here).
 * Ordering: rows and d2t entries are written by kernels on `stream`; later
 * calls on that stream see them.  The first reducing call after the learn
 * on that stream must not set DVL_HEAD_STATIC on the trimmed head (the flag
 * lets a kernel read the head before the preceding kernel has finished);
 * later calls may set it again.  The ids are copied from pageable memory;
 * the call returns once they have been read.
 * Errors: DVL_ERR_INVALID_ARG, DVL_ERR_OUT_OF_RANGE (nothing enqueued),
 * DVL_ERR_CUDA. */
dvl_status dvl_learn_rows(const dvl_head *full, const int32_t *ids, int32_t n, int32_t row0,
                          void *w_trim, uint8_t *scales_trim, int32_t *d2t, void *stream);

/* The whole repair step of a shortlist that learns while serving ("Masked
 * MTP drafts", section "Update (November 2026)": the ids a static trim
 * missed, learned into spare head rows): given the ids the target emitted,
 * pick those the list does not hold -- each id's first occurrence, in the
 * order given, while spare rows remain -- and copy them in as
 * dvl_learn_rows does, into rows *n_rows, *n_rows + 1, ...
 *   full:     the full head: N == V, d2t == NULL, id_base == 0.
 *   ids:      HOST int32 [n], each in [0, V), in any order, repeats allowed
 *             (n may be 0).
 *   row_of:   HOST int32 [V] (in/out): the trimmed row that holds id t, or
 *             -1 for an id the list lacks; learned ids get their rows.
 *   n_rows:   HOST (in/out): rows in use; the first spare row.
 *   capacity: rows the trimmed buffers hold (>= *n_rows).
 *   w_trim, scales_trim (NVFP4; NULL otherwise), d2t: the trimmed head's
 *             device buffers from row 0, sized for `capacity` rows.
 *   learned:  HOST int32 [n] (out): the ids learned, in row order; also the
 *             source of the d2t copy, read before the call returns.
 *   n_learned: HOST (out): how many.
 * Nothing is enqueued when nothing is learned.  Ordering as for
 * dvl_learn_rows: the first reducing call after a learn on that stream
 * must not set DVL_HEAD_STATIC on the trimmed head.  The host work is
 * O(n); nothing is allocated.
 * Errors: DVL_ERR_INVALID_ARG, DVL_ERR_OUT_OF_RANGE (an id outside [0, V):
 * nothing changed, nothing enqueued), DVL_ERR_CUDA (row_of and *n_rows
 * unchanged). */
dvl_status dvl_learn_missing(const dvl_head *full, const int32_t *ids, int32_t n,
                             int32_t *row_of, int32_t *n_rows, int32_t capacity, void *w_trim,
                             uint8_t *scales_trim, int32_t *d2t, int32_t *learned,
                             int32_t *n_learned, void *stream);

/* ---------------------------------------------------------------------- */
/* Host-only ranks builder (no GPU involved)                              */
/* ---------------------------------------------------------------------- */

/* counts[t] += 1 for every token t of tokens[0..n).  All host memory.
 * DVL_ERR_OUT_OF_RANGE (nothing counted) if a token lies outside [0, V). */
dvl_status dvl_histogram(const int32_t *tokens, int64_t n, int64_t V, int64_t *counts);

/* A shortlist of N ids from a histogram: the distinct forced ids first, in
 * rank order, then the other ids in rank order, cut at N (rank order =
 * higher count first, then lower id).  sorted != 0 sorts the result by id.
 * All host memory; ranks_out holds min(N, V) entries; *n_out receives that
 * count.  DVL_ERR_OUT_OF_RANGE if a forced id lies outside [0, V). */
dvl_status dvl_build_ranks(const int64_t *counts, int64_t V, const int32_t *forced,
                           int32_t n_forced, int32_t N, int32_t sorted,
                           int32_t *ranks_out, int32_t *n_out);

/* The sorted set union of two id lists (each taken as a set).  All host
 * memory; out holds na + nb entries; *n_out receives the union's size. */
dvl_status dvl_union_sorted(const int32_t *a, int32_t na, const int32_t *b, int32_t nb,
                            int32_t *out, int32_t *n_out);

#ifdef __cplusplus
}
#endif
#endif /* DVL_H */
