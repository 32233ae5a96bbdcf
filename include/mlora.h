/*
 * mlora.h -- C ABI of libmlora: gathered multi-LoRA shrink / expand on NVIDIA GB300 (sm_103a).
 *
 * THE OPERATION
 *   A LoRA-adapted projection computes y = x·W + s·(x·A)·B with a per-adapter A (d_in x r),
 *   B (r x d_out) and scale s = alpha / r ("Multi-LoRA Serving, in depth", section "The
 *   computation, unmerged"). The shared base product x·W is NOT part of this library: the
 *   caller passes its result as y, and the library adds the low-rank delta in place.
 *   Punica (arXiv 2310.18547), section 3.4 "The SGMV Operator", splits the delta into
 *       shrink   v = x·A        (d_in -> r; v starts from zero)
 *       expand   y += v·B       (r -> d_out, in place)
 *   and batches rows that use different adapters. For every row i whose adapter slot s is
 *   not -1 this library computes
 *       v[i][j] = sum_k x[i][k] · A_s[k][j]                                  j < rank[s]
 *       y[i][n] = round( y[i][n] + scale[s] · sum_{j<rank[s]} v[i][j] · B_s[j][n] )
 *   with fp32 accumulation, bf16/fp16 inputs, and one round-to-nearest-even of y.
 *
 *   Two ways to say which row uses which adapter:
 *     SGMV  segments: rows off[t] .. off[t+1]-1 use slot seg_slot[t], with
 *           0 = off[0] <= off[1] <= ... <= off[n] = num_rows (Punica section 3.4, segment
 *           boundaries s_0 = 0 < ... < s_n; the "sgmv" semantics quoted in the zh-TW Punica
 *           digest, section 5.4: y[s[i]:s[i+1]] += x[s[i]:s[i+1]] @ w[i]).
 *     BGMV  a slot per row, row_slot[i], -1 = no adapter (the "add_lora_bgmv" semantics in
 *           the zh-TW Punica digest, section 5.5; the reference loop of "Multi-LoRA Serving,
 *           in depth", section "Why a mixed batch needs special kernels").
 *   Empty segments are allowed and do nothing; the same slot may appear in several segments.
 *
 * ADAPTER POOLS  (mlora_pool, a host struct of device pointers; see below)
 *   stacked  A^T [num_slots][num_layers][r_max][d_in]   row j of A^T = column j of A
 *            B   [num_slots][num_layers][r_max][d_out]  row j of B
 *            (Punica's LoraWeight, zh-TW digest section 5.4: wa [layers, r, in_features],
 *            wb [layers, r, out_features]; slots padded to the largest rank as in the
 *            reference loop). Rows j >= rank[s] are never read.
 *   paged    S-LoRA (arXiv 2311.03285) "Unified Paging": a page is one vector of
 *            page_elems elements (one H-vector). A of rank R is R vectors of d_in elements
 *            (its columns), B is R vectors of d_out elements (its rows); pages sit anywhere
 *            in one pool of num_pages x page_elems elements. A vector longer than a page
 *            spans ceil(d / page_elems) pages (d = d_in for A, d_out for B), so the page
 *            tables are [num_slots][num_layers][r_max][ceil(d / page_elems)] int32: element
 *            k of vector j is element k % page_elems of page table[..][j][k / page_elems].
 *            With page_elems >= d this is one page per vector ([..][r_max][1]). Ranks differ
 *            per adapter and nothing is padded. Page elements past a vector's end are never
 *            read.
 *
 * CONVENTIONS FOR EVERY CALL
 *   - All array pointers are DEVICE pointers unless stated; the mlora_pool / mlora_problem
 *     structs themselves are read on the host during the call and may be freed afterwards.
 *   - The caller owns all memory (inputs, outputs, the pool, v). The library allocates no
 *     device memory in any call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *     and never synchronise the host.
 *   - x [num_rows][ldx], y [num_rows][ldy]: row-major bf16/fp16 (the pool's dtype), ldx >=
 *     d_in, ldy >= d_out. v [num_rows][r_max]: fp32, written by shrink at columns < rank[s]
 *     of adapted rows (other entries unspecified), read by expand.
 *   - Alignment (16-byte rows for bulk copies): x, y, a_t, b, pages 16-byte aligned; ldx,
 *     ldy, d_in, d_out, page_elems multiples of 8 elements; v 4-byte aligned.
 *   - Limits: 1 <= r_max <= MLORA_MAX_RANK; d_in, d_out >= 8; num_rows >= 0; 0 <= layer <
 *     num_layers; num_segments >= 0. num_rows == 0 is a no-op that launches nothing; then x,
 *     y, v and row_slot may be NULL (empty arrays), the pool is still validated.
 *   - Host-detectable errors return a negative MLORA_ERR_* code BEFORE anything is launched
 *     (nothing is written). A failed launch returns MLORA_ERR_CUDA (text: lora_error_string).
 *   - Device-detectable metadata errors never trap: the kernel ORs an MLORA_STATUS_* bit
 *     into *dev_status (if dev_status is not NULL) and skips the affected rows, leaving
 *     their y and v untouched:
 *        offsets not 0 = off[0] <= ... <= off[n] = num_rows   -> BAD_OFFSETS, whole call skipped
 *        slot < -1 or slot >= num_slots                      -> BAD_SLOT, rows skipped
 *        rank[s] outside [1, r_max]                          -> BAD_RANK, rows skipped
 *        a page id of a vector j < rank[s] outside [0, num_pages) -> BAD_PAGE, rows skipped
 *     A wait that exceeds its time limit inside a kernel sets MLORA_STATUS_TIMEOUT.
 *   - Slot -1 rows are never written (their y keeps its exact bits).
 *   - Calls whose outputs overlap on the device must be ordered by the caller (one stream).
 */
#ifndef MLORA_H
#define MLORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MLORA_API __attribute__((visibility("default")))
#else
#define MLORA_API
#endif

#define MLORA_ABI_VERSION 1
#define MLORA_MAX_RANK 128

/* Return codes. */
#define MLORA_OK 0
#define MLORA_ERR_NULL (-1)        /* a required pointer is NULL */
#define MLORA_ERR_DTYPE (-2)       /* dtype is not MLORA_BF16 / MLORA_FP16 */
#define MLORA_ERR_SHAPE (-3)       /* a size or index is out of range */
#define MLORA_ERR_ALIGN (-4)       /* a pointer, leading dimension or size breaks the alignment rule */
#define MLORA_ERR_POOL (-5)        /* malformed pool descriptor */
#define MLORA_ERR_CUDA (-6)        /* a CUDA call failed; see lora_error_string(MLORA_ERR_CUDA) */
#define MLORA_ERR_TOO_LARGE (-7)   /* the call needs more than the built-in scratch of lora_sgmv_noalloc */

/* Device status bits, OR-ed into *dev_status. */
#define MLORA_STATUS_BAD_OFFSETS 1
#define MLORA_STATUS_BAD_SLOT 2
#define MLORA_STATUS_BAD_RANK 4
#define MLORA_STATUS_BAD_PAGE 8
#define MLORA_STATUS_TIMEOUT 16

typedef enum { MLORA_BF16 = 0, MLORA_FP16 = 1 } mlora_dtype;
typedef enum { MLORA_POOL_STACKED = 0, MLORA_POOL_PAGED = 1 } mlora_pool_kind;

/* One adapter pool for one projection shape (d_in -> d_out), every layer, every slot.
 * Host struct; every pointer in it is a device pointer owned by the caller. */
typedef struct {
  int32_t kind;        /* mlora_pool_kind */
  int32_t dtype;       /* mlora_dtype: the element type of the pool, x and y */
  int32_t num_slots;   /* adapters resident in the pool (slot ids 0 .. num_slots-1) */
  int32_t num_layers;
  int32_t r_max;       /* stride of the rank dimension (stacked) / of the page tables */
  int32_t d_in;        /* h1: columns of x, rows of A */
  int32_t d_out;       /* h2: columns of y and of B */
  const void *a_t;     /* stacked: A^T [num_slots][num_layers][r_max][d_in]  (NULL when paged) */
  const void *b;       /* stacked: B   [num_slots][num_layers][r_max][d_out] (NULL when paged) */
  const void *pages;   /* paged: [num_pages][page_elems]                     (NULL when stacked) */
  int64_t page_elems;  /* paged: elements per page, a multiple of 8, at least 8 */
  int64_t num_pages;   /* paged */
  const int32_t *a_page_table; /* paged: [num_slots][num_layers][r_max][ceil(d_in/page_elems)], pages of column j of A */
  const int32_t *b_page_table; /* paged: [num_slots][num_layers][r_max][ceil(d_out/page_elems)], pages of row j of B */
  const int32_t *rank;  /* [num_slots], each in [1, r_max] */
  const float *scale;   /* [num_slots], alpha / rank, applied by the expand */
} mlora_pool;

/* Launch flags of the _ex calls. */
#define MLORA_LAUNCH_PROGRAMMATIC 1u /* programmatic dependent launch for this call (see
                                        lora_set_programmatic_launch) */

/* ---- two-phase form (Punica section 3.4: one shrink launch, one expand launch) --------- */

/* SGMV shrink: v[i][j] = sum_k x[i][k] A_s[k][j] for rows of segments with slot s != -1.
 * seg_offsets [num_segments+1] and seg_slot [num_segments] are int32 device arrays. */
MLORA_API int lora_sgmv_shrink(float *v, const void *x, int64_t ldx, const mlora_pool *pool, const int32_t *seg_offsets,
                     const int32_t *seg_slot, int32_t num_segments, int32_t num_rows, int32_t layer,
                     int32_t *dev_status, void *stream);

/* SGMV expand: y[i][n] = round(y[i][n] + scale[s] sum_j v[i][j] B_s[j][n]), in place. */
MLORA_API int lora_sgmv_expand(void *y, int64_t ldy, const float *v, const mlora_pool *pool, const int32_t *seg_offsets,
                     const int32_t *seg_slot, int32_t num_segments, int32_t num_rows, int32_t layer,
                     int32_t *dev_status, void *stream);

/* BGMV shrink: as lora_sgmv_shrink with slot row_slot[i] per row (int32 [num_rows], -1 = none). */
MLORA_API int lora_bgmv_shrink(float *v, const void *x, int64_t ldx, const mlora_pool *pool, const int32_t *row_slot,
                     int32_t num_rows, int32_t layer, int32_t *dev_status, void *stream);

/* BGMV expand: as lora_sgmv_expand with slot row_slot[i] per row. */
MLORA_API int lora_bgmv_expand(void *y, int64_t ldy, const float *v, const mlora_pool *pool, const int32_t *row_slot,
                     int32_t num_rows, int32_t layer, int32_t *dev_status, void *stream);

/* ---- fused form: shrink and expand of one projection in one call ------------------------
 * Same result as shrink followed by expand. For decode-sized segments both phases run in one
 * launch and v stays on chip (a cluster of CTAs splits d_in, sums its partial v through
 * distributed shared memory, then splits d_out). v_scratch [num_rows][r_max] fp32 is
 * caller-owned scratch that the library may use when it runs the two phases as separate
 * launches (long prefill segments); its contents afterwards are unspecified. It is required. */
MLORA_API int lora_sgmv(void *y, int64_t ldy, const void *x, int64_t ldx, const mlora_pool *pool, const int32_t *seg_offsets,
              const int32_t *seg_slot, int32_t num_segments, int32_t num_rows, int32_t layer, float *v_scratch,
              int32_t *dev_status, void *stream);

MLORA_API int lora_bgmv(void *y, int64_t ldy, const void *x, int64_t ldx, const mlora_pool *pool, const int32_t *row_slot,
              int32_t num_rows, int32_t layer, float *v_scratch, int32_t *dev_status, void *stream);

/* lora_bgmv with launch flags. Device-side grouping of the rows (Punica section 3.4, "Batch
 * Layout Construction": rows that share an adapter form one group; "Multi-LoRA Serving, in
 * depth", section "The decode cost model": each adapter read once per step): a first small
 * kernel orders the rows by (rank descending, slot) on the GPU, the main kernel then walks the
 * rows in that order. Rows of one adapter run side by side, so the adapter comes from HBM once;
 * the heaviest rows start first. The caller's row order, x and y are unchanged; the order is
 * kept in v_scratch (2 x num_rows int32). On pools of r_max 32 to 128 (S-LoRA section 3,
 * "Heterogeneous Batching Kernels": adapters of many ranks in one pool) the grouped order is
 * also cut into segments of up to 4 rows that share a slot (num_rows + 1 more int32 of
 * v_scratch), and a streaming kernel takes over: a cluster of CTAs per segment streams the
 * adapter's A^T and B rank-rows through shared-memory rings once for the segment's rows,
 * segments in snake order over the clusters, largest first. lora_bgmv groups batches of at least
 * 128 rows (up to 4096 rows, r_max >= 2); the flags override that:
 *   MLORA_LAUNCH_GROUP_ROWS   group (when num_rows <= 4096 and r_max >= 2)
 *   MLORA_LAUNCH_NO_GROUPING  never group
 *   MLORA_LAUNCH_PROGRAMMATIC programmatic dependent launch for the first kernel of the call
 * Other bits are rejected with MLORA_ERR_SHAPE. Grouped on the main kernel, results are the same
 * bits as ungrouped (every row's arithmetic is the same); streamed, the sums run in another fixed
 * order (the same bits on every call, within the same tolerance of the exact result). */
#define MLORA_LAUNCH_GROUP_ROWS 2u
#define MLORA_LAUNCH_NO_GROUPING 4u
MLORA_API int lora_bgmv_ex(void *y, int64_t ldy, const void *x, int64_t ldx, const mlora_pool *pool,
                           const int32_t *row_slot, int32_t num_rows, int32_t layer, float *v_scratch, uint32_t flags,
                           int32_t *dev_status, void *stream);

/* ---- fused form without a scratch argument -------------------------------------------------
 * lora_sgmv_noalloc: lora_sgmv for callers that cannot hand the library a device buffer --
 * code that may not allocate device memory, such as a plugin running inside a host engine
 * that owns all device memory and passes the plugin only its inputs and outputs, or a
 * latency-critical path where cudaMalloc (which can synchronise the device) is not acceptable.
 * Instead of v_scratch it uses an array built into the library: MLORA_NOALLOC_MAX_FLOATS fp32
 * values (4 MiB) in device memory, which every GPU that loads the library holds until the
 * process exits. The call itself allocates nothing (no cudaMalloc, no cudaFree, no library
 * allocator).
 *   - Limit: num_rows * pool->r_max <= MLORA_NOALLOC_MAX_FLOATS; a larger call returns
 *     MLORA_ERR_TOO_LARGE and launches nothing.
 *   - The first call on a device, with that device current, looks up the array's device
 *     address (cudaGetSymbolAddress); make that first call before any stream capture.
 *   - Every call shares the one array, and it keeps the last call's contents. Nothing in it
 *     must start at zero: the shrink writes every entry the expand later reads.
 *   - Calls whose kernels may run at the same time on the GPU (other streams, other host
 *     threads) race on the array; order them, e.g. on one stream.
 * Same arguments, results and errors as lora_sgmv otherwise. (No counterpart on the pages:
 * an interface convenience of this library.) */
#define MLORA_NOALLOC_MAX_FLOATS (1 << 20)
MLORA_API int lora_sgmv_noalloc(void *y, int64_t ldy, const void *x, int64_t ldx, const mlora_pool *pool,
                                const int32_t *seg_offsets, const int32_t *seg_slot, int32_t num_segments,
                                int32_t num_rows, int32_t layer, int32_t *dev_status, void *stream);

/* ---- grouped form: several projections over the same rows in one call --------------------
 * Punica builds the segments once per batch and reuses them for all 7 projections of every
 * layer (section 3.4, "Batch Layout Construction"). A group runs the fused op of each problem
 * in one launch: typically the projections that read the same x (q, k, v; or gate, up).
 * Each problem has its own x, y, pool, layer and v_scratch; all share the rows' metadata.
 * The mlora_problem array is a host array of at most MLORA_MAX_GROUP entries, and every pool
 * in a group must have the same dtype. */
#define MLORA_MAX_GROUP 8
typedef struct {
  void *y;
  int64_t ldy;
  const void *x;
  int64_t ldx;
  const mlora_pool *pool; /* host pointer */
  int32_t layer;
  float *v_scratch;       /* [num_rows][pool->r_max] fp32 */
} mlora_problem;

MLORA_API int lora_sgmv_grouped(const mlora_problem *problems, int32_t num_problems, const int32_t *seg_offsets,
                      const int32_t *seg_slot, int32_t num_segments, int32_t num_rows, int32_t *dev_status,
                      void *stream);

/* lora_sgmv_grouped with launch flags given per call instead of taken from the calling thread's
 * setting (lora_set_programmatic_launch). flags: 0 or MLORA_LAUNCH_PROGRAMMATIC; other bits are
 * rejected with MLORA_ERR_SHAPE. (No counterpart on the pages: a launch-latency measure for
 * GB300.) */
MLORA_API int lora_sgmv_grouped_ex(const mlora_problem *problems, int32_t num_problems, const int32_t *seg_offsets,
                                   const int32_t *seg_slot, int32_t num_segments, int32_t num_rows, uint32_t flags,
                                   int32_t *dev_status, void *stream);

/* ---- sequence form: the grouped calls of a whole step in one call ------------------------
 * A decoder step issues one grouped call per dependent stage of every layer (q,k,v; o;
 * gate,up; down for a Llama layer: 4 x num_layers calls). lora_sgmv_sequence issues such a
 * list of grouped calls, in order, on `stream`, from native code: the same launches as
 * num_groups calls of lora_sgmv_grouped_ex, for one call's host cost. Every group is validated
 * before anything is launched (a host-detectable error in any group returns its code and
 * launches nothing). flags: MLORA_LAUNCH_PROGRAMMATIC gives every call after the first
 * programmatic dependent launch (the first keeps an ordinary dependency on whatever ran
 * before); the groups then must not write each other's metadata or pools, which this
 * library's calls never do. Each group's problems must not write the x of a later group
 * while that group may read it -- as in a real step, where x of the next stage comes from
 * other kernels. (No counterpart on the pages: Punica issues 7 x L launches per step from
 * the host; this is the same schedule issued natively.) */
typedef struct {
  const mlora_problem *problems; /* host array of num_problems entries */
  int32_t num_problems;          /* 1 .. MLORA_MAX_GROUP */
  const int32_t *seg_offsets;    /* device [num_segments + 1] */
  const int32_t *seg_slot;       /* device [num_segments] */
  int32_t num_segments;
  int32_t num_rows;
} mlora_group;

MLORA_API int lora_sgmv_sequence(const mlora_group *groups, int32_t num_groups, uint32_t flags, int32_t *dev_status,
                                 void *stream);

/* ---- utilities --------------------------------------------------------------------------- */

/* Static text for a return code; for MLORA_ERR_CUDA it names the last CUDA error this thread saw. */
MLORA_API const char *lora_error_string(int code);

/* Programmatic dependent launch (off by default), for the calling host thread. When on, every
 * later call from this thread launches its kernels so that they may start while the previous
 * kernel in the stream is still running: before waiting for that kernel a kernel reads only its
 * rows' metadata (offsets, slots), the pool descriptor arrays (rank, scale, page tables) and the
 * adapter weights, and it requests the weights; x, y, v and dev_status are touched only after
 * the wait. Turn it on only where the kernel launched just before each call does not write those
 * inputs -- e.g. a sequence of this library's calls, or calls whose inputs were written by copies
 * or at least one kernel earlier. Other host threads keep their own setting. Returns this
 * thread's previous setting. (No counterpart on the pages: a launch-latency measure for GB300.) */
MLORA_API int lora_set_programmatic_launch(int enable);

/* MLORA_ABI_VERSION of the loaded library. */
MLORA_API int lora_abi_version(void);

/* Number of kernel launches the library has issued from this process (all threads). */
MLORA_API int64_t lora_launch_count(void);

/* Testing hook for the time-out path: limit, in nanoseconds, of the waits inside the CUDA-core
 * kernels launched later by the calling thread (the waits for their own bulk copies and for
 * their cluster peers' partial sums). 0 restores the default of 2 s. With a limit of a few
 * nanoseconds a wait gives up unless its data has already landed, the kernel sets
 * MLORA_STATUS_TIMEOUT and skips the work that needed the data, and copies still in flight are
 * drained (with the default limit) before the kernel exits. Not for production use: results of
 * rows whose waits gave up are left unwritten. (No counterpart on the pages.) */
MLORA_API void lora_test_set_wait_limit_ns(uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* MLORA_H */
