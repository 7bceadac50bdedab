/*
 * libtopk: ragged per-row top-K over fp32 logits on one NVIDIA GB300 (sm_103a).
 *
 * The operation is the token selection of long-context sparse attention
 * (vLLM PR #54110 page, "Feature and motivation": the persistent_topk kernel
 * serves DSA models in long-context inference). Every row r of a logits matrix
 * has its own valid length len_r. For every row, the library returns the
 * indices of its topk largest values among x[r, 0:len_r]. The per-row lengths
 * and the TopK values the pages' kernel is built for (512 / 1024 / 2048) follow
 * the persistent_topk launcher excerpt on the vLLM PR #41189 page
 * ("Implementation breakdown"); here any TopK from 1 to 4096 is accepted. MTP layouts,
 * where a request contributes next_n adjacent rows, each with its own length,
 * follow the vLLM PR #54110 page ("Implementation breakdown" item 2: next_n is
 * the second dimension of a 2-D lengths tensor).
 *
 * Selection rule (the pages leave it open; this library fixes it):
 *   - larger value first; on equal values, the smaller index first;
 *   - values compare exactly as IEEE floats: -0.0 equals +0.0, subnormals are
 *     not flushed, +inf and -inf are ordinary values;
 *   - NaN inside a valid prefix is outside the contract (result unspecified);
 *   - a row with len_r < topk returns its len_r indices, then -1 padding;
 *   - the order of the indices inside an output row is unspecified (the
 *     result is a set; sort it by (value desc, index asc) if order matters).
 *
 * Conventions for every entry point:
 *   - pointers named logits, lengths, out_idx and workspace are DEVICE
 *     pointers owned by the caller; the library allocates and frees nothing;
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream); all device work is enqueued on it, nothing synchronises it
 *     except topk_get_status;
 *   - errors found on the host are returned synchronously as a topk_status
 *     code and nothing is enqueued; no C++ exception crosses this boundary;
 *   - conditions found on the device (a clamped length, a timed-out wait) set
 *     sticky bits in the workspace status word, read with topk_get_status.
 */
#ifndef LIBTOPK_H_
#define LIBTOPK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum {
  TOPK_OK = 0,
  TOPK_ERR_INVALID_ARG = 1,         /* null pointer, negative size, next_n not dividing num_rows ... */
  TOPK_ERR_UNSUPPORTED_TOPK = 2,    /* topk outside [1, 4096] (or above 2048 with the paired shape) */
  TOPK_ERR_MISALIGNED = 3,          /* logits/lengths/out_idx not 4-byte, workspace not 16-byte aligned */
  TOPK_ERR_WORKSPACE_TOO_SMALL = 4, /* topk_options.workspace_bytes below topk_workspace_size */
  TOPK_ERR_CUDA = 5,                /* a CUDA runtime call failed (launch, query, copy) */
  TOPK_ERR_BARRIER_TIMEOUT = 6,     /* reported by topk_get_status: a wait on the device gave up */
  TOPK_ERR_LENGTH_CLAMPED = 7,      /* reported by topk_get_status: some length was outside [0, row_stride] */
  TOPK_ERR_PLAN = 8                 /* no launch configuration fits the device (e.g. kernel not resident) */
} topk_status;

/* Sticky bits of the device status word (first 4 bytes of the workspace). */
#define TOPK_DEV_LENGTH_CLAMPED 0x1u  /* a length < 0 was read as 0, or > row_stride as row_stride */
#define TOPK_DEV_BARRIER_TIMEOUT 0x2u /* a CTA of a row group waited longer than the barrier limit */
#define TOPK_DEV_STAGE_TIMEOUT 0x4u   /* a staging copy did not land within the limit */
/* A launch that splits rows found TOPK_DEV_BARRIER_TIMEOUT or TOPK_DEV_STAGE_TIMEOUT
 * already set: the timed-out launch left the workspace's group words as they were,
 * so this launch wrote rows of -1 instead of merging through them. Every such
 * launch does the same until topk_workspace_init clears the workspace. */
#define TOPK_DEV_WORKSPACE_DIRTY 0x8u

/* Tuning and test knobs for topk_ragged_ex. Zero-initialise, then set fields.
 * A field left at 0 takes the value of its environment variable, read once per
 * process, where one exists: LIBTOPK_FORCE_CTAS_PER_GROUP,
 * LIBTOPK_LONG_ROW_THRESHOLD, LIBTOPK_BARRIER_TIMEOUT_US, LIBTOPK_MERGE and
 * LIBTOPK_DEPENDENT_LAUNCH (topk_ragged and topk_ragged_static read them too). */
typedef struct {
  /* 0 = planner decides; 1 = one CTA per row; 2..16 = that many CTAs split each row
   * (with shape 4: 2..8, the CTAs of one thread-block cluster per row). */
  int force_ctas_per_group;
  /* 0 = default; rows whose row_stride exceeds this may be split across CTAs. */
  int64_t long_row_threshold;
  /* 0 = default (1 s); limit of every device-side wait, in microseconds. */
  uint32_t barrier_timeout_us;
  /* Test only. 1 = CTA 1 of row group 0 leaves before its first group barrier
   * (workspace merge), so the other CTAs' waits run out and set
   * TOPK_DEV_BARRIER_TIMEOUT; 2 = CTA 1 of cluster 0 withholds its arrivals at
   * the launch's first cluster merge sync, so every member's bounded wait runs
   * out (TOPK_DEV_BARRIER_TIMEOUT) and all of them leave through the cluster's
   * exit barrier. Either way the workspace must then be re-initialised with
   * topk_workspace_init (see TOPK_DEV_WORKSPACE_DIRTY). 3 = the short-row
   * kernel's row split over a cluster (shapes 4 and 5 with G > 1): CTA 1 of
   * cluster 0 treats the first copy it waits for as late and gives up as on a
   * time-out: TOPK_DEV_STAGE_TIMEOUT is set, row 0 is left unwritten, every
   * other row is selected, and every CTA of the cluster leaves through the
   * same barriers. The workspace needs no re-initialisation after it. */
  int inject_skip_arrival;
  /* 0 = unchecked; otherwise the workspace's size, checked against topk_workspace_size. */
  size_t workspace_bytes;
  /* 0 = every SM; otherwise at most this many co-resident CTAs are planned. */
  int max_ctas;
  /* How the CTAs splitting a row merge their candidates. 0 = planner decides;
   * 1 = through the workspace, with a grid-level barrier (any G); 2 = inside a
   * thread-block cluster, through its distributed shared memory (G <= 8). */
  int merge;
  /* CTA shape. 0 = planner decides; 1 = one CTA of 24 consumer warps per SM;
   * 2 = two CTAs of 12 consumer warps per SM (whole rows only); 3 = a CTA of 8
   * consumer warps in about 83 KB of shared memory (whole rows only), the
   * low-shared-memory mode for devices or partitions where 1 and 2 do not fit;
   * 4 = the short-row kernel: one CTA of 32 warps per SM owns whole rows, held
   * in a 128 KB shared-memory ring (rows of up to 32768 elements) or streamed
   * through it, or the CTAs of a thread-block cluster share each row (planned
   * for few long rows, or forced with force_ctas_per_group 2..8; contiguous
   * rows only: strided views keep whole rows); 5 = the same kernel with 16
   * warps per CTA (512 threads), faster on short rows and split rows. */
  int shape;
  /* Programmatic dependent launch of the short-row kernel (shapes 4 and 5).
   * 0 = default (on); 1 = on; 2 = off. On, the kernel is launched with
   * programmatic stream serialisation: its CTAs may start while the kernel
   * before it on `stream` finishes, and every thread waits for that kernel to
   * complete (griddepcontrol.wait, its writes then visible) before its first
   * access to global memory; each CTA then lets the next kernel on the stream
   * start early in the same way (griddepcontrol.launch_dependents), which is
   * safe only for a kernel that waits likewise before it reads the indices.
   * Off, plain stream order. The other shapes always launch in plain order.
   * Any other value: TOPK_ERR_INVALID_ARG. */
  int dependent_launch;
} topk_options;

/* Properties of a device as the planner sees them. */
typedef struct {
  int num_sms;        /* streaming multiprocessors */
  int max_smem_optin; /* opt-in shared memory per block, bytes */
  int smem_per_cta;   /* dynamic shared memory the kernel needs, bytes */
  int ctas_per_sm;    /* resident CTAs per SM for the exact kernel instance (occupancy) */
  /* cluster_groups[c], c = 2..8: clusters of c CTAs of the kernel that can be
   * resident at once (0 = none; entries 0 and 1 are unused). */
  int cluster_groups[9];
  int pair_smem_per_cta; /* the same for the paired shape (two CTAs per SM) */
  int pair_ctas_per_sm;
  int small_smem_per_cta; /* the same for the small shape */
  int small_ctas_per_sm;
  int short_smem_per_cta; /* the same for the short-row kernel */
  int short_ctas_per_sm;
  /* short_cluster_groups[c], c = 2..8: resident clusters of c CTAs of the
   * short-row kernel's cluster form (a row split over a cluster). */
  int short_cluster_groups[9];
  int short16_smem_per_cta; /* the same three for the short-row kernel with 16 warps per CTA */
  int short16_ctas_per_sm;
  int short16_cluster_groups[9];
} topk_device_props;

/* A launch configuration. */
typedef struct {
  int ctas_per_group; /* G: CTAs that split one row (1 = a CTA owns whole rows) */
  int num_groups;     /* row groups; group g handles rows g, g + num_groups, ... */
  int grid;           /* CTAs launched = num_groups * ctas_per_group */
  int threads;        /* threads per CTA */
  int smem_bytes;     /* dynamic shared memory per CTA */
  int cooperative;    /* 1 when the CTAs of a group wait on one another through the workspace */
  int cluster;        /* 1 when the CTAs of a group form a cluster and merge in its shared memory */
  int shape;          /* 1 = one CTA of 24 consumer warps per SM, 2 = two CTAs of 12 per SM,
                         3 = the small shape (8 consumer warps, low shared memory),
                         4 = the short-row kernel, 5 = the short-row kernel with 16 warps */
} topk_plan;

/*
 * Workspace bytes needed on `device` (the other arguments are accepted for
 * forward compatibility; the size depends only on the device). The workspace
 * holds the device status word and, per row group, the histograms, counters
 * and barrier words that CTAs splitting one row exchange (the role of the
 * RadixRowState workspace on the vLLM PR #41444 page, "Executive summary").
 * Returns 0 if the device cannot be queried.
 */
size_t topk_workspace_size(int device, int64_t num_rows, int64_t row_stride, int next_n, int topk);

/*
 * Zeroes a workspace once, after allocation (stream-ordered memset). After that
 * no per-call clearing is needed: every successful topk_ragged leaves the
 * workspace zeroed again, apart from the sticky status word, which this call
 * also clears (the per-call memset it replaces is the one the vLLM PR #41748
 * page, "Motivation", removes for a 3-5 us saving per decode step).
 * After a TOPK_DEV_BARRIER_TIMEOUT or TOPK_DEV_STAGE_TIMEOUT the workspace must
 * be re-initialised: until then, launches that split rows refuse to merge
 * through it and write rows of -1 (TOPK_DEV_WORKSPACE_DIRTY).
 */
int topk_workspace_init(void* workspace, size_t bytes, void* stream);

/*
 * Ragged per-row top-K.
 *   logits     fp32 [num_rows, row_stride], row-major, 4-byte aligned; row r
 *              starts at logits + r * row_stride; the buffer holds all
 *              num_rows * row_stride elements. Only x[r, 0:len_r] is used;
 *              elements of a row past len_r may be read, never used.
 *   row_stride elements between row starts, >= 1; also the upper bound of
 *              every length (it plays the role of max_seq_len).
 *   lengths    int32 [num_rows] (or [num_rows / next_n, next_n] flattened):
 *              valid length of each row; values outside [0, row_stride] are
 *              clamped and flagged with TOPK_DEV_LENGTH_CLAMPED.
 *   num_rows   rows; 0 is a no-op.
 *   next_n     rows per request (MTP); must divide num_rows.
 *   topk       1..4096, any value (the pages' kernel is built for 512, 1024 and
 *              2048; here TopK is a run-time argument of one kernel).
 *   out_idx    int32 [num_rows, topk], written in full.
 *   workspace  at least topk_workspace_size bytes, 16-byte aligned, zeroed once
 *              by topk_workspace_init. Calls that may run concurrently on the
 *              GPU must not share a workspace.
 *   stream     cudaStream_t.
 * One kernel launch per call; no allocation, memset or host synchronisation, so
 * the call can be captured in a CUDA graph. The first call on a device queries
 * and caches its properties; make it before any stream capture.
 */
int topk_ragged(const float* logits, int64_t row_stride, const int32_t* lengths,
                int64_t num_rows, int next_n, int topk, int32_t* out_idx,
                void* workspace, void* stream);

/*
 * topk_ragged without a workspace argument, for callers that cannot allocate
 * device memory (they may only enqueue work on the streams and buffers they
 * are given). The pages describe no such entry point; it has no counterpart
 * there. Scratch comes from a fixed device array inside the library, about
 * 3.8 MB per GPU that loads it, held until the process exits; it fits every
 * plan on a GPU with up to 152 SMs, and a plan needing more row groups returns
 * TOPK_ERR_WORKSPACE_TOO_SMALL. Arguments, layout and host-side errors are
 * those of topk_ragged. No allocation is made, ever.
 *   - The first call on a device looks up the array and zeroes it on `stream`;
 *     make that first call before any stream capture.
 *   - All calls on a device share the one array: calls that may overlap on
 *     the GPU (different streams without ordering) race and must not be made.
 *   - The device status word is not readable through this entry point. A
 *     device-side time-out (a wait of a second, which a working GPU never
 *     reaches) leaves the array marked: from then on, calls whose plan splits
 *     rows write rows of -1 instead of merging through stale words, until the
 *     process restarts (use topk_ragged with a workspace where that matters).
 *   - The LIBTOPK_* environment knobs apply as they do to topk_ragged.
 */
int topk_ragged_static(const float* logits, int64_t row_stride, const int32_t* lengths,
                       int64_t num_rows, int next_n, int topk, int32_t* out_idx, void* stream);

/*
 * topk_ragged over a strided logits view: element (r, i) is
 * logits[r * row_stride + i * col_stride], for 0 <= i < max_len. The pages'
 * decode fallback receives both strides of the logits tensor (vLLM PR #54110
 * page, "Implementation breakdown", the top_k_per_row_decode call with
 * logits.stride(0) and logits.stride(1)); a transposed view has row_stride 1
 * and col_stride equal to the number of rows.
 *   row_stride  >= 0 elements between row starts.
 *   col_stride  >= 1 elements between consecutive columns; 1 = contiguous rows
 *               (then this is topk_ragged with max_len as the length bound).
 *   max_len     1..2^31-1 columns per row: every length is clamped into
 *               [0, max_len], and only elements i < max_len are ever read.
 * Other arguments, ownership and errors as in topk_ragged; options may be
 * NULL. With col_stride > 1 the rows are read element by element (no bulk
 * copies): correct for any layout, but each element costs a memory sector.
 */
int topk_ragged_strided(const float* logits, int64_t row_stride, int64_t col_stride, int64_t max_len,
                        const int32_t* lengths, int64_t num_rows, int next_n, int topk, int32_t* out_idx,
                        void* workspace, void* stream, const topk_options* options);

/*
 * Values and order of selected rows (one extra launch on `stream`). For every
 * row r of out_idx (int32 [num_rows, topk], as written by topk_ragged or
 * topk_ragged_strided on the same logits): if out_val is not NULL, writes the
 * value of each selected index to out_val (fp32 [num_rows, topk]; -inf where
 * the index is -1); if sort != 0, first reorders the row in place by value
 * descending, then index ascending, -1 entries last (the order the pages' tie
 * rule implies; the selection itself returns a set). Logits are addressed as
 * in topk_ragged_strided; an index outside [0, max_len) is treated as -1 and
 * never read. No workspace; the launch needs up to 32 KB of shared memory.
 * It is launched with programmatic dependent launch (unless
 * LIBTOPK_DEPENDENT_LAUNCH=2): its CTAs may start while the kernel before it
 * on `stream` (the selection) finishes, and wait for it to complete before
 * they read out_idx or the logits.
 * Returns the topk_status codes of topk_ragged (TOPK_OK when num_rows is 0, or
 * when sort is 0 and out_val is NULL: nothing to do).
 */
int topk_gather_sort(const float* logits, int64_t row_stride, int64_t col_stride, int64_t max_len,
                     int64_t num_rows, int topk, int32_t* out_idx, float* out_val, int sort, void* stream);

/*
 * topk_ragged with options (NULL options = topk_ragged). The pages have no
 * counterpart: this is the library's own entry for tests and tuning (forced
 * splits, merge kind, CTA shape, time-out, injected failures); the selection
 * it computes is the one topk_ragged computes.
 */
int topk_ragged_ex(const float* logits, int64_t row_stride, const int32_t* lengths,
                   int64_t num_rows, int next_n, int topk, int32_t* out_idx,
                   void* workspace, void* stream, const topk_options* options);

/*
 * Synchronises `stream` and copies the workspace's sticky status word
 * (TOPK_DEV_* bits) to *device_status. For tests and debugging, not for the
 * hot path. Returns TOPK_OK, or TOPK_ERR_CUDA if the copy failed. The library's
 * own: the pages' launcher reports errors by exceptions on the host and has no
 * device-side status. The word is a bit set, hence unsigned (uint32_t*).
 */
int topk_get_status(const void* workspace, void* stream, uint32_t* device_status);

/* Static description of a topk_status code (never NULL). The library's own (the
 * pages report errors as exception messages); no passage corresponds. */
const char* topk_status_string(int code);

/*
 * Fills *props for `device`: SM count, opt-in shared memory per block, and for
 * each CTA shape of the kernel its shared memory and occupancy (queried for
 * the exact kernel, as the vLLM PR #41189 page's "Implementation breakdown"
 * item 1 requires), plus the co-resident cluster counts.
 */
int topk_query_device(int device, topk_device_props* props);

/*
 * The host planner, a pure function of its arguments (no CUDA call), so it can
 * be checked against made-up devices. It sizes the grid from the occupancy in
 * *props and never plans more co-resident CTAs than num_sms * ctas_per_sm when
 * CTAs of a group wait on one another through the workspace; the deadlock of
 * an oversized cooperative grid (vLLM PR #41189 page, "Feature and
 * motivation": TopK=1024 with MTP=1) cannot be planned. A cluster merge waits
 * only inside a cluster, whose CTAs the hardware schedules together, and plans
 * at most cluster_groups[G] groups. options may be NULL.
 */
int topk_make_plan(const topk_device_props* props, int64_t num_rows, int64_t row_stride,
                   int next_n, int topk, const topk_options* options, topk_plan* plan);

#ifdef __cplusplus
}
#endif

#endif /* LIBTOPK_H_ */
