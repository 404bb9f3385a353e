/*
 * tt_emb.h -- C ABI of the GB300 (sm_103a) TT-EmbeddingBag library, libttemb.so.
 *
 * A TT-EmbeddingBag is a drop-in EmbeddingBag whose E x D table is held as
 * three tensor-train cores (TT-Rec / FBTT-Embedding pages; FBTT README,
 * opening paragraph and "How FBTT-Embedding works").  Row i, decoded as
 * i = i1 p2 p3 + i2 p3 + i3, is the chain product G1[i1] G2[i2] G3[i3]; the
 * rows named by each bag are sum- or mean-pooled (optionally weighted) into
 * one output row, and the backward pass applies a fused sparse SGD update to
 * the touched core slices (FBTT README, "Fused Kernel", sparse=True).
 *
 * Conventions for every entry point:
 *   - Pointers named *_dev are CUDA device pointers; the caller owns them and
 *     keeps them valid until the work queued on `stream` has completed.
 *   - Core k of a table is float32 [p_k][r_{k-1}][q_k][r_k] (r_0 = r_3 = 1),
 *     C-contiguous, so slice G_k[i_k] is contiguous.  The FBTT README's
 *     "Initialization" section gives the cores as r_{k-1} x p_k x q_k x r_k;
 *     the slice index is moved first here, which changes no value.
 *   - Column j of a row is j = j1 q2 q3 + j2 q3 + j3.
 *   - Bags are CSR: offsets_dev has num_bags + 1 int64 entries, offsets[0] = 0,
 *     offsets[num_bags] = nnz, non-decreasing; bag g holds the lookups
 *     offsets[g] .. offsets[g+1]-1.  (PyTorch's EmbeddingBag passes the B
 *     start positions only; append nnz to convert.)
 *   - A handle is not thread-safe; calls on one handle must be issued from
 *     one host thread and be ordered on the streams they are given.
 *   - No call throws; each returns a tt_status.  Host-side validation runs
 *     before anything is queued, and on failure nothing is modified.  Errors
 *     found on the device (an index outside [0, E), malformed offsets) are
 *     recorded in a sticky per-handle flag read by tt_emb_get_last_error();
 *     the offending lookups contribute nothing to the output, and a backward
 *     pass that follows such a forward pass leaves every core unchanged.
 */
#ifndef TT_EMB_H
#define TT_EMB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tt_emb tt_emb;          /* opaque handle */
typedef struct CUstream_st* tt_stream; /* same type as cudaStream_t; NULL = legacy default stream */

typedef enum {
    TT_OK = 0,
    TT_ERR_ARG = 1,     /* bad argument: null pointer, negative size, unknown mode */
    TT_ERR_SHAPE = 2,   /* inconsistent TT shape: p1 p2 p3 < E, q1 q2 q3 != D, rank <= 0, limits */
    TT_ERR_INDEX = 3,   /* device found an index outside [0, E) */
    TT_ERR_CUDA = 4,    /* a CUDA runtime call failed */
    TT_ERR_STATE = 5,   /* call out of order, e.g. backward without a forward */
    TT_ERR_TIMEOUT = 6, /* a bounded device wait gave up */
    TT_ERR_NOMEM = 7,   /* device workspace allocation failed */
    TT_ERR_BOUNDS = 8   /* debug build only (libttemb_debug.so): an internal index left its bound */
} tt_status;

typedef enum { TT_POOL_SUM = 0, TT_POOL_MEAN = 1 } tt_pool;

/* What tt_emb_backward does with the gradient g of each element of every
 * touched core slice (FBTT README, "Parameters": sparse, optimizer,
 * learning_rate, eps; "Fused Kernel"). */
typedef enum {
    TT_OPT_SGD = 0,     /* sparse=True, SGD:     G -= lr g                                   */
    TT_OPT_ADAGRAD = 1, /* sparse=True, Adagrad: s += g^2; G -= lr g / (sqrt(s) + eps)       */
    TT_OPT_GRAD = 2     /* sparse=False: the gradient is written out, the cores stay as they are */
} tt_optim;

/* Limits checked by the create calls. */
#define TT_MAX_P 1048576 /* each p_k */
#define TT_MAX_Q 64      /* each q_k */
#define TT_MAX_RANK 128  /* each r_k */
#define TT_MAX_D 256     /* q1 q2 q3 */

/* One table of a table-batched handle (FBTT README, "TableBatchedTTEmbeddingBag"). */
typedef struct {
    int64_t num_embeddings; /* E: rows of this table */
    int64_t p[3];           /* row factorisation, p1 p2 p3 >= E (FBTT README, "Parameters": tt_p_shapes) */
    int32_t q[3];           /* column factorisation, q1 q2 q3 = D (tt_q_shapes) */
    int32_t ranks[2];       /* r1, r2 (tt_ranks) */
    float* cores_dev[3];    /* caller-owned, 16-byte aligned device cores, updated in place by tt_emb_backward */
} tt_table_desc;

/*
 * Create a single-table handle.  FBTT README, "Parameters" (num_embeddings,
 * tt_p_shapes, tt_q_shapes, tt_ranks).  cores_dev[k] must hold
 * p_k * r_{k-1} * q_k * r_k floats and be 16-byte aligned (the kernels read
 * the cores as float4; a fresh cudaMalloc or torch allocation always is).
 * The handle keeps the core pointers (not
 * the data); the caller keeps the cores alive while the handle is used.
 * Device memory for the handle's fixed tables is allocated on the current
 * CUDA device, which every later call on the handle must also use.
 * Returns TT_ERR_ARG (null out/cores, misaligned cores), TT_ERR_SHAPE (see
 * limits above).
 */
tt_status tt_emb_create(int64_t num_embeddings, const int64_t p[3], const int32_t q[3],
                        const int32_t ranks[2], float* const cores_dev[3], tt_emb** out);

/*
 * Create a table-batched handle over num_tables >= 1 tables that share D
 * (FBTT README, "TableBatchedTTEmbeddingBag": many tables in one call; unlike
 * the README's version, the tables may differ in E, p, q and ranks).  Bags of
 * a batched call are ordered table-major: bag g = t * B + b is sample b of
 * table t, and its indices are row ids of table t.
 */
tt_status tt_emb_batch_create(int32_t num_tables, const tt_table_desc* descs, tt_emb** out);

/* Release the handle's device memory (not the caller's cores).  NULL is a no-op. */
void tt_emb_destroy(tt_emb* h);

/*
 * Size the handle's workspace for up to max_nnz lookups and max_bags bags, so
 * that later forward/backward calls within those sizes allocate nothing (and
 * may be captured in a CUDA graph).  Forward calls beyond the reserved sizes
 * grow the workspace themselves.
 */
tt_status tt_emb_reserve(tt_emb* h, int64_t max_nnz, int64_t max_bags);

/*
 * Forward pass (FBTT README, "How FBTT-Embedding works": forward(input,
 * offsets); the pooling of PyTorch's EmbeddingBag).
 *   indices_dev          int64 [nnz]          row ids (of the bag's table)
 *   offsets_dev          int64 [num_bags + 1] CSR bag boundaries
 *   per_sample_weights   float [nnz] or NULL   (NULL: every weight is 1)
 *   mode                 TT_POOL_SUM: out[g] = sum_n w_n row_n
 *                        TT_POOL_MEAN: out[g] = (1/L_g) sum_n w_n row_n, L_g = bag length
 *   out_dev              float [num_bags][D], written completely (empty bag: zeros)
 * num_bags must be a multiple of the handle's table count.  The decoded
 * lookups, their grouping and the partial products G1[i1] G2[i2] are kept in
 * the handle for the next tt_emb_backward().  Asynchronous on `stream`.
 * Returns TT_ERR_ARG (null pointers with nnz > 0, negative sizes, bad mode,
 * num_bags not a multiple of the table count), TT_ERR_NOMEM, TT_ERR_CUDA.
 */
tt_status tt_emb_forward(tt_emb* h, const int64_t* indices_dev, int64_t nnz,
                         const int64_t* offsets_dev, int64_t num_bags,
                         const float* per_sample_weights_dev, tt_pool mode, float* out_dev,
                         tt_stream stream);

/*
 * Backward pass fused with SGD (FBTT README, "Fused Kernel", sparse=True with
 * OptimType.SGD): for L = sum_g <out[g], grad_out[g]> of the most recent
 * forward pass on this handle, every touched slice becomes
 * G_k[s] - lr * dL/dG_k[s], all gradients taken at the pre-update cores;
 * no gradient is returned.  grad_out_dev is float [num_bags][D] of that
 * forward pass.  Consumes the saved forward state: a second backward without
 * a new forward returns TT_ERR_STATE.  If the forward pass recorded a device
 * error, no core is changed.  Asynchronous on `stream`.
 */
tt_status tt_emb_backward(tt_emb* h, const float* grad_out_dev, float lr, tt_stream stream);

/*
 * Choose the update that tt_emb_backward applies (default TT_OPT_SGD; the
 * tt_emb_backward description above is the SGD case).  FBTT README,
 * "Parameters": sparse selects between the fused update and returning the
 * core gradients to an external optimizer; optimizer and eps configure the
 * fused update.  No page fixes the Adagrad variant: this is element-wise
 * Adagrad with one accumulator per core element, lr_decay and weight decay 0.
 *   optim  TT_OPT_SGD, TT_OPT_ADAGRAD or TT_OPT_GRAD
 *   eps    Adagrad denominator term, finite and >= 0 (ignored otherwise)
 *   aux    3 * num_tables caller-owned device pointers, table-major
 *          (aux[3 t + k] belongs to core k of table t), each with the shape of
 *          that core, 16-byte aligned; NULL for TT_OPT_SGD.
 *            TT_OPT_ADAGRAD: the accumulators s, read and updated in place
 *              (a new run starts them at 0, or at an initial value >= 0);
 *            TT_OPT_GRAD: every tt_emb_backward overwrites the whole buffer
 *              with dL/dG_k (zeros for untouched slices).
 * The handle keeps the pointers, which must stay valid while it is used.
 * Synchronous (copies the handle's device tables); not for stream capture.
 * Returns TT_ERR_ARG (null handle, unknown optim, bad eps, null or misaligned
 * aux), TT_ERR_CUDA.
 */
tt_status tt_emb_set_optimizer(tt_emb* h, int32_t optim, float eps, float* const* aux);

/*
 * Update from summed gradients: the data-parallel step.  Bags are independent
 * in the forward pass and every core gradient is a sum over bags, so ranks that
 * hold disjoint shares of a batch's bags and identical cores can each run
 * tt_emb_forward + tt_emb_backward with TT_OPT_GRAD on their share, sum the
 * gradient buffers over the ranks (one all-reduce, outside this library), and
 * then apply the same update on every rank with this call; the cores then equal
 * those of one fused step over the whole batch, up to the order of summation.
 * The update rules are those of tt_emb_set_optimizer (FBTT README,
 * "Parameters": optimizer, learning_rate, eps; "Fused Kernel").
 *   optim      TT_OPT_SGD (G -= lr g) or TT_OPT_ADAGRAD (s += g^2;
 *              G -= lr g / (sqrt(s) + eps))
 *   grads_dev  3 * num_tables caller-owned device pointers (table-major, each
 *              shaped like its core, 16-byte aligned): the summed gradients
 *   state_dev  3 * num_tables Adagrad accumulators (same layout), updated in
 *              place; NULL for TT_OPT_SGD
 * An element whose summed gradient is exactly 0 keeps its bits (as every
 * element of an untouched slice does in the fused step).  An exact-copy
 * hot-row cache sees the changed slices as stale.  Allocates nothing;
 * asynchronous on `stream`.  Returns TT_ERR_ARG (null or misaligned
 * pointers, unknown optim, bad eps), TT_ERR_STATE (trainable cache rows,
 * whose gradients this call does not carry), TT_ERR_CUDA.
 */
tt_status tt_emb_apply_gradients(tt_emb* h, int32_t optim, float lr, float eps, float* const* grads_dev,
                                 float* const* state_dev, tt_stream stream);

/*
 * Expand rows [row0, row0 + nrows) of table `table` (0 for a single-table
 * handle) to a dense float [nrows][D] block (FBTT README,
 * "TableBatchedTTEmbeddingBag": expanding to full weight).  Row i of the table
 * is G1[i1] G2[i2] G3[i3] with i = i1 p2 p3 + i2 p3 + i3, read from the cores
 * as they are when the kernel runs.  out_dev is caller-owned, nrows * D
 * floats.  Asynchronous on `stream`.  Returns TT_ERR_ARG (null handle, null
 * out with nrows > 0, table out of range, rows outside [0, E)), TT_ERR_CUDA.
 */
tt_status tt_emb_full_weight(tt_emb* h, int32_t table, int64_t row0, int64_t nrows, float* out_dev,
                             tt_stream stream);

/*
 * Hot-row cache (FBTT README, "Software Cache"): decompress the n rows of
 * table 0 listed in rows_dev (n <= 2^29 int64 rows, distinct, within [0, E)) into a
 * device-resident fp32 cache, slot i holding the i-th smallest row (rows are
 * found through a hash index).  By default the cached rows are exact copies:
 * later forward passes read a cached row instead of contracting it, as long as
 * its three core slices have not changed since it was filled; a backward pass
 * marks the slices it updated and the next forward pass recomputes a stale row
 * (one lookup per row) and writes it back into the cache.  Results are the same
 * as without a cache.  With tt_emb_cache_set_trainable the rows are parameters
 * of their own, initialised here from the cores.  Replaces any previous cache
 * content; a forward pass made with the previous cache can no longer be
 * followed by a backward pass (TT_ERR_STATE) when its rows were trainable.
 * Synchronous.  Returns TT_ERR_ARG (bad n, rows, or a null pointer),
 * TT_ERR_STATE (a table-batched handle), TT_ERR_NOMEM, TT_ERR_CUDA.
 */
tt_status tt_emb_cache_populate(tt_emb* h, const int64_t* rows_dev, int64_t n, tt_stream stream);

/* Drop the cache and free its memory (also the LFU policy's cache; the access
 * counts stay).  Returns TT_ERR_ARG for a null handle. */
tt_status tt_emb_cache_disable(tt_emb* h);

/*
 * LFU cache policy (FBTT README, "Parameters": use_cache, cache_size,
 * hashtbl_size; "Software Cache": access frequencies are counted in an
 * open-addressing hash table during forward propagation, the cache is a
 * 32-way set-associative least-frequently-used cache, and it changes only
 * when it is populated, with values initialised from the TT cores).
 * Single-table handles only (TT_ERR_STATE otherwise).
 *
 * tt_emb_lfu_enable: allocate a frequency table of hashtbl_size entries (a
 *   power of two, 32 .. 2^30) and size the cache at cache_size rows rounded up
 *   to a multiple of 32 (cache_size / 32 sets of 32 ways).  From then on every
 *   forward pass counts each lookup's row: hash h = SplitMix64(row) (the first
 *   output of a SplitMix64 generator seeded with row), entry h mod hashtbl_size,
 *   linear probing over at most 64 entries; a row that finds no free or
 *   matching entry there is not counted.  Counting uses integer atomics, so
 *   the counts do not depend on the order of the lookups while the table has
 *   room.  Replaces any previous frequency table (counts start at 0).
 * tt_emb_lfu_populate: rebuild the cache from the counts: set k (k =
 *   (h >> 32) mod sets) holds the 32 most frequently counted rows whose hash
 *   maps to k (ties: the smaller row id); each cached value is computed from
 *   the cores.  By default cached rows are exact copies of TT rows: gradients
 *   go to the cores and a row whose slices change is recomputed on its next
 *   hit, so results equal the no-cache results.  With
 *   tt_emb_cache_set_trainable the cached rows are parameters of their own
 *   (see there).  Synchronous.
 * tt_emb_lfu_read: copy the counted (row, count) pairs, sorted by row, into
 *   caller-owned host arrays of cap entries; *n_out = number of pairs.
 * tt_emb_lfu_cached_rows: copy the cache's rows per slot (slot = set * 32 +
 *   way, -1 = empty way; or the sorted rows of tt_emb_cache_populate) into a
 *   host array of cap entries; *n_out = number of slots.  Synchronous.
 * tt_emb_lfu_disable: stop counting and free the frequency table.
 * Return TT_ERR_ARG (bad sizes, null pointers), TT_ERR_STATE (batched handle;
 * populate or read before enable), TT_ERR_NOMEM, TT_ERR_CUDA.
 */
tt_status tt_emb_lfu_enable(tt_emb* h, int64_t cache_size, int64_t hashtbl_size);
tt_status tt_emb_lfu_populate(tt_emb* h, tt_stream stream);
tt_status tt_emb_lfu_read(tt_emb* h, int64_t* rows_host, uint32_t* counts_host, int64_t cap, int64_t* n_out);
tt_status tt_emb_lfu_cached_rows(tt_emb* h, int64_t* rows_host, int64_t cap, int64_t* n_out);
tt_status tt_emb_lfu_disable(tt_emb* h);

/*
 * Trainable cache rows (FBTT README, "Parameters": sparse, where backward
 * gives the gradient w.r.t. the TT cores or the cache; "Software Cache":
 * cached rows are loaded without decompressing them).  Single-table handles
 * only (TT_ERR_STATE otherwise).
 *
 * tt_emb_cache_set_trainable(h, 1): from the next forward pass on, a lookup
 *   whose row is cached (a hit) reads the cached value instead of its TT row,
 *   and backward gives the hit's gradient to the cached value and none to the
 *   cores: the gradient of cached value [slot][j] is the sum over the hits of
 *   that slot of (the lookup's pooling scale: weight, divided by the bag
 *   length in mean mode) x grad_out[bag][j].  The sum is taken in 64-bit fixed
 *   point with integer atomics, so it does not depend on the order of the
 *   hits (each term, the fp32 product, is rounded to a step of 2^-S with
 *   |sum| < 2^62, S set by max|grad_out| x max|hit scale| and the lookup
 *   count).  The optimizer of
 *   tt_emb_set_optimizer then updates the cached values that some hit touched
 *   (SGD; Adagrad with its own state per cached value, zero at populate; or
 *   TT_OPT_GRAD, which keeps the gradient for tt_emb_cache_read and gives
 *   untouched values 0); misses train the cores as before.  Hits take no part
 *   in the TT contractions or their grouping: a core slice that only hits use
 *   is not touched.  The cache state (installed now or later by a populate
 *   call) is initialised from the cores.  (h, 0): back to exact-copy rows,
 *   recomputed from the cores now.  Synchronous.
 * tt_emb_cache_read: copy the cached values ([slots][D] fp32, slot order of
 *   tt_emb_lfu_cached_rows) into vals_dev and, trainable mode only, the last
 *   gradients of TT_OPT_GRAD into grads_dev (caller-owned device buffers; either
 *   may be NULL).  Stream-ordered.
 * tt_emb_cache_write: overwrite the cached values from vals_dev (same layout;
 *   trainable mode only: an external optimizer's step on the values after
 *   TT_OPT_GRAD).  Stream-ordered.
 * Return TT_ERR_ARG, TT_ERR_STATE (batched handle; grads_dev or a write
 * outside trainable mode), TT_ERR_NOMEM, TT_ERR_CUDA.
 */
tt_status tt_emb_cache_set_trainable(tt_emb* h, int32_t trainable, tt_stream stream);
tt_status tt_emb_cache_read(tt_emb* h, float* vals_dev, float* grads_dev, tt_stream stream);
tt_status tt_emb_cache_write(tt_emb* h, const float* vals_dev, tt_stream stream);

/*
 * Copy the decode of the most recent forward pass: for every lookup its
 * table, its slice indices (i1, i2, i3) and its bag.  Each *_dev is a
 * caller-owned int32 [nnz] device buffer; any may be NULL.  For checks.
 */
tt_status tt_emb_get_decoded(tt_emb* h, int32_t* table_dev, int32_t* i1_dev, int32_t* i2_dev,
                             int32_t* i3_dev, int32_t* bag_dev, tt_stream stream);

/*
 * Wait for the handle's queued work, then return and clear the sticky device
 * error (TT_ERR_INDEX, TT_ERR_ARG for malformed offsets, TT_ERR_TIMEOUT) or
 * TT_OK.  Returns TT_ERR_CUDA if the wait itself fails.
 */
tt_status tt_emb_get_last_error(tt_emb* h);

/*
 * Stage timing: when enabled, each forward/backward records a CUDA event
 * after each of its kernels on the call's stream.  tt_emb_stage_times()
 * waits for the last call and writes up to cap per-kernel durations in
 * milliseconds (kernel order of that call) with their names; returns the
 * number of kernels the call launched, or -1 on error.
 */
tt_status tt_emb_set_stage_timing(tt_emb* h, int enable);
int tt_emb_stage_times(tt_emb* h, int which /* 0 forward, 1 backward */, float* ms, const char** names,
                       int cap);

/* Kernels launched by the most recent forward (which = 0) or backward (1). */
int tt_emb_last_launch_count(tt_emb* h, int which);

/*
 * Bound of the handle's device waits.  The pages have no counterpart: the
 * tensor-core kernels wait for their own MMAs and for the bulk copies of their
 * G2 slices on mbarriers, at most `polls` polls (default 2^24, far longer than
 * any MMA batch or copy).  A wait that gives up records TT_ERR_TIMEOUT (read by
 * tt_emb_get_last_error), issues no further MMA, waits with the default bound
 * for the MMAs or copies already in flight and frees its tensor memory; the
 * call's results are then undefined and a following backward changes no core.  polls = 0 makes every such wait give up at once
 * (a test of that path).  Takes effect from the next call.  Returns
 * TT_ERR_ARG for a null handle.
 */
tt_status tt_emb_set_wait_limit(tt_emb* h, uint32_t polls);

/*
 * Forward pass that allocates no device memory.  The pages have no
 * counterpart: this entry point exists for callers that cannot call
 * cudaMalloc -- code running under a memory manager that owns all device
 * memory (a framework's caching allocator, a serving runtime with a fixed
 * budget), and code that must not synchronize the device or that runs while a
 * stream is captured into a CUDA graph.
 *
 * It computes what tt_emb_forward() computes for one table, without a handle:
 * the arguments mean what they mean for tt_emb_create() and tt_emb_forward()
 * (cores_dev are only read), and the caller owns every buffer.  err_dev, if
 * not NULL, is a caller-owned device int32 into which the kernel ORs 1 for an
 * index outside [0, E) (that lookup contributes nothing) and 2 for malformed
 * offsets; the caller clears it.  The only scratch is a static device array of
 * TT_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until the
 * process exits; one partial product of q1 q2 r2 floats per warp must fit in
 * it (TT_ERR_SHAPE otherwise).  Calls share that array, so calls whose work
 * overlaps on the GPU (unordered streams) race and give wrong results.  The
 * first call on a device looks up the array's device address (a CUDA runtime
 * call); make that first call before any stream capture.  Calls no cudaMalloc,
 * cudaFree or allocating library routine.  Asynchronous on `stream`.
 */
#define TT_NOALLOC_SCRATCH_BYTES (8 * 1024 * 1024)
tt_status tt_emb_forward_noalloc(int64_t num_embeddings, const int64_t p[3], const int32_t q[3],
                                 const int32_t ranks[2], const float* const cores_dev[3],
                                 const int64_t* indices_dev, int64_t nnz, const int64_t* offsets_dev,
                                 int64_t num_bags, const float* per_sample_weights_dev, tt_pool mode,
                                 float* out_dev, int32_t* err_dev, tt_stream stream);

/* Static description of a status code; never NULL. */
const char* tt_emb_status_string(tt_status s);

#ifdef __cplusplus
}
#endif

#endif /* TT_EMB_H */
