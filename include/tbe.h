/*
 * tbe.h: C ABI of the GB300 (sm_103a) table-batched embedding library.
 *
 * A table-batched embedding (TBE) holds T embedding tables and, in one call,
 * looks up and pools a batch of sparse indices across all of them (forward),
 * then scatters the upstream gradient back to the looked-up rows with exactly
 * one optimizer update per touched (table, row) (backward).
 *
 * Sources (web pages on FBTriton table-batched embeddings):
 *  - "Optimizing Recommendation Systems with FBTriton Table Batched
 *    Embeddings", "Implementation Guide: Integrating TBE": the forward call
 *    takes the tables, a flat index list and an offsets list (CSR layout).
 *  - "FBTriton Rewrites Table Batched Embedding", "Responsibilities of the
 *    forward and backward passes": gather + aggregate per sample; scatter the
 *    upstream gradient back and accumulate repeated rows.
 *  - kimbodo "What Happened": pooling across tables in one launch, per-sample
 *    weights, higher-precision accumulation, a histogram + tensor-core path
 *    for eligible small tables; backward grouped by (table, row) with one
 *    optimizer update per row, a streaming path for short runs and gradient
 *    accumulation for runs of at least 256 lookups.
 *  - kimbodo "Kimbodo Engineering Perspective": transpose, sort and
 *    run-length encoding are the backward's preparation steps, and can be run
 *    ahead of time (during forward).
 *
 * Conventions for every call below
 *  - Pointers marked "device" are CUDA device pointers of the current device;
 *    pointers marked "host" are ordinary host memory.  The library never
 *    takes ownership of caller memory and never allocates per call; the only
 *    allocation is the small descriptor block that tbe_create makes.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call is asynchronous on that stream and performs no host
 *    synchronisation, except tbe_get_error.
 *  - A handle must not be used from two host threads, or on two streams whose
 *    work overlaps, at the same time.  It belongs to the device that was
 *    current at tbe_create; a call made while another device is current
 *    returns TBE_ERR_INVALID_ARG before anything is launched.
 *  - Return value: TBE_OK (0) or a negative TBE_ERR_* code.  Argument errors
 *    are reported synchronously and nothing is launched.  Problems only the
 *    GPU can see (an index out of range, malformed offsets, a bounded wait
 *    that ran out) raise a sticky flag in the handle that tbe_get_error reads.
 *
 * Batch layout (CSR, table-major): B bags per table; bag b of table t is flat
 * bag t*B+b, and its lookups are indices[offsets[t*B+b] .. offsets[t*B+b+1]).
 * `offsets` has T*B+1 entries, starts at 0, never decreases and ends at N.
 * indices and offsets share one integer type (int32 or int64).  An index
 * outside [0, rows_t) is skipped (contributes nothing, updates nothing) and
 * raises TBE_ERR_INDEX_OOB.
 *
 * Pooled output and upstream gradient: fp32 row-major [B, sum_t dim_t];
 * table t owns columns [Doff_t, Doff_t + dim_t), Doff_t = sum of the dims of
 * the tables before t.  Scale of lookup i: s_i = w_i (per-sample weight, or
 * 1 without weights), times 1/L for mean pooling (L = the bag's CSR length);
 * an empty bag pools to 0.
 *
 * Limits: at most 4096 tables; sum of all tables' rows < 2^32 - 1; every
 * table's rows < 2^31; N < 2^30 lookups per call; T*B < 2^31; dim in
 * [1, 4096].
 */
#ifndef TBE_GB300_H
#define TBE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ status codes */
#define TBE_OK 0
#define TBE_ERR_INVALID_ARG -1         /* null pointer, bad size, bad enum */
#define TBE_ERR_UNSUPPORTED -2         /* outside the limits listed above */
#define TBE_ERR_WORKSPACE_TOO_SMALL -3 /* workspace_bytes below the query */
#define TBE_ERR_CUDA -4                /* a CUDA runtime call failed */
#define TBE_ERR_INDEX_OOB -5           /* device: an index outside [0, rows) */
#define TBE_ERR_BAD_OFFSETS -6         /* device: offsets not 0..N monotone */
#define TBE_ERR_TIMEOUT -7             /* device: a bounded inter-CTA wait ran out */
#define TBE_ERR_NO_MEMORY -8           /* tbe_create could not allocate */

/* ------------------------------------------------------------------- enums */
typedef enum { TBE_F32 = 0, TBE_F16 = 1, TBE_BF16 = 2 } tbe_dtype;
typedef enum { TBE_I32 = 0, TBE_I64 = 1 } tbe_index_dtype;
typedef enum { TBE_POOL_SUM = 0, TBE_POOL_MEAN = 1 } tbe_pooling;
typedef enum { TBE_OPT_SGD = 1, TBE_OPT_ROWWISE_ADAGRAD = 2 } tbe_optimizer_kind;

/* tbe_create flags.  A "small table" has 16-bit rows (fp16 or bf16), a dim
 * that is a multiple of 16 in [16, 256], 16-byte aligned data and at most 512
 * rows (1024 with TBE_FLAG_FORCE_HISTOGRAM).
 *  - Backward of a small table (default): its lookups are not sorted; the
 *    table's whole gradient H^T . G is one tensor-core product (bf16 operands
 *    split three ways for fp32 accuracy, fp32 accumulation), then every
 *    touched row gets one optimizer step.  TBE_FLAG_SORTED_BACKWARD sends
 *    these tables through the sort and segment reduction like the others.
 *  - Forward of a small table: the gather, like every other table, unless
 *    TBE_FLAG_FORCE_HISTOGRAM, which pools it on the tensor cores as a
 *    per-bag histogram times the table (kimbodo "What Happened"), for the
 *    small tables of each dtype that fit one CTA's shared memory together.
 *    The default follows measurement: on 64 fp16 tables of 512 x 64 rows
 *    with 1..64 lookups per bag the gather was the faster of the two.
 *  - TBE_FLAG_NO_HISTOGRAM: neither tensor-core path.
 *  - TBE_FLAG_LENGTH_ORDER: the forward pools each table's bags in order of
 *    length (a per-table counting sort of the bag lengths, two extra kernels
 *    per call) whenever the table's bags are not all equally long, so the
 *    bags a CTA pools side by side take about the same time (the scheduling
 *    of bags onto warps by length that kimbodo "How We Would Implement It"
 *    calls load balancing).  Results are bit-identical either way.  Measured
 *    on 64 fp16 tables of 512 x 64 rows with 1..64 lookups per bag (four bags
 *    per warp): forward 1.38 -> 1.10 ms; on Poisson(20) or Poisson(40)
 *    lengths it was slower (the sort costs more than the balance gains), so
 *    it is off unless asked for.  The handle then keeps a device array of
 *    4*(T*B + 258*T) bytes, allocated (or grown) by the first forward call of
 *    a larger batch and freed by tbe_destroy. */
#define TBE_FLAG_NO_HISTOGRAM 0x1u    /* no tensor-core path (forward or backward) */
#define TBE_FLAG_FORCE_HISTOGRAM 0x2u /* histogram tensor-core forward for small tables */
#define TBE_FLAG_SORTED_BACKWARD 0x4u /* small tables too take the sorted backward */
#define TBE_FLAG_LENGTH_ORDER 0x8u    /* forward bags of varying length pooled in order of length */

/* One embedding table.  data: device, row-major rows x dim of dtype,
 * caller-owned, read by forward and updated in place by backward.  The
 * fastest path wants data 16-byte aligned and dim*sizeof(dtype) a multiple of
 * 16; other shapes run on a slower element-wise path. */
typedef struct {
    int64_t rows;
    int32_t dim;
    int32_t dtype; /* tbe_dtype */
    void* data;
} tbe_table;

/* Optimizer applied once per touched row by the backward calls.
 *  SGD:               w <- w - lr * g
 *  row-wise Adagrad:  m <- m + mean_j g_j^2 ;  w_j <- w_j - lr * g_j / (sqrt(m) + eps)
 * with g the row's summed gradient in fp32 and one round-to-nearest-even to
 * the table's dtype.  state: device fp32 [sum of rows], row r of table t at
 * rowbase_t + r (rowbase_t = rows of the tables before t), caller-owned,
 * zero-initialised by the caller; unused by SGD. */
typedef struct {
    int32_t kind; /* tbe_optimizer_kind */
    float lr;
    float eps;
    float* state;
} tbe_optimizer;

typedef struct tbe_handle tbe_handle;

/* Byte offsets, inside a backward workspace, of the arrays the preparation
 * step (transpose, sort, run-length encoding) leaves there.  All arrays are
 * uint32.  sorted_keys/sorted_vals: Ns entries (key = rowbase_t + row, or
 * sum-of-rows for a skipped lookup; val = the lookup's position in indices
 * when the batch has per-sample weights or mean pooling, else its flat bag
 * t*B + b), stably sorted by key (equal keys keep ascending positions, hence
 * ascending bags), where Ns = N, or, when the handle has dense-backward
 * tables (histogram tables, unless TBE_FLAG_SORTED_BACKWARD), the number of
 * lookups of the other tables: a dense table's lookups are not sorted.
 * uniq: the distinct keys ascending; runstart: the first sorted slot of each
 * (runstart[U] = Ns); num_unique: one entry, U. */
typedef struct {
    uint64_t sorted_keys;
    uint64_t sorted_vals;
    uint64_t uniq;
    uint64_t runstart;
    uint64_t num_unique;
    uint64_t total_bytes;
} tbe_ws_layout;

/* ------------------------------------------------------------------ handle */

/* Validates the table list and builds the device descriptor block (row
 * bases, column offsets, per-table lookup schedule).  Defining passages: the
 * operator holds the tables it pools ("Optimizing Recommendation Systems
 * with FBTriton Table Batched Embeddings", "Implementation Guide: Integrating
 * TBE": the call takes the embedding tables); the choice of the histogram
 * tensor-core path for eligible small tables is made here (kimbodo "What
 * Happened"; the pages give no eligibility rule, this library's is stated
 * under TBE_FLAG_*).  `tables`: host array
 * of num_tables entries (copied; the data pointers are kept).  pooling:
 * tbe_pooling.  flags: TBE_FLAG_*.  On success *out receives the handle.
 * Errors: INVALID_ARG (null/zero/negative sizes, bad enums), UNSUPPORTED
 * (limits), CUDA, NO_MEMORY. */
int tbe_create(const tbe_table* tables, int32_t num_tables, int32_t pooling, uint32_t flags,
               tbe_handle** out);

/* Frees the descriptor block.  The caller's memory is untouched.  Must not be
 * called while work that uses the handle may still run.  (Resource
 * management of this library; the pages have no counterpart.) */
void tbe_destroy(tbe_handle* h);

/* ----------------------------------------------------------------- forward */

/* Pooled lookup of all T*B bags in one pass (forward of the kimbodo "What
 * Happened" section; CSR call of the integration guide).
 *  indices: device [num_indices] of index_dtype; offsets: device [T*B+1];
 *  per_sample_weights: device fp32 [num_indices] or NULL;
 *  out: device fp32 [batch_size, sum of dims], fully overwritten.
 * Accumulation is fp32 for every table dtype. */
int tbe_forward(tbe_handle* h, const void* indices, const void* offsets, int32_t index_dtype,
                int64_t num_indices, int32_t batch_size, const float* per_sample_weights,
                float* out, void* stream);

/* ---------------------------------------------------------------- backward */

/* Bytes of device workspace the backward calls need for this batch shape:
 * the arrays of the backward's preparation steps (one key and one sort value
 * per lookup, and room for each lookup's bag and scale, which batches with
 * per-lookup scales use; the sort's ping-pong buffers and digit counts; distinct
 * keys and run starts; partial sums of the runs of at least 256 lookups), as
 * kimbodo "Kimbodo Engineering Perspective" (transpose, sort, run-length
 * encoding) and "What Happened" (separate accumulation for long runs) define
 * them.  0 for a null handle or a negative count. */
size_t tbe_backward_workspace_bytes(const tbe_handle* h, int64_t num_indices, int32_t batch_size);

/* Where the preparation step leaves its arrays inside the workspace (the
 * sorted keys and run-length encoding of kimbodo "Kimbodo Engineering
 * Perspective"), for tests and inspection. */
int tbe_backward_workspace_layout(const tbe_handle* h, int64_t num_indices, int32_t batch_size,
                                  tbe_ws_layout* out);

/* Backward preparation only (kimbodo "Kimbodo Engineering Perspective"):
 * transpose the batch into one (table,row) key per lookup, radix-sort the
 * keys stably, run-length encode them.  Results stay in `workspace` (device,
 * caller-owned, at least tbe_backward_workspace_bytes) for
 * tbe_backward_apply.  Depends only on indices, offsets and weights, so it
 * may run as soon as the batch is known, e.g. beside the forward pass. */
int tbe_backward_prepare(tbe_handle* h, const void* indices, const void* offsets,
                         int32_t index_dtype, int64_t num_indices, int32_t batch_size,
                         const float* per_sample_weights, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Forward and backward preparation of one batch, run side by side (kimbodo
 * "Kimbodo Engineering Perspective": moving transpose, sort and run-length
 * encoding into forward).  The forward pass is queued on `stream`, the
 * preparation on a high-priority second stream owned by the handle that
 * starts after the work already queued on `stream`; `stream` then waits for
 * the preparation, so anything queued on it afterwards (tbe_backward_apply)
 * sees both results.  Arguments and results as tbe_forward plus
 * tbe_backward_prepare; argument errors are reported before anything is
 * queued. */
int tbe_forward_prepare(tbe_handle* h, const void* indices, const void* offsets, int32_t index_dtype,
                        int64_t num_indices, int32_t batch_size, const float* per_sample_weights,
                        float* out, void* workspace, size_t workspace_bytes, void* stream);

/* Backward from a prepared workspace: per unique (table,row) sums
 * s_i * grad_out[bag_i, Doff_t : Doff_t+dim_t] in fp32 (runs of fewer than 256
 * lookups stream through one warp; longer runs are split into chunks of 256
 * to 1024 lookups, by batch size, whose partial sums are added in a fixed
 * order), then applies the optimizer once to that row.  grad_out: device
 * fp32 [batch_size, sum of dims].  num_indices and batch_size must equal the
 * prepare call's.  When
 * the handle's tables fall into more than one backward class (dtype x row
 * shape), the class kernels run on side streams owned by the handle that
 * start after the work already queued on `stream`, and `stream` waits for
 * all of them before its next work (a fork and join that stream capture
 * records as well). */
int tbe_backward_apply(tbe_handle* h, int64_t num_indices, int32_t batch_size,
                       const float* grad_out, const tbe_optimizer* opt, void* workspace,
                       size_t workspace_bytes, void* stream);

/* prepare + apply with SGD: the backward pass of "FBTriton Rewrites Table
 * Batched Embedding", "Responsibilities of the forward and backward passes"
 * (scatter the upstream gradient to the looked-up rows, accumulating repeated
 * rows) with kimbodo "What Happened"'s grouping by (table, row) and one
 * optimizer update per row.  The pages name no optimizer; SGD is the plain
 * w <- w - lr * g (no momentum, no weight decay).  Arguments as
 * tbe_backward_prepare and tbe_backward_apply. */
int tbe_backward_sgd(tbe_handle* h, const void* indices, const void* offsets, int32_t index_dtype,
                     int64_t num_indices, int32_t batch_size, const float* per_sample_weights,
                     const float* grad_out, float lr, void* workspace, size_t workspace_bytes,
                     void* stream);

/* prepare + apply with row-wise Adagrad (state as in tbe_optimizer): the same
 * backward pass as tbe_backward_sgd ("FBTriton Rewrites Table Batched
 * Embedding", "Responsibilities of the forward and backward passes"; kimbodo
 * "What Happened"), with the row-wise Adagrad step defined at tbe_optimizer.
 * The pages do not define row-wise Adagrad; that formula is this library's
 * reading (eps outside the root, the mean of g_j^2 added to the state). */
int tbe_backward_rowwise_adagrad(tbe_handle* h, const void* indices, const void* offsets,
                                 int32_t index_dtype, int64_t num_indices, int32_t batch_size,
                                 const float* per_sample_weights, const float* grad_out,
                                 float* state, float lr, float eps, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* Backward + SGD that allocates nothing.  The paper has no counterpart to
 * this call; it exists for callers that cannot call cudaMalloc when they run
 * the backward pass (their device memory is owned by another allocator, or
 * their rules forbid device allocation after set-up), so they cannot pass a
 * workspace.  Same arguments and result as tbe_backward_sgd, but the
 * workspace is a 32 MiB static device array inside the library:
 *  - a batch whose tbe_backward_workspace_bytes exceeds 32 MiB (33554432) is
 *    rejected with TBE_ERR_WORKSPACE_TOO_SMALL and nothing is launched;
 *  - the first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture;
 *  - every device that loads the library holds the array until exit;
 *  - all calls on a device share the array and it keeps the last call's
 *    contents (the call clears what must start at zero), so calls whose GPU
 *    work overlaps (other streams or host threads) race: order them.
 * The handle comes from tbe_create (called at set-up). */
int tbe_backward_sgd_noalloc(tbe_handle* h, const void* indices, const void* offsets,
                             int32_t index_dtype, int64_t num_indices, int32_t batch_size,
                             const float* per_sample_weights, const float* grad_out, float lr,
                             void* stream);

/* ----------------------------------------------- per-sample weight gradient */

/* Gradient of the loss with respect to each per-sample weight, for callers
 * that train the weights (kimbodo "What Happened": per-sample weights on the
 * generic path; the pages give no formula, this is the derivative of the
 * forward pass's definition):
 *   grad_weights[i] = (1/L if mean) * sum_j grad_out[b, Doff_t + j] * W_t[idx_i, j]
 * for lookup i of bag (t, b) of length L; 0 for a lookup whose index is out
 * of range (the forward pass skips it; reported as TBE_ERR_INDEX_OOB by
 * tbe_get_error).  fp32 products and sums for every table dtype.
 *  indices, offsets, index_dtype, num_indices, batch_size: the batch, as
 *    for tbe_forward (device, CSR, T*B+1 offsets);
 *  grad_out: device fp32 [batch_size, sum of dims], read only;
 *  grad_weights: device fp32 [num_indices], caller-owned, fully written
 *    when the offsets are well formed (a malformed bag is reported as
 *    TBE_ERR_BAD_OFFSETS by tbe_get_error and its entries are not written).
 * It reads the table rows as they are when it runs on `stream`: call it
 * before tbe_backward_apply (or the fused backward calls) updates them.
 * Errors: INVALID_ARG (null pointers, bad enums or sizes), UNSUPPORTED
 * (more than 2^26 bags), CUDA. */
int tbe_per_sample_weight_grad(tbe_handle* h, const void* indices, const void* offsets,
                               int32_t index_dtype, int64_t num_indices, int32_t batch_size,
                               const float* grad_out, float* grad_weights, void* stream);

/* ------------------------------------------------------------- diagnostics */

/* Synchronises `stream`, returns the first device-detected error since the
 * last call (TBE_ERR_TIMEOUT before TBE_ERR_BAD_OFFSETS before
 * TBE_ERR_INDEX_OOB) or TBE_OK, and clears it.  The pages define no error
 * reporting; this reports the conditions of the batch layout read from
 * "Optimizing Recommendation Systems with FBTriton Table Batched
 * Embeddings", "Implementation Guide: Integrating TBE" (offsets cut one flat
 * index list into bags, so they must rise from 0 to N; an index names a row
 * of its table), plus the bounded waits of the tensor-core kernels. */
int tbe_get_error(tbe_handle* h, void* stream);

/* Static description of a status code.  (Library plumbing; the pages have no
 * counterpart.) */
const char* tbe_strerror(int code);

/* The cudaError_t of the last CUDA call that failed in a tbe_* call of this
 * host thread (0 if none), for diagnosing TBE_ERR_CUDA. */
int tbe_last_cuda_error(void);

/* Per-table schedule chosen at create time, for tests and tuning:
 * out_path[t] = 0 gather path (vector), 1 gather path (element-wise),
 * 2 histogram tensor-core path (kimbodo "What Happened": eligible small
 * tables take the histogram path). */
int tbe_table_paths(const tbe_handle* h, int32_t* out_path);

/* Per-table backward schedule chosen at create time, for tests and tuning:
 * out_path[t] = 0 sorted (transpose, sort, segment reduction), 1 dense
 * tensor-core product H^T . G (small tables; see the flags above). */
int tbe_table_backward_paths(const tbe_handle* h, int32_t* out_path);

#ifdef __cplusplus
}
#endif

#endif /* TBE_GB300_H */
