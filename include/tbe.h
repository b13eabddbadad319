/*
 * tbe.h -- C ABI of the GB300 table-batched embedding (TBE) training hot path.
 *
 * The operation (FBTriton TBE redesign, accesspath.com, section "Backward
 * kernels: three paths by segment length", notation paragraph): T embedding
 * tables, table t with E_t rows of D elements; a batch of B bags per table,
 * bag (t,b) holding L_(t,b) row indices (L is the pooling factor).  Input is
 * KeyedJagged CSR (TorchEasyRec analysis, 39.107.221.112 article 1724244,
 * section 1 "KeyedJaggedTensor"): one `indices` array with every lookup of
 * every table concatenated, and `offsets[T*B+1]`, bag (t,b) being
 * indices[offsets[t*B+b] .. offsets[t*B+b+1]).  Tables are key-major: all
 * bags of table 0, then all bags of table 1, ...
 *
 *   forward:    out[b, t*D + d] = sum_{p in bag (t,b)} w_p * W_t[idx_p, d]
 *   backward:   for each unique (t,row) touched by the batch,
 *               g[d] = sum_{p touching it} w_p * grad_out[b(p), t*D + d],
 *               then exactly one exact-rowwise-Adagrad update of that row:
 *               m[row] += mean_d g[d]^2;  W[row,d] -= lr*g[d]/(sqrt(m[row])+eps)
 *
 * w_p is the per-sample weight (1 on unweighted tables).
 *
 * Conventions for every entry point
 *  - Ownership: the caller allocates and owns every buffer.  The library
 *    allocates nothing and frees nothing; all scratch memory comes from the
 *    caller's `workspace`.  The one exception is tbe_preprocess_static,
 *    whose scratch is a device array inside the library (see there).
 *  - Pointers named device are device memory; those named host are host
 *    memory read synchronously during the call.
 *  - Streams: every device operation is enqueued on `stream`; the calls
 *    return before the work completes and never synchronise the host.
 *  - Errors found on the host (null or misaligned pointers, unsupported
 *    sizes, too-small buffers) return a non-zero tbe_status before anything
 *    is enqueued.  Errors that depend on the data are reported in the
 *    caller's device status words (`dev_status`, TBE_STATUS_WORDS int32),
 *    to be read after the stream completes:
 *        dev_status[0]  += number of out-of-range indices seen by tbe_forward
 *                          (tbe_preprocess skips them without counting)
 *        dev_status[1]  |= TBE_FLAG_* bits
 *    The caller zeroes dev_status when it wants a fresh count.  No kernel
 *    traps, asserts or waits without bound.
 *  - Malformed offsets (the pages do not cover them): a bag (t,b) is well
 *    formed when 0 <= offsets[g] <= offsets[g+1] <= N (g = t*B+b).  A
 *    malformed bag is empty (zero output, no part in the backward).
 *    Lookups outside every well-formed bag (before offsets[0], after
 *    offsets[T*B], inside a malformed bag) are ignored by forward and
 *    backward.  When offsets decrease anywhere (a bag with end < start), two
 *    well-formed bags can both hold a lookup, and the batch gets no backward
 *    update at all; its forward still pools each well-formed bag over its
 *    own range.  Any of these, and offsets[0] != 0 or offsets[T*B] != N,
 *    sets TBE_FLAG_BAD_OFFSETS.
 *  - Threading: the functions are reentrant; calls on different streams
 *    must use different workspace and meta buffers.
 *  - Per-device state: the first call on a device looks up, once, its SM
 *    count, each kernel's resident blocks per SM and shared-memory limit,
 *    and (tbe_preprocess_static) the built-in scratch array's address, and
 *    keeps them for the life of the process.  A process that resets a
 *    device (cudaDeviceReset) must not call the library on it again.
 *  - CUDA graphs: the calls enqueue only kernels and event records, so a
 *    step can be captured; during capture the timing events of
 *    tbe_config.kernel_events become event-record nodes of the graph.
 */
#ifndef TBE_GB300_TBE_H
#define TBE_GB300_TBE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tbe_status {
    TBE_OK = 0,
    TBE_ERR_NULL_POINTER = 1,       /* a required pointer is NULL */
    TBE_ERR_INVALID_ARGUMENT = 2,   /* T, B, N, D out of range, table_offset not monotone,
                                       grad_out of 64 GB or more on the generic path, ... */
    TBE_ERR_UNSUPPORTED_DIM = 3,    /* D*sizeof(weight) not one of the supported row sizes */
    TBE_ERR_UNSUPPORTED_DTYPE = 4,
    TBE_ERR_MISALIGNED = 5,         /* a device pointer is not 16-byte aligned */
    TBE_ERR_KEY_RANGE = 6,          /* sum of E_t is 2^62 or more */
    TBE_ERR_BUFFER_TOO_SMALL = 7,   /* workspace or meta smaller than tbe_query_sizes says */
    TBE_ERR_META = 8,               /* meta not bound, or bound for another problem */
    TBE_ERR_HISTOGRAM_SHAPE = 9,    /* histogram path forced on a shape it does not cover */
    TBE_ERR_CUDA = 10,              /* a kernel launch failed (see cudaGetLastError) */
    TBE_ERR_SCRATCH_LIMIT = 11      /* batch too large for tbe_preprocess_static's scratch */
} tbe_status;

typedef enum tbe_dtype { TBE_F32 = 0, TBE_F16 = 1, TBE_BF16 = 2 } tbe_dtype;

/* dev_status[1] bits */
#define TBE_FLAG_BAD_OFFSETS   0x1  /* malformed offsets (see the conventions above) */
#define TBE_FLAG_FP16_OVERFLOW 0x2  /* |grad| > 65504 in the histogram path's FP16 hi/lo split */
#define TBE_FLAG_SORT_TIMEOUT  0x4  /* radix-sort look-back gave up waiting: sort output invalid */
#define TBE_FLAG_HIST_COUNT    0x8  /* a histogram count exceeded 2048 (not exact in FP16) */
#define TBE_FLAG_MMA_TIMEOUT   0x10 /* a tensor-core completion wait gave up: output invalid */
#define TBE_FLAG_COPY_TIMEOUT  0x20 /* a bulk-copy completion wait gave up: output invalid */
#define TBE_STATUS_WORDS 4

/* Where runs with SL >= sl_threshold are reduced (FBTriton TBE redesign,
 * "Backward kernels", paths 2 and 3). */
typedef enum tbe_long_run_mode {
    TBE_LONG_AUTO = 0,       /* = TBE_LONG_TWO_KERNEL: on GB300 the fused launch's per-chunk
                                fence and arrival round trip queue behind the gather's
                                DRAM misses and cost more than the extra launch */
    TBE_LONG_TWO_KERNEL = 1, /* grad_accum into the workspace + a separate apply kernel */
    TBE_LONG_FUSED = 2       /* one launch; the last-arriving chunk applies the update */
} tbe_long_run_mode;

/* Small-table histogram path (FBTriton TBE redesign, "Forward state reuse
 * and preprocessing" and decision checklist item 2). */
typedef enum tbe_hist_mode {
    TBE_HIST_AUTO = 0,   /* used when E_t <= 64, 64 <= D <= 128, D % 16 == 0, FP16
                            weights, no per-sample weights and N >= 64*T*B */
    TBE_HIST_OFF = 1,    /* always the generic gather path */
    TBE_HIST_FORCE = 2   /* histogram path whenever the shape is covered (any L) */
} tbe_hist_mode;

typedef struct tbe_config {
    int32_t sl_threshold;    /* runs with fewer lookups take the short-run kernel; default 256 */
    int32_t chunk;           /* lookups per chunk of a long run, 32..1024; default 256 */
    int32_t long_run_mode;   /* tbe_long_run_mode */
    int32_t hist_mode;       /* tbe_hist_mode */
    /* Optional timing hook: when kernel_events is non-NULL, the library
     * records kernel_events[2i] before and kernel_events[2i+1] after each of
     * its kernel launches on `stream`, for i = *kernel_events_used, +1, ...
     * up to n_kernel_events pairs, writes the kernel's static name to
     * kernel_names[i] when kernel_names is non-NULL, and advances
     * *kernel_events_used (host int, required with kernel_events), so
     * consecutive calls append. */
    cudaEvent_t *kernel_events;
    const char **kernel_names;
    int32_t n_kernel_events;
    int32_t *kernel_events_used;
    /* Width of the linearised keys: 0 = automatic (4 bytes while rows_total
     * < 2^31 - 1, else 8), 8 = 64-bit keys for any problem (the wide path
     * on small tables, e.g. to test it).  4 is accepted where 0 would pick it. */
    int32_t key_bytes;
} tbe_config;

/* Shape of one table when tables differ (TorchEasyRec analysis, section 1:
 * one fused lookup for all features of a KeyedJagged batch, whose embedding
 * sizes differ). */
typedef struct tbe_table_layout {
    int64_t weights_byte_offset;        /* first byte of the table's rows in `weights`;
                                           16-byte aligned, tables' regions disjoint */
    int32_t D;                          /* elements per row */
    int32_t dtype;                      /* tbe_dtype of its rows */
} tbe_table_layout;

/* The tables.  Uniform (layout == NULL): all T tables back to back in one
 * [rows_total, D] array of dtype.  Otherwise table t holds E_t rows of
 * layout[t].D elements of layout[t].dtype at byte layout[t].weights_byte_offset
 * of `weights`; D and dtype are then ignored.  Either way table t owns the
 * linearised rows [table_offset[t], table_offset[t+1]) (the keys of the batch
 * inversion and the indices of the momentum array). */
typedef struct tbe_tables {
    void *weights;                      /* device, 16-byte aligned */
    const int64_t *table_offset;        /* device, [T+1]: table t owns rows [off[t], off[t+1]) */
    const int64_t *table_offset_host;   /* host copy of the same [T+1] values */
    int32_t T;
    int32_t D;
    int32_t dtype;                      /* tbe_dtype */
    const tbe_table_layout *layout;     /* device [T] or NULL (uniform) */
    const tbe_table_layout *layout_host;/* host copy of the same [T] records */
} tbe_tables;

/* Where one table's bags and their output rows lie in a batch: its bags are
 * CSR bags bag_offset .. bag_offset + B - 1 (tables follow one another,
 * bag_offset[0] = 0), and bag b's pooled row (D_t floats) starts at
 * out[out_offset + b * out_stride]; grad_out has the same layout.  Variable
 * batch size per table (VBE, FBTriton TBE redesign, decision checklist item
 * 5) is a different B per table, its rows packed one after another
 * (out_offset = sum of earlier tables' B*D, out_stride = D); tables of
 * different D with one B use out_offset = sum of earlier tables' D and
 * out_stride = the sum of all D (rows of a [B, sum D] matrix). */
typedef struct tbe_bag_layout {
    int64_t bag_offset;
    int64_t B;
    int64_t out_offset;                 /* multiple of 4 */
    int64_t out_stride;                 /* multiple of 4 */
} tbe_bag_layout;

/* Element type of a batch's indices and offsets (decision checklist item 6:
 * int32 where the range allows, int64 otherwise; KeyedJagged tensors often
 * carry int64). */
typedef enum tbe_index_type { TBE_INDEX_I32 = 0, TBE_INDEX_I64 = 1 } tbe_index_type;

/* One batch in KeyedJagged CSR form. */
typedef struct tbe_batch {
    const void *indices;                /* device, [N] of index_type; row index within its table */
    const void *offsets;                /* device, [T*B+1] of index_type; offsets[0] = 0,
                                           offsets[T*B] = N */
    int64_t N;                          /* number of lookups, 0 <= N < 2^30 */
    int64_t B;                          /* bags per table */
    const float *per_sample_weights;    /* device, [N] or NULL (unweighted) */
    const uint8_t *weighted_tables;     /* device, [T] or NULL: nonzero = table uses the weights;
                                           NULL with weights given = every table weighted */
    int32_t index_type;                 /* tbe_index_type of indices and offsets */
    /* NULL: every table has B bags, bag (t,b) is CSR bag t*B+b and its row is
     * out[b, t*D .. t*D+D) of a [B, T*D] out.  Required when the tables have
     * a layout; B is then ignored. */
    const tbe_bag_layout *bag_layout;      /* device [T] or NULL */
    const tbe_bag_layout *bag_layout_host; /* host copy */
    int64_t out_size;                   /* with bag_layout: floats in out and in grad_out */
} tbe_batch;

/*
 * Batch-inversion metadata (FBTriton TBE redesign, "Forward state reuse and
 * preprocessing" and "transpose_embedding_input"): produced by tbe_forward
 * (when given a meta) or tbe_preprocess, consumed by the backward.  Bind it to
 * a caller device buffer with tbe_meta_bind; the fields are device pointers
 * into that buffer plus the problem it was bound for, and are read-only to
 * the caller.  Linearised keys are uint32 (key_bytes = 4) when rows_total
 * is below 2^31 - 1, uint64 (key_bytes = 8) otherwise (decision checklist
 * item 6: int32 keys while the linearised range fits).  After a generic-path
 * forward/preprocess, on the device:
 *   sorted_keys[0..N)  linearised keys table_offset[t]+idx in ascending order,
 *                      out-of-range lookups and lookups outside every
 *                      well-formed bag last with key = rows_total
 *   sorted_vals[0..N)  payload in the same (stable) order: the bag index b
 *                      within its table when the batch is unweighted, else
 *                      the lookup position p (bag_of[p] then gives t*B+b)
 *   unique_keys[0..U), seg_off[0..U]  run r = positions [seg_off[r], seg_off[r+1])
 *   counters[0] = U (unique rows), counters[1] = N' (in-range lookups),
 *   counters[2] = long runs, counters[3] = chunks of long runs
 * After a histogram-path forward/preprocess: hist[(t*B+b)*64 + e] holds the
 * FP16 count of lookups of row e in bag (t,b).
 */
typedef struct tbe_meta {
    int64_t bound_N, bound_B;
    int32_t bound_T, path;              /* path: 1 = generic, 2 = histogram */
    int32_t payload_is_pos, key_bits;
    int64_t rows_total;
    int32_t key_bytes;                  /* 4 (uint32 keys) or 8 (uint64 keys) */
    int32_t index_type;                 /* the batch's tbe_index_type */
    void *sorted_keys;                  /* key arrays hold key_bytes per key */
    uint32_t *sorted_vals;
    void *keys_a;
    uint32_t *vals_a;
    void *keys_b;
    uint32_t *vals_b;
    int32_t *bag_of;
    void *unique_keys;
    int32_t *seg_off;
    int32_t *counters;
    int32_t *long_run;                  /* [max_long] run id of long run l */
    int32_t *long_chunk_base;           /* [max_long] first chunk slot of long run l */
    int32_t *chunk_order;               /* [max_chunks] chunk slot taken c-th by the long-run
                                           kernel: slots grouped by table and batch window of
                                           their first lookup's bag (B >= 4096 and T <= 4096);
                                           scratch otherwise, and slot c is taken c-th */
    int32_t *arrive;                    /* [max_long] arrival counters of the fused long-run path */
    int32_t *chunk_desc;                /* [max_chunks][8] per chunk slot: first and end sorted
                                           position, key (low and high 32 bits), long run, first
                                           slot of the run, chunks of the run, window key */
    uint16_t *hist;
    size_t bytes;
} tbe_meta;

/* Fill *cfg with the defaults (SL threshold 256, chunk 256, AUTO modes, no events). */
void tbe_config_default(tbe_config *cfg);

/*
 * Device memory the caller must provide for this problem: the meta buffer
 * (bound with tbe_meta_bind) and the scratch workspace passed to every call.
 * One workspace may serve forward, preprocess and backward in turn on one
 * stream.  Returns TBE_OK or an argument error for an unsupported problem.
 */
tbe_status tbe_query_sizes(const tbe_tables *tables, const tbe_batch *batch,
                           const tbe_config *cfg, size_t *meta_bytes, size_t *workspace_bytes);

/* The two sizes of tbe_query_sizes one at a time (host only): bytes of the
 * meta buffer and of the workspace, or 0 when the problem is rejected (the
 * status then comes from tbe_query_sizes). */
size_t tbe_workspace_bytes(const tbe_tables *tables, const tbe_batch *batch, const tbe_config *cfg);
size_t tbe_meta_bytes(const tbe_tables *tables, const tbe_batch *batch, const tbe_config *cfg);

/* Carve `meta` out of device_buf (>= meta_bytes, 256-byte aligned).  Host only. */
tbe_status tbe_meta_bind(tbe_meta *meta, void *device_buf, size_t bytes,
                         const tbe_tables *tables, const tbe_batch *batch, const tbe_config *cfg);

/*
 * Forward pooled lookup with fused bounds check (decision checklist item 5):
 * writes out[B, T*D] (device, float32; every element written, empty bags give
 * 0), or, with a bag layout, each bag's row where the layout puts it.  Out-of-range indices contribute nothing and are counted into
 * dev_status[0].  Accumulation is FP32 for FP16/BF16 tables and FP64 for FP32
 * tables (decision checklist item 1).
 * When `meta` is non-NULL the batch inversion also runs here ("Forward state
 * reuse and preprocessing": sort and RLE moved into forward) and the
 * backward reuses it; on the histogram path the forward saves its counts.
 */
tbe_status tbe_forward(const tbe_tables *tables, const tbe_batch *batch, float *out,
                       tbe_meta *meta, void *workspace, size_t workspace_bytes,
                       int32_t *dev_status, const tbe_config *cfg, cudaStream_t stream);

/*
 * Batch inversion alone (the pages' default placement, at the start of the
 * backward): linearise (t,idx) to int32 keys (decision checklist item 6),
 * stable radix sort, run-length encode, route runs by segment length.  On
 * the histogram path: build the per-bag counts.  Fills `meta`.
 */
tbe_status tbe_preprocess(const tbe_tables *tables, const tbe_batch *batch, tbe_meta *meta,
                          void *workspace, size_t workspace_bytes, int32_t *dev_status,
                          const tbe_config *cfg, cudaStream_t stream);

/*
 * Backward with the fused exact rowwise Adagrad update ("Backward kernels";
 * TorchEasyRec analysis section 4, fused optimizer).  grad_out is the
 * gradient of `out` (device, float32, laid out as out).  Updates tables->weights and
 * momentum (device, float32 [rows_total]) in place, once per touched row;
 * rows no in-range lookup touches are not written.  Runs with SL < 256 take
 * the short-run kernel; longer runs are reduced in 256-lookup chunks (two
 * kernels or one fused launch, cfg->long_run_mode).  Weighted tables scale
 * each gradient row by its per-sample weight before accumulation.
 * `batch` must be the one `meta` was filled from.  On the generic path
 * grad_out must be smaller than 64 GB (B*T*D < 2^34 elements): gradient-row
 * offsets are staged as 32-bit counts of 16-byte vectors.
 */
tbe_status tbe_backward_rowwise_adagrad(const tbe_tables *tables, const tbe_batch *batch,
                                        float *momentum, const float *grad_out,
                                        const tbe_meta *meta, float lr, float eps,
                                        void *workspace, size_t workspace_bytes,
                                        int32_t *dev_status, const tbe_config *cfg,
                                        cudaStream_t stream);

/*
 * The batch inversion of tbe_preprocess without a caller workspace.  The pages
 * have no counterpart to this call; it is an addition of this library.
 *
 * For callers that cannot allocate device memory where they run the batch
 * inversion: code running inside a device-memory allocator or pool callback
 * (allocating there would recurse into it), plug-ins that a host framework
 * hands only fixed input and output buffers, and services that must not grow
 * their device footprint after start-up.  It allocates nothing: no
 * cudaMalloc, cudaFree or allocating library call.  The caller still passes
 * the inputs (tables, batch), the output `meta` (bound with tbe_meta_bind)
 * and `dev_status`; the scratch of the sort and the run-length encoding is a
 * 8 MiB + 64 KiB device array inside this library, which every GPU that loads
 * the library holds until the process exits.
 *
 * Limit: batch->N <= 4,194,304 (2^22) lookups; a larger batch returns
 * TBE_ERR_SCRATCH_LIMIT before anything is enqueued.  Results equal
 * tbe_preprocess's.
 *
 * The first call on each device looks up the array's address on that device
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  All calls on a device share the one array and
 * it keeps the last call's contents (each call re-initialises what it reads):
 * calls whose work can overlap on the GPU -- on different streams without an
 * order between them -- race on it and corrupt each other's results, so order
 * them on one stream.
 */
tbe_status tbe_preprocess_static(const tbe_tables *tables, const tbe_batch *batch, tbe_meta *meta,
                                 int32_t *dev_status, const tbe_config *cfg, cudaStream_t stream);

/*
 * Self-test of the failure detection of device waits (no counterpart on the
 * pages).  Every device-side wait of this library -- the radix sort's
 * look-back on earlier tiles, the mbarrier waits of the bulk-copy rings and
 * of the tensor-core path -- gives up after one second, sets a dev_status[1]
 * flag and returns, so a wait that can never end costs a second and an error
 * status instead of a hung GPU.  This call runs one such wait on a condition
 * that nothing will ever satisfy, so the caller can check that the limit
 * works and that the context stays usable afterwards:
 *   TBE_SELFTEST_SORT_LOOKBACK  one radix-sort CTA looks back at a tile that
 *       no CTA publishes; sets TBE_FLAG_SORT_TIMEOUT.  Needs `workspace`
 *       (device, 256-byte aligned, >= tbe_selftest_workspace_bytes()).
 *   TBE_SELFTEST_COPY_WAIT      one warp waits on an mbarrier phase that no
 *       copy completes; sets TBE_FLAG_COPY_TIMEOUT.  workspace unused.
 * Nothing is copied while the waits run.  Asynchronous on `stream`; the flag
 * is visible after the stream completes (about one second later).
 */
#define TBE_SELFTEST_SORT_LOOKBACK 0
#define TBE_SELFTEST_COPY_WAIT 1
size_t tbe_selftest_workspace_bytes(void);
tbe_status tbe_selftest_wait_limit(int32_t kind, void *workspace, size_t workspace_bytes,
                                   int32_t *dev_status, cudaStream_t stream);

/* Which path tbe_forward will take for this problem: 1 generic, 2 histogram. */
int32_t tbe_select_path(const tbe_tables *tables, const tbe_batch *batch, const tbe_config *cfg);

/* Static string naming a status code. */
const char *tbe_status_string(tbe_status status);
const char *tbe_status_str(tbe_status status);   /* the same text */

/* Library version, major*10000 + minor*100 + patch. */
int32_t tbe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TBE_GB300_TBE_H */
