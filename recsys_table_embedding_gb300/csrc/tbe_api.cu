// Host side of the C ABI declared in tbe.h: argument checks, buffer sizing,
// metadata binding and the order of kernel launches for each entry point.
// Everything here runs on the host and only enqueues work on the caller's
// stream; no device memory is allocated and no host synchronisation happens.
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <utility>
#include <vector>

#include "tbe_internal.cuh"

namespace tbe {

static int device_sms(int dev);

Launch::Launch(cudaStream_t s, const tbe_config *c) : stream(s), cfg(c) {
    // event recording continues after the pairs earlier calls recorded
    if (cfg != nullptr && cfg->kernel_events_used != nullptr) used = *cfg->kernel_events_used;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
    num_sms = device_sms(dev);
    if (cfg != nullptr && cfg->kernel_events != nullptr) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        capturing = cudaStreamIsCapturing(stream, &cs) == cudaSuccess &&
                    cs == cudaStreamCaptureStatusActive;
    }
}

// Timing events: during stream capture an event record must be an external
// event node of the graph (a plain record there only orders streams), so the
// graph records the timestamps each time it runs.
static void record(cudaEvent_t ev, cudaStream_t s, bool capturing) {
    if (capturing) cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
    else cudaEventRecord(ev, s);
}

void Launch::before(const char *name) {
    if (cfg == nullptr || cfg->kernel_events == nullptr || used >= cfg->n_kernel_events) return;
    record(cfg->kernel_events[2 * used], stream, capturing);
    if (cfg->kernel_names != nullptr) cfg->kernel_names[used] = name;
}

void Launch::after() {
    if (cudaPeekAtLastError() != cudaSuccess) failed = true;
    if (cfg == nullptr || cfg->kernel_events == nullptr || used >= cfg->n_kernel_events) return;
    record(cfg->kernel_events[2 * used + 1], stream, capturing);
    ++used;
    if (cfg->kernel_events_used != nullptr) *cfg->kernel_events_used = used;
}

// ---- per-device caches of launch properties
static std::mutex g_launch_mu;
static std::map<int, int> g_sms;
static std::map<std::tuple<int, const void *, int, size_t>, int> g_blocks;
static std::set<std::tuple<int, const void *, size_t>> g_smem;

static int device_sms(int dev) {
    std::lock_guard<std::mutex> lock(g_launch_mu);
    auto it = g_sms.find(dev);
    if (it != g_sms.end()) return it->second;
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n < 1) n = 1;
    g_sms[dev] = n;
    return n;
}

int cached_blocks_per_sm(int dev, const void *fn, int threads, size_t smem) {
    std::lock_guard<std::mutex> lock(g_launch_mu);
    const auto key = std::make_tuple(dev, fn, threads, smem);
    auto it = g_blocks.find(key);
    if (it != g_blocks.end()) return it->second;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess)
        per_sm = 0;
    if (per_sm < 1) per_sm = 1;
    g_blocks[key] = per_sm;
    return per_sm;
}

void cached_smem_attr(int dev, const void *fn, size_t smem) {
    std::lock_guard<std::mutex> lock(g_launch_mu);
    const auto key = std::make_tuple(dev, fn, smem);
    if (g_smem.count(key)) return;
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                         cudaSharedmemCarveoutMaxShared);
    g_smem.insert(key);
}

static bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

static int bits_for(int64_t v) {   // bits needed to represent v >= 0
    int b = 0;
    while (b < 63 && (v >> b) != 0) ++b;
    return b;
}

struct Problem {
    int64_t N, B, NB, rows_total, max_rows;
    int T, D, dtype;    // with layouts: D = the largest D, dtype = TBE_F32 if any table is FP32
    int key_bits, key_bytes, index_type;
    int path;           // 1 generic, 2 histogram
    int payload_pos;
    int64_t max_long, max_chunks;
    int sl_threshold, chunk, long_mode;
    bool layouts;       // tables or bags described by per-table layouts
    TableClasses classes;
};

// Tables and bags described by layouts: every table's shape is supported,
// weight regions are disjoint, bags follow one another and every output row
// lies inside out.  Fills the launch classes, NB, and the largest D.
static tbe_status check_layouts(const tbe_tables *tab, const tbe_batch *bt, Problem *pr) {
    const int T = tab->T;
    const int64_t *to = tab->table_offset_host;
    if (tab->layout != nullptr && (tab->layout_host == nullptr || bt->bag_layout == nullptr))
        return TBE_ERR_NULL_POINTER;
    if (bt->bag_layout != nullptr && bt->bag_layout_host == nullptr) return TBE_ERR_NULL_POINTER;
    if (!aligned(tab->layout, 8) || !aligned(bt->bag_layout, 8)) return TBE_ERR_MISALIGNED;
    pr->classes.classes.clear();
    pr->classes.B.assign(T, 0);
    int Dmax = 0, any32 = 0;
    // table shapes and disjoint weight regions
    std::vector<std::pair<int64_t, int64_t>> regions;
    for (int t = 0; t < T; ++t) {
        const int D = tab->layout_host ? tab->layout_host[t].D : tab->D;
        const int dt = tab->layout_host ? tab->layout_host[t].dtype : tab->dtype;
        if (dt != TBE_F32 && dt != TBE_F16 && dt != TBE_BF16) return TBE_ERR_UNSUPPORTED_DTYPE;
        const int esz = dt == TBE_F32 ? 4 : 2;
        if (D < 1 || !row_plan(D, esz).ok || !row_plan(D, 4).ok) return TBE_ERR_UNSUPPORTED_DIM;
        if (tab->layout_host) {
            const int64_t w0 = tab->layout_host[t].weights_byte_offset;
            if (w0 < 0 || w0 % 16) return TBE_ERR_MISALIGNED;
            regions.push_back({w0, w0 + (to[t + 1] - to[t]) * D * esz});
        }
        Dmax = D > Dmax ? D : Dmax;
        any32 |= dt == TBE_F32;
        size_t k = 0;
        while (k < pr->classes.classes.size() &&
               (pr->classes.classes[k].D != D || pr->classes.classes[k].dtype != dt))
            ++k;
        if (k == pr->classes.classes.size()) pr->classes.classes.push_back(TableClass{D, dt, {}});
        pr->classes.classes[k].tables.push_back(t);
    }
    std::sort(regions.begin(), regions.end());
    for (size_t i = 1; i < regions.size(); ++i)
        if (regions[i].first < regions[i - 1].second) return TBE_ERR_INVALID_ARGUMENT;
    // bags and output rows
    int64_t NB = 0;
    for (int t = 0; t < T; ++t) {
        const int D = tab->layout_host ? tab->layout_host[t].D : tab->D;
        int64_t B = bt->B, o0 = (int64_t)t * D, os = (int64_t)T * D;
        if (bt->bag_layout_host) {
            const tbe_bag_layout &L = bt->bag_layout_host[t];
            if (L.bag_offset != NB || L.B < 0) return TBE_ERR_INVALID_ARGUMENT;
            B = L.B;
            o0 = L.out_offset;
            os = L.out_stride;
            if (o0 < 0 || o0 % 4 || os % 4 || (B > 1 && os < D)) return TBE_ERR_INVALID_ARGUMENT;
            if (B > 0 && o0 + (B - 1) * os + D > bt->out_size) return TBE_ERR_INVALID_ARGUMENT;
        }
        pr->classes.B[t] = B;
        NB += B;
    }
    if (NB >= (int64_t(1) << 31)) return TBE_ERR_INVALID_ARGUMENT;
    // the backward stages gradient-row offsets as 32-bit counts of 16-byte
    // vectors: grad_out must stay under 64 GB
    if (bt->out_size / 4 >= (int64_t(1) << 32) - 1) return TBE_ERR_INVALID_ARGUMENT;
    pr->NB = NB;
    pr->D = Dmax;
    pr->dtype = any32 ? TBE_F32 : TBE_BF16;
    return TBE_OK;
}

static tbe_config defaults(const tbe_config *cfg) {
    tbe_config c;
    tbe_config_default(&c);
    if (cfg != nullptr) {
        c = *cfg;
        if (c.sl_threshold <= 0) c.sl_threshold = 256;
        if (c.chunk <= 0) c.chunk = 256;
    }
    return c;
}

static tbe_status check_problem(const tbe_tables *tab, const tbe_batch *bt, const tbe_config *cfg,
                                Problem *pr) {
    if (tab == nullptr || bt == nullptr) return TBE_ERR_NULL_POINTER;
    if (tab->weights == nullptr || tab->table_offset == nullptr || tab->table_offset_host == nullptr)
        return TBE_ERR_NULL_POINTER;
    const bool layouts = tab->layout != nullptr || bt->bag_layout != nullptr;
    if (tab->T < 1 || (tab->layout == nullptr && tab->D < 1)) return TBE_ERR_INVALID_ARGUMENT;
    if (tab->layout == nullptr && tab->dtype != TBE_F32 && tab->dtype != TBE_F16 &&
        tab->dtype != TBE_BF16)
        return TBE_ERR_UNSUPPORTED_DTYPE;
    if (bt->N < 0 || bt->N >= (int64_t(1) << 30) || (!layouts && bt->B < 0))
        return TBE_ERR_INVALID_ARGUMENT;
    if (!layouts && (int64_t)tab->T * bt->B >= (int64_t(1) << 31)) return TBE_ERR_INVALID_ARGUMENT;
    if (bt->offsets == nullptr) return TBE_ERR_NULL_POINTER;
    if (bt->N > 0 && bt->indices == nullptr) return TBE_ERR_NULL_POINTER;
    if (bt->index_type != TBE_INDEX_I32 && bt->index_type != TBE_INDEX_I64)
        return TBE_ERR_INVALID_ARGUMENT;
    const size_t isz = bt->index_type == TBE_INDEX_I64 ? 8 : 4;
    if (!aligned(tab->weights, 16) || !aligned(tab->table_offset, 8) || !aligned(bt->offsets, isz) ||
        !aligned(bt->indices, isz) || !aligned(bt->per_sample_weights, 4))
        return TBE_ERR_MISALIGNED;
    const int64_t *to = tab->table_offset_host;
    if (to[0] != 0) return TBE_ERR_INVALID_ARGUMENT;
    int64_t max_rows = 0;
    for (int t = 0; t < tab->T; ++t) {
        if (to[t + 1] < to[t]) return TBE_ERR_INVALID_ARGUMENT;
        if (to[t + 1] - to[t] > max_rows) max_rows = to[t + 1] - to[t];
    }
    const int64_t rows_total = to[tab->T];
    // linearised keys: int32 while the range (rows_total itself is the
    // sentinel key of ignored lookups) stays below 2^31 - 1 (decision
    // checklist item 6), 64-bit beyond
    if (rows_total >= (int64_t(1) << 62)) return TBE_ERR_KEY_RANGE;
    tbe_config c = defaults(cfg);
    if (c.long_run_mode < 0 || c.long_run_mode > 2 || c.hist_mode < 0 || c.hist_mode > 2)
        return TBE_ERR_INVALID_ARGUMENT;
    // a chunk's lookup table lives in shared memory next to the copy ring
    if (c.chunk < 32 || c.chunk > 1024) return TBE_ERR_INVALID_ARGUMENT;
    pr->N = bt->N;
    pr->B = bt->B;
    pr->NB = (int64_t)tab->T * bt->B;
    pr->T = tab->T;
    pr->D = tab->D;
    pr->dtype = tab->dtype;
    pr->layouts = layouts;
    if (layouts) {
        const tbe_status ls = check_layouts(tab, bt, pr);
        if (ls != TBE_OK) return ls;
    } else {
        pr->classes.classes.assign(1, TableClass{tab->D, tab->dtype, {}});
        pr->classes.B.clear();
    }
    pr->rows_total = rows_total;
    pr->max_rows = max_rows;
    pr->key_bits = bits_for(rows_total);
    pr->key_bytes = rows_total < (int64_t(1) << 31) - 1 ? 4 : 8;
    if (c.key_bytes != 0 && c.key_bytes != 4 && c.key_bytes != 8) return TBE_ERR_INVALID_ARGUMENT;
    if (c.key_bytes == 4 && pr->key_bytes == 8) return TBE_ERR_KEY_RANGE;
    if (c.key_bytes == 8) pr->key_bytes = 8;
    pr->index_type = bt->index_type;
    pr->payload_pos = bt->per_sample_weights != nullptr ? 1 : 0;
    pr->sl_threshold = c.sl_threshold;
    pr->chunk = c.chunk;
    pr->long_mode = c.long_run_mode == TBE_LONG_FUSED ? TBE_LONG_FUSED : TBE_LONG_TWO_KERNEL;
    pr->max_long = bt->N / c.sl_threshold + 1;
    pr->max_chunks = bt->N / c.chunk + pr->max_long + 1;
    pr->path = 1;
    if (c.hist_mode != TBE_HIST_OFF && !layouts && hist_shape_ok(tab, bt, max_rows)) {
        const bool dense_enough = bt->N >= 64 * pr->NB;   // L >= 64 on average
        if (c.hist_mode == TBE_HIST_FORCE || dense_enough) pr->path = 2;
    } else if (c.hist_mode == TBE_HIST_FORCE) {
        return TBE_ERR_HISTOGRAM_SHAPE;
    }
    if (layouts) return TBE_OK;   // shapes and sizes checked per table above
    // the generic path reads weight rows and gradient rows as 16-byte vectors
    const int esz = tab->dtype == TBE_F32 ? 4 : 2;
    if (pr->path == 1 && (!row_plan(tab->D, esz).ok || !row_plan(tab->D, 4).ok))
        return TBE_ERR_UNSUPPORTED_DIM;
    // the backward stages gradient-row offsets as 32-bit counts of 16-byte
    // vectors: grad_out must stay under 64 GB
    // (one value short of 2^32: the backward marks a missing row with all ones)
    if (pr->path == 1 && pr->NB * tab->D / 4 >= (int64_t(1) << 32) - 1) return TBE_ERR_INVALID_ARGUMENT;
    return TBE_OK;
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Meta layout (each array 256-byte aligned).
struct MetaLayout {
    size_t keys_a, vals_a, keys_b, vals_b, bag_of, unique_keys, seg_off, counters, long_run,
        long_chunk_base, arrive, chunk_order, chunk_desc, hist, total;
};

static MetaLayout meta_layout(const Problem &pr) {
    MetaLayout m;
    memset(&m, 0, sizeof(m));
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    const size_t N = (size_t)pr.N;
    const size_t kb = (size_t)pr.key_bytes;
    if (pr.path == 1) {
        m.keys_a = take(N * kb + 16);
        m.vals_a = take(N * 4 + 16);
        m.keys_b = take(N * kb + 16);
        m.vals_b = take(N * 4 + 16);
        m.bag_of = pr.payload_pos ? take(N * 4 + 16) : (size_t)-1;
        m.unique_keys = take(N * kb + 16);
        m.seg_off = take((N + 1) * 4 + 16);
        m.counters = take(C_COUNT * 4);
        m.long_run = take((size_t)pr.max_long * 4);
        m.long_chunk_base = take((size_t)pr.max_long * 4);
        m.arrive = take((size_t)pr.max_long * 4);
        m.chunk_order = take((size_t)pr.max_chunks * 4);
        m.chunk_desc = take((size_t)pr.max_chunks * 32);
        m.hist = (size_t)-1;
    } else {
        m.keys_a = m.vals_a = m.keys_b = m.vals_b = m.bag_of = m.unique_keys = m.seg_off =
            m.long_run = m.long_chunk_base = m.arrive = m.chunk_order = m.chunk_desc = (size_t)-1;
        m.counters = take(C_COUNT * 4);
        m.hist = take((size_t)pr.NB * 64 * 2);
    }
    m.total = off;
    return m;
}

// bytes between chunk slots' partials in the workspace: D accumulators of
// the table's precision, or with layouts the largest D in FP64 (any class)
static int64_t part_stride(const Problem &pr) {
    if (pr.layouts) return (int64_t)pr.D * 8;
    return (int64_t)bwd_partials_bytes(1, pr.D, pr.dtype);
}

static size_t workspace_size(const tbe_tables *tab, const tbe_batch *bt, const Problem &pr) {
    size_t ws = 256;
    if (pr.path == 1) {
        size_t pre = sort_workspace_bytes(pr.N, pr.key_bits);
        const size_t rle = rle_workspace_bytes(pr.N);
        if (rle > pre) pre = rle;
        const size_t bwd = (size_t)pr.max_chunks * part_stride(pr);
        ws = pre > bwd ? pre : bwd;
    } else {
        ws = hist_workspace_bytes(tab, bt);
    }
    return align_up(ws + 256, 256);
}

static tbe_status check_meta(const tbe_meta *meta, const Problem &pr) {
    if (meta->bound_N != pr.N || meta->bound_B != pr.B || meta->bound_T != pr.T ||
        meta->path != pr.path || meta->payload_is_pos != pr.payload_pos ||
        meta->rows_total != pr.rows_total || meta->key_bytes != pr.key_bytes ||
        meta->index_type != pr.index_type)
        return TBE_ERR_META;
    return TBE_OK;
}

static tbe_status finish(const Launch &L, tbe_status st) {
    if (st != TBE_OK) return st;
    return L.failed ? TBE_ERR_CUDA : TBE_OK;
}

// After the forward or linearize kernel wrote keys and payloads: the
// malformed-offsets fixup, sort, RLE/route (generic path)
static tbe_status run_inversion(Launch &L, const tbe_tables *tab, const tbe_batch *bt,
                                tbe_meta *meta, const Problem &pr, void *ws, int32_t *status) {
    tbe_status st = launch_offsets_fixup(L, tab, bt, meta->keys_a, pr.key_bytes, meta->vals_a,
                                         meta->bag_of, (uint64_t)pr.rows_total, meta->counters);
    if (st != TBE_OK) return st;
    bool in_b = false;
    st = launch_sort(L, meta->keys_a, meta->vals_a, meta->keys_b, meta->vals_b, pr.N, pr.key_bits,
                     pr.key_bytes, ws, status, &in_b);
    if (st != TBE_OK) return st;
    meta->sorted_keys = in_b ? meta->keys_b : meta->keys_a;
    meta->sorted_vals = in_b ? meta->vals_b : meta->vals_a;
    RleArgs a;
    a.sorted_keys = meta->sorted_keys;
    a.sorted_vals = meta->sorted_vals;
    a.bag_of = meta->bag_of;
    a.N = pr.N;
    a.B = pr.B;
    a.sentinel = (uint64_t)pr.rows_total;
    a.key_bytes = pr.key_bytes;
    a.payload_pos = meta->payload_is_pos;
    a.unique_keys = meta->unique_keys;
    a.seg_off = meta->seg_off;
    a.counters = meta->counters;
    a.long_run = meta->long_run;
    a.long_chunk_base = meta->long_chunk_base;
    a.chunk_order = meta->chunk_order;
    a.chunk_desc = meta->chunk_desc;
    a.arrive = meta->arrive;
    a.table_offset = tab->table_offset;
    a.T = tab->T;
    a.sl_threshold = pr.sl_threshold;
    a.chunk = pr.chunk;
    a.order_ok = bt->bag_layout == nullptr;
    return launch_rle(L, a, ws);
}

}  // namespace tbe

using namespace tbe;

extern "C" {

void tbe_config_default(tbe_config *cfg) {
    if (cfg == nullptr) return;
    memset(cfg, 0, sizeof(*cfg));
    cfg->sl_threshold = 256;
    cfg->chunk = 256;
    cfg->long_run_mode = TBE_LONG_AUTO;
    cfg->hist_mode = TBE_HIST_AUTO;
}

tbe_status tbe_query_sizes(const tbe_tables *tables, const tbe_batch *batch, const tbe_config *cfg,
                           size_t *meta_bytes, size_t *workspace_bytes) {
    Problem pr;
    tbe_status st = check_problem(tables, batch, cfg, &pr);
    if (st != TBE_OK) return st;
    if (meta_bytes) *meta_bytes = meta_layout(pr).total;
    if (workspace_bytes) *workspace_bytes = workspace_size(tables, batch, pr);
    return TBE_OK;
}

size_t tbe_workspace_bytes(const tbe_tables *tables, const tbe_batch *batch, const tbe_config *cfg) {
    size_t w = 0;
    return tbe_query_sizes(tables, batch, cfg, nullptr, &w) == TBE_OK ? w : 0;
}

size_t tbe_meta_bytes(const tbe_tables *tables, const tbe_batch *batch, const tbe_config *cfg) {
    size_t m = 0;
    return tbe_query_sizes(tables, batch, cfg, &m, nullptr) == TBE_OK ? m : 0;
}

int32_t tbe_select_path(const tbe_tables *tables, const tbe_batch *batch, const tbe_config *cfg) {
    Problem pr;
    if (check_problem(tables, batch, cfg, &pr) != TBE_OK) return 0;
    return pr.path;
}

tbe_status tbe_meta_bind(tbe_meta *meta, void *device_buf, size_t bytes, const tbe_tables *tables,
                         const tbe_batch *batch, const tbe_config *cfg) {
    if (meta == nullptr || device_buf == nullptr) return TBE_ERR_NULL_POINTER;
    if (!aligned(device_buf, 256)) return TBE_ERR_MISALIGNED;
    Problem pr;
    tbe_status st = check_problem(tables, batch, cfg, &pr);
    if (st != TBE_OK) return st;
    const MetaLayout L = meta_layout(pr);
    if (bytes < L.total) return TBE_ERR_BUFFER_TOO_SMALL;
    char *b = (char *)device_buf;
    auto at = [&](size_t off) -> void * { return off == (size_t)-1 ? nullptr : (void *)(b + off); };
    memset(meta, 0, sizeof(*meta));
    meta->bound_N = pr.N;
    meta->bound_B = pr.B;
    meta->bound_T = pr.T;
    meta->path = pr.path;
    meta->payload_is_pos = pr.payload_pos;
    meta->key_bits = pr.key_bits;
    meta->rows_total = pr.rows_total;
    meta->key_bytes = pr.key_bytes;
    meta->index_type = pr.index_type;
    meta->keys_a = at(L.keys_a);
    meta->vals_a = (uint32_t *)at(L.vals_a);
    meta->keys_b = at(L.keys_b);
    meta->vals_b = (uint32_t *)at(L.vals_b);
    meta->sorted_keys = meta->keys_a;
    meta->sorted_vals = meta->vals_a;
    meta->bag_of = (int32_t *)at(L.bag_of);
    meta->unique_keys = at(L.unique_keys);
    meta->seg_off = (int32_t *)at(L.seg_off);
    meta->counters = (int32_t *)at(L.counters);
    meta->long_run = (int32_t *)at(L.long_run);
    meta->long_chunk_base = (int32_t *)at(L.long_chunk_base);
    meta->chunk_order = (int32_t *)at(L.chunk_order);
    meta->chunk_desc = (int32_t *)at(L.chunk_desc);
    meta->hist = (uint16_t *)at(L.hist);
    meta->bytes = L.total;
    meta->arrive = (int32_t *)at(L.arrive);
    return TBE_OK;
}

tbe_status tbe_forward(const tbe_tables *tables, const tbe_batch *batch, float *out, tbe_meta *meta,
                       void *workspace, size_t workspace_bytes, int32_t *dev_status,
                       const tbe_config *cfg, cudaStream_t stream) {
    Problem pr;
    tbe_status st = check_problem(tables, batch, cfg, &pr);
    if (st != TBE_OK) return st;
    if (out == nullptr || dev_status == nullptr) return TBE_ERR_NULL_POINTER;
    if (!aligned(out, 16)) return TBE_ERR_MISALIGNED;
    if (meta != nullptr) {
        if ((st = check_meta(meta, pr)) != TBE_OK) return st;
        if (workspace == nullptr) return TBE_ERR_NULL_POINTER;
        if (workspace_bytes < workspace_size(tables, batch, pr)) return TBE_ERR_BUFFER_TOO_SMALL;
    }
    Launch L(stream, cfg);
    if (meta != nullptr) launch_zero_counters(L, meta->counters);
    if (pr.path == 2) {
        st = launch_hist_forward(L, tables, batch, out, meta ? meta->hist : nullptr, dev_status,
                                 meta ? meta->counters : nullptr);
        return finish(L, st);
    }
    // the forward kernel writes 32-bit keys itself; 64-bit keys come from
    // the linearize kernel after it
    const bool fused_keys = meta != nullptr && pr.key_bytes == 4;
    st = launch_forward(L, tables, batch, out, fused_keys ? (uint32_t *)meta->keys_a : nullptr,
                        fused_keys ? meta->vals_a : nullptr, fused_keys ? meta->bag_of : nullptr,
                        (uint64_t)pr.rows_total, dev_status, meta ? meta->counters : nullptr,
                        pr.classes);
    if (st == TBE_OK && meta != nullptr && !fused_keys)
        st = launch_linearize(L, tables, batch, meta->keys_a, pr.key_bytes, meta->vals_a,
                              meta->bag_of, (uint64_t)pr.rows_total, dev_status, meta->counters);
    if (st == TBE_OK && meta != nullptr)
        st = run_inversion(L, tables, batch, meta, pr, workspace, dev_status);
    return finish(L, st);
}

tbe_status tbe_preprocess(const tbe_tables *tables, const tbe_batch *batch, tbe_meta *meta,
                          void *workspace, size_t workspace_bytes, int32_t *dev_status,
                          const tbe_config *cfg, cudaStream_t stream) {
    Problem pr;
    tbe_status st = check_problem(tables, batch, cfg, &pr);
    if (st != TBE_OK) return st;
    if (meta == nullptr || workspace == nullptr || dev_status == nullptr) return TBE_ERR_NULL_POINTER;
    if ((st = check_meta(meta, pr)) != TBE_OK) return st;
    if (workspace_bytes < workspace_size(tables, batch, pr)) return TBE_ERR_BUFFER_TOO_SMALL;
    Launch L(stream, cfg);
    launch_zero_counters(L, meta->counters);
    if (pr.path == 2)
        return finish(L, launch_hist_count(L, tables, batch, meta->hist, dev_status, meta->counters));
    st = launch_linearize(L, tables, batch, meta->keys_a, pr.key_bytes, meta->vals_a, meta->bag_of,
                          (uint64_t)pr.rows_total, dev_status, meta->counters);
    if (st == TBE_OK) st = run_inversion(L, tables, batch, meta, pr, workspace, dev_status);
    return finish(L, st);
}

tbe_status tbe_backward_rowwise_adagrad(const tbe_tables *tables, const tbe_batch *batch,
                                        float *momentum, const float *grad_out,
                                        const tbe_meta *meta, float lr, float eps, void *workspace,
                                        size_t workspace_bytes, int32_t *dev_status,
                                        const tbe_config *cfg, cudaStream_t stream) {
    Problem pr;
    tbe_status st = check_problem(tables, batch, cfg, &pr);
    if (st != TBE_OK) return st;
    if (momentum == nullptr || grad_out == nullptr || meta == nullptr || workspace == nullptr ||
        dev_status == nullptr)
        return TBE_ERR_NULL_POINTER;
    if (!aligned(grad_out, 16) || !aligned(momentum, 4) || !aligned(workspace, 256))
        return TBE_ERR_MISALIGNED;
    if ((st = check_meta(meta, pr)) != TBE_OK) return st;
    if (workspace_bytes < workspace_size(tables, batch, pr)) return TBE_ERR_BUFFER_TOO_SMALL;
    Launch L(stream, cfg);
    if (pr.path == 2)
        return finish(L, launch_hist_backward(L, tables, batch, meta->hist, momentum, grad_out, lr,
                                              eps, workspace, dev_status, meta->counters));
    BwdArgs a;
    a.tab = tables;
    a.bt = batch;
    a.meta = meta;
    a.momentum = momentum;
    a.grad_out = grad_out;
    a.lr = lr;
    a.eps = eps;
    a.partials = workspace;
    a.arrive = meta->arrive;
    a.status = dev_status;
    a.max_chunks = pr.max_chunks;
    a.max_long = pr.max_long;
    a.sl_threshold = pr.sl_threshold;
    a.chunk = pr.chunk;
    a.long_mode = pr.long_mode;
    a.classes = &pr.classes;
    a.part_stride = part_stride(pr);
    return finish(L, launch_backward(L, a));
}

const char *tbe_status_str(tbe_status s) { return tbe_status_string(s); }

const char *tbe_status_string(tbe_status s) {
    switch (s) {
    case TBE_OK: return "ok";
    case TBE_ERR_NULL_POINTER: return "null pointer";
    case TBE_ERR_INVALID_ARGUMENT: return "invalid argument";
    case TBE_ERR_UNSUPPORTED_DIM: return "unsupported embedding dimension";
    case TBE_ERR_UNSUPPORTED_DTYPE: return "unsupported weight dtype";
    case TBE_ERR_MISALIGNED: return "misaligned pointer";
    case TBE_ERR_KEY_RANGE: return "linearised key range of 2^62 rows or more";
    case TBE_ERR_BUFFER_TOO_SMALL: return "workspace or meta buffer too small";
    case TBE_ERR_META: return "meta not bound for this problem";
    case TBE_ERR_HISTOGRAM_SHAPE: return "histogram path does not cover this shape";
    case TBE_ERR_CUDA: return "CUDA launch failure";
    case TBE_ERR_SCRATCH_LIMIT:
        return "batch larger than tbe_preprocess_static's built-in scratch (at most 4194304 lookups)";
    }
    return "unknown status";
}

int32_t tbe_version(void) { return 200; }

size_t tbe_selftest_workspace_bytes(void) { return sort_selftest_bytes(); }

tbe_status tbe_selftest_wait_limit(int32_t kind, void *workspace, size_t workspace_bytes,
                                   int32_t *dev_status, cudaStream_t stream) {
    if (dev_status == nullptr) return TBE_ERR_NULL_POINTER;
    if (kind != TBE_SELFTEST_SORT_LOOKBACK && kind != TBE_SELFTEST_COPY_WAIT)
        return TBE_ERR_INVALID_ARGUMENT;
    Launch L(stream, nullptr);
    if (kind == TBE_SELFTEST_COPY_WAIT) return finish(L, launch_copy_wait_selftest(L, dev_status));
    if (workspace == nullptr) return TBE_ERR_NULL_POINTER;
    if (!aligned(workspace, 256)) return TBE_ERR_MISALIGNED;
    if (workspace_bytes < sort_selftest_bytes()) return TBE_ERR_BUFFER_TOO_SMALL;
    return finish(L, launch_sort_selftest(L, workspace, dev_status));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Batch inversion without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// batch inversion: code running inside a device-memory allocator or memory
// pool callback (allocating there would recurse), plug-ins that a host
// framework hands only fixed input and output buffers, and services that must
// not grow their device footprint after start-up.  tbe_preprocess_static
// serves them: the scratch of the radix sort and the run-length encoding is
// one file-scope device array of this library, so the call allocates nothing.
// The array occupies STATIC_SCRATCH_BYTES on every GPU that loads the library
// until the process exits, and bounds the batch at STATIC_SCRATCH_MAX_N
// lookups.  All calls on a device share the array.

namespace tbe {

constexpr size_t STATIC_SCRATCH_BYTES = (size_t)8 * 1024 * 1024 + 64 * 1024;  // 8 MiB + 64 KiB
constexpr int64_t STATIC_SCRATCH_MAX_N = (int64_t)1 << 22;                    // 4,194,304 lookups
constexpr int STATIC_MAX_DEVICES = 64;

static __device__ __align__(256) unsigned char g_static_scratch[STATIC_SCRATCH_BYTES];

static std::mutex g_static_mu;
static void *g_static_scratch_ptr[STATIC_MAX_DEVICES];

// Device address of g_static_scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
static tbe_status static_scratch(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= STATIC_MAX_DEVICES) return TBE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (g_static_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || p == nullptr) return TBE_ERR_CUDA;
        g_static_scratch_ptr[dev] = p;
    }
    *out = g_static_scratch_ptr[dev];
    return TBE_OK;
}

}  // namespace tbe

extern "C" tbe_status tbe_preprocess_static(const tbe_tables *tables, const tbe_batch *batch,
                                            tbe_meta *meta, int32_t *dev_status,
                                            const tbe_config *cfg, cudaStream_t stream) {
    Problem pr;
    tbe_status st = check_problem(tables, batch, cfg, &pr);
    if (st != TBE_OK) return st;
    if (meta == nullptr || dev_status == nullptr) return TBE_ERR_NULL_POINTER;
    if ((st = check_meta(meta, pr)) != TBE_OK) return st;
    if (pr.N > STATIC_SCRATCH_MAX_N) return TBE_ERR_SCRATCH_LIMIT;
    size_t need = sort_workspace_bytes(pr.N, pr.key_bits);
    if (rle_workspace_bytes(pr.N) > need) need = rle_workspace_bytes(pr.N);
    if (need > STATIC_SCRATCH_BYTES) return TBE_ERR_SCRATCH_LIMIT;
    Launch L(stream, cfg);
    launch_zero_counters(L, meta->counters);
    // the histogram path's counting needs no scratch
    if (pr.path == 2)
        return finish(L, launch_hist_count(L, tables, batch, meta->hist, dev_status, meta->counters));
    void *scratch = nullptr;
    if ((st = static_scratch(&scratch)) != TBE_OK) return st;
    // The sort zeroes its digit counts, tile tickets and look-back words, and
    // the RLE writes its tile counts before reading them, so the contents a
    // previous call left in the array are never read.
    st = launch_linearize(L, tables, batch, meta->keys_a, pr.key_bytes, meta->vals_a, meta->bag_of,
                          (uint64_t)pr.rows_total, dev_status, meta->counters);
    if (st == TBE_OK) st = run_inversion(L, tables, batch, meta, pr, scratch, dev_status);
    return finish(L, st);
}
