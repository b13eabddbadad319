// Run-length encoding of the sorted keys and segment-length routing: the
// last step of the batch inversion (FBTriton TBE redesign, accesspath.com,
// "transpose_embedding_input": one run = one unique (table,row) with all the
// positions that touch it; "Backward kernels", paths 1-3: SL < 256 takes the
// short-run kernel, SL >= 256 is cut into chunks of 256 lookups).
//
// Three passes over the sorted keys (no waits between CTAs):
//   count:  heads per 4096-key tile (a head starts a run; sentinel keys of
//           out-of-range lookups start none) and the first sentinel position
//   scan:   one CTA scans the tile head counts -> U = number of runs
//   write:  each head writes unique_keys[r] and seg_off[r]; seg_off[U] = N'
// then the route pass gives each long run a slot and a range of chunk slots.
#include "tbe_internal.cuh"

namespace tbe {

constexpr int RLE_THREADS = 256;
constexpr int RLE_IPT = 16;
constexpr int RLE_TILE = RLE_THREADS * RLE_IPT;

// tile head counts, then CHUNK_WINDOWS_MAX window counters
size_t rle_workspace_bytes(int64_t N) {
    const int64_t ntiles = (N + RLE_TILE - 1) / RLE_TILE;
    return ((size_t)(ntiles + 1) * 4 + 255) / 256 * 256 + (size_t)CHUNK_WINDOWS_MAX * 4;
}

// ordering needs at least one window per table within CHUNK_WINDOWS_MAX keys
bool chunk_order_on(int64_t B, int T) {
    return B >= CHUNK_ORDER_MIN_B && T >= 1 && T <= CHUNK_WINDOWS_MAX;
}

// windows of 2^shift bags (at least 512) with T * windows <= CHUNK_WINDOWS_MAX;
// with T <= CHUNK_WINDOWS_MAX the loop ends by the time one window covers B
int chunk_window_shift(int64_t B, int T) {
    int s = 9;
    while (s < 62 && (int64_t)T * ((B + (int64_t(1) << s) - 1) >> s) > CHUNK_WINDOWS_MAX) ++s;
    return s;
}

__device__ __forceinline__ int block_excl_scan(int x, int *tot_smem, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int y = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int z = __shfl_up_sync(FULL, y, o);
        if (lane >= o) y += z;
    }
    if (lane == 31) tot_smem[warp] = y;
    __syncthreads();
    int wp = 0, all = 0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        if (w < warp) wp += tot_smem[w];
        all += tot_smem[w];
    }
    total = all;
    return wp + y - x;
}

// the RLE_IPT consecutive keys of one thread from `base` (16-byte vector
// loads when all are inside the array, `fill` past its end)
template <typename KeyT>
__device__ __forceinline__ void load_run_keys(const KeyT *__restrict__ k, int64_t base, int64_t N,
                                              KeyT fill, KeyT (&kk)[RLE_IPT]) {
    constexpr int PER = 16 / (int)sizeof(KeyT);   // keys per vector
    if (base + RLE_IPT <= N) {
#pragma unroll
        for (int v = 0; v < RLE_IPT / PER; ++v) {
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(k + base) + v);
            const KeyT *e = reinterpret_cast<const KeyT *>(&q);
#pragma unroll
            for (int j = 0; j < PER; ++j) kk[v * PER + j] = e[j];
        }
    } else {
#pragma unroll
        for (int i = 0; i < RLE_IPT; ++i) kk[i] = base + i < N ? __ldg(k + base + i) : fill;
    }
}

template <typename KeyT>
__global__ void __launch_bounds__(RLE_THREADS) rle_count_kernel(const KeyT *__restrict__ k,
                                                                int64_t N, KeyT sentinel,
                                                                int32_t *tile_heads,
                                                                int32_t *counters) {
    __shared__ int tot[RLE_THREADS / 32];
    const int64_t base = (int64_t)blockIdx.x * RLE_TILE + threadIdx.x * RLE_IPT;
    int heads = 0;
    KeyT prev = base > 0 && base - 1 < N ? __ldg(k + base - 1) : ~KeyT(0);
    KeyT kk[RLE_IPT];
    load_run_keys(k, base, N, sentinel, kk);
#pragma unroll
    for (int i = 0; i < RLE_IPT; ++i) {
        const int64_t pos = base + i;
        if (pos < N) {
            // keys >= sentinel (out-of-range lookups and lookups outside every
            // well-formed bag; they sort last) start no run
            const KeyT cur = kk[i];
            const bool first = pos == 0 || cur != prev;
            if (first && cur < sentinel) ++heads;
            if (cur >= sentinel && (pos == 0 || prev < sentinel)) counters[C_N_VALID] = (int32_t)pos;
            if (pos == N - 1 && cur < sentinel) counters[C_N_VALID] = (int32_t)N;
            prev = cur;
        }
    }
    int total;
    block_excl_scan(heads, tot, total);
    if (threadIdx.x == 0) tile_heads[blockIdx.x] = total;
}

// One CTA of 1024 threads: exclusive scan of the tile head counts in place.
// Exclusive scan of the tile head counts in place, SCAN_PT consecutive
// counts per thread per round (one round up to 16K tiles: 64M keys).
constexpr int SCAN_PT = 16;
__global__ void __launch_bounds__(1024) rle_scan_kernel(int32_t *tile_heads, int64_t ntiles,
                                                        int32_t *counters) {
    __shared__ int tot[32];
    __shared__ int carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int64_t b0 = 0; b0 < ntiles; b0 += 1024 * SCAN_PT) {
        const int64_t i0 = b0 + (int64_t)threadIdx.x * SCAN_PT;
        int x[SCAN_PT];
        int sum = 0;
#pragma unroll
        for (int j = 0; j < SCAN_PT; ++j) {
            x[j] = i0 + j < ntiles ? tile_heads[i0 + j] : 0;
            sum += x[j];
        }
        int total;
        const int ex = block_excl_scan(sum, tot, total);
        int run = carry + ex;
#pragma unroll
        for (int j = 0; j < SCAN_PT; ++j) {
            if (i0 + j < ntiles) tile_heads[i0 + j] = run;
            run += x[j];
        }
        __syncthreads();
        if (threadIdx.x == 0) carry += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) counters[C_NUM_UNIQUE] = carry;
}

template <typename KeyT>
__global__ void __launch_bounds__(RLE_THREADS) rle_write_kernel(
    const KeyT *__restrict__ k, int64_t N, KeyT sentinel,
    const int32_t *__restrict__ tile_base, KeyT *unique_keys, int32_t *seg_off,
    const int32_t *counters) {
    __shared__ int tot[RLE_THREADS / 32];
    const int64_t base = (int64_t)blockIdx.x * RLE_TILE + threadIdx.x * RLE_IPT;
    KeyT kk[RLE_IPT];
    unsigned headmask = 0;
    KeyT prev = base > 0 && base - 1 < N ? __ldg(k + base - 1) : ~KeyT(0);
    load_run_keys(k, base, N, sentinel, kk);
#pragma unroll
    for (int i = 0; i < RLE_IPT; ++i) {
        const int64_t pos = base + i;
        if (pos < N && (pos == 0 || kk[i] != prev) && kk[i] < sentinel) headmask |= 1u << i;
        prev = kk[i];
    }
    int total;
    int r = tile_base[blockIdx.x] + block_excl_scan(__popc(headmask), tot, total);
#pragma unroll
    for (int i = 0; i < RLE_IPT; ++i)
        if (headmask & (1u << i)) {
            unique_keys[r] = kk[i];
            seg_off[r] = (int32_t)(base + i);
            ++r;
        }
    if (blockIdx.x == 0 && threadIdx.x == 0) seg_off[counters[C_NUM_UNIQUE]] = counters[C_N_VALID];
}

// Long runs (SL >= sl_threshold) get a slot l and ceil(SL/chunk) chunk slots.
// The order of slots depends on atomic arrival; results do not (each chunk
// covers a fixed position range and partials are summed in chunk order).
// Each chunk slot then gets a descriptor -- its position range, key (low and
// high 32 bits), long run, the run's first slot and chunk count, and the
// batch window of its first lookup's bag -- so the long-run kernel reads one
// 32-byte record per chunk.  With ordering on, each chunk is also counted in its window.
struct RouteParams {
    const int32_t *seg_off;
    const void *unique_keys;   // uint32 or uint64 (key64)
    int key64;
    const uint32_t *vals;
    const int32_t *bag_of;
    const int64_t *table_offset;
    int64_t B;
    int T;
    int payload_pos;
    int wshift;         // < 0: no ordering
    int32_t *counters;
    int32_t *long_run;
    int32_t *long_chunk_base;
    int32_t *chunk_desc;
    int32_t *owner;     // [max_chunks] long run of each slot (the order array's memory)
    int32_t *arrive;
    int32_t *win;       // [CHUNK_WINDOWS_MAX] chunks per window (zeroed before)
    int sl_threshold;
    int chunk;
};

__global__ void __launch_bounds__(256) route_kernel(const RouteParams p) {
    const int U = p.counters[C_NUM_UNIQUE];
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < U; r += gridDim.x * blockDim.x) {
        const int32_t rs = p.seg_off[r], re = p.seg_off[r + 1];
        const int len = re - rs;
        if (len < p.sl_threshold) continue;
        const int nch = (len + p.chunk - 1) / p.chunk;
        const int l = atomicAdd(p.counters + C_NUM_LONG, 1);
        const int cb = atomicAdd(p.counters + C_NUM_CHUNKS, nch);
        p.long_run[l] = r;
        p.long_chunk_base[l] = cb;
        p.arrive[l] = 0;
        for (int c = 0; c < nch; ++c) p.owner[cb + c] = l;
    }
}

// One thread per chunk slot: the slot's descriptor and, with ordering on,
// its window key t * windows_per_table + (first bag >> shift) (counted per
// CTA in shared memory, then added globally).  Ordering by key makes the
// warps of the long-run kernel work on one table's gradient rows of nearby
// bags at a time, a working set that L2 holds.
__global__ void __launch_bounds__(256) chunk_desc_kernel(const RouteParams p) {
    __shared__ int32_t wc[CHUNK_WINDOWS_MAX];
    const int wpt = p.wshift >= 0 ? (int)((p.B + (int64_t(1) << p.wshift) - 1) >> p.wshift) : 0;
    const int nwin = p.T * wpt;
    for (int i = threadIdx.x; i < nwin; i += blockDim.x) wc[i] = 0;
    __syncthreads();
    const int n = p.counters[C_NUM_CHUNKS];
    for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < n; c += gridDim.x * blockDim.x) {
        const int l = __ldg(p.owner + c);
        const int r = __ldg(p.long_run + l);
        const int cb = __ldg(p.long_chunk_base + l);
        const int32_t rs = __ldg(p.seg_off + r), re = __ldg(p.seg_off + r + 1);
        const uint64_t key = p.key64 ? __ldg(reinterpret_cast<const unsigned long long *>(p.unique_keys) + r)
                                     : __ldg(reinterpret_cast<const uint32_t *>(p.unique_keys) + r);
        const int t = table_of_key(p.table_offset, p.T, (int64_t)key);
        const int32_t s = rs + (c - cb) * p.chunk;
        int w = 0;
        if (p.wshift >= 0) {
            const uint32_t v = __ldg(p.vals + s);
            int64_t b = p.payload_pos ? (int64_t)__ldg(p.bag_of + v) - (int64_t)t * p.B : (int64_t)v;
            if (b < 0 || b >= p.B) b = 0;   // malformed offsets only
            w = t * wpt + (int)(b >> p.wshift);
            atomicAdd(wc + w, 1);
        }
        int4 *d = reinterpret_cast<int4 *>(p.chunk_desc + (int64_t)c * 8);
        d[0] = make_int4(s, min(s + p.chunk, re), (int)(uint32_t)key, (int)(uint32_t)(key >> 32));
        d[1] = make_int4(l, cb, (re - rs + p.chunk - 1) / p.chunk, w);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nwin; i += blockDim.x)
        if (wc[i]) atomicAdd(p.win + i, wc[i]);
}

// Exclusive scan of the window counts, in place (one CTA).
__global__ void __launch_bounds__(1024) chunk_window_scan_kernel(int32_t *win, int nwin) {
    __shared__ int tot[32];
    constexpr int PER = CHUNK_WINDOWS_MAX / 1024;
    int v[PER], x = 0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int w = threadIdx.x * PER + i;
        v[i] = w < nwin ? win[w] : 0;
        x += v[i];
    }
    int total;
    int run = block_excl_scan(x, tot, total);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int w = threadIdx.x * PER + i;
        if (w < nwin) win[w] = run;
        run += v[i];
    }
}

// chunk_order[window start + k] = slot: slots grouped by window.
__global__ void __launch_bounds__(256) chunk_order_kernel(const int32_t *__restrict__ chunk_desc,
                                                          const int32_t *counters, int32_t *win,
                                                          int32_t *chunk_order) {
    const int n = counters[C_NUM_CHUNKS];
    for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < n; c += gridDim.x * blockDim.x) {
        const int w = __ldg(chunk_desc + (int64_t)c * 8 + 7);
        chunk_order[atomicAdd(win + w, 1)] = c;
    }
}

__global__ void zero_words_kernel(int32_t *p, int n) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = 0;
}

__global__ void zero_counters_kernel(int32_t *counters) {
    if (threadIdx.x < C_COUNT) counters[threadIdx.x] = 0;
}

__global__ void zero_first_kernel(int32_t *p) { p[0] = 0; }

void launch_zero_counters(Launch &L, int32_t *counters) {
    L.before("tbe_zero_counters");
    zero_counters_kernel<<<1, 32, 0, L.stream>>>(counters);
    L.after();
}

// The counters were zeroed before the forward or linearize kernel.
tbe_status launch_rle(Launch &L, const RleArgs &a, void *ws) {
    if (a.N == 0) {
        // seg_off[0] = 0 for an empty batch
        L.before("tbe_rle_zero");
        zero_first_kernel<<<1, 1, 0, L.stream>>>(a.seg_off);
        L.after();
        return TBE_OK;
    }
    const int64_t ntiles = (a.N + RLE_TILE - 1) / RLE_TILE;
    int32_t *tile_heads = (int32_t *)ws;
    int32_t *win = (int32_t *)((char *)ws + ((size_t)(ntiles + 1) * 4 + 255) / 256 * 256);
    const bool order = a.order_ok && chunk_order_on(a.B, a.T);
    const int wshift = order ? chunk_window_shift(a.B, a.T) : -1;
    const int nwin = order ? a.T * (int)((a.B + (int64_t(1) << wshift) - 1) >> wshift) : 0;
    L.before("tbe_rle_count");
    if (a.key_bytes == 8)
        rle_count_kernel<uint64_t><<<(unsigned)ntiles, RLE_THREADS, 0, L.stream>>>(
            (const uint64_t *)a.sorted_keys, a.N, a.sentinel, tile_heads, a.counters);
    else
        rle_count_kernel<uint32_t><<<(unsigned)ntiles, RLE_THREADS, 0, L.stream>>>(
            (const uint32_t *)a.sorted_keys, a.N, (uint32_t)a.sentinel, tile_heads, a.counters);
    L.after();
    L.before("tbe_rle_scan");
    rle_scan_kernel<<<1, 1024, 0, L.stream>>>(tile_heads, ntiles, a.counters);
    L.after();
    L.before("tbe_rle_write");
    if (a.key_bytes == 8)
        rle_write_kernel<uint64_t><<<(unsigned)ntiles, RLE_THREADS, 0, L.stream>>>(
            (const uint64_t *)a.sorted_keys, a.N, a.sentinel, tile_heads, (uint64_t *)a.unique_keys,
            a.seg_off, a.counters);
    else
        rle_write_kernel<uint32_t><<<(unsigned)ntiles, RLE_THREADS, 0, L.stream>>>(
            (const uint32_t *)a.sorted_keys, a.N, (uint32_t)a.sentinel, tile_heads,
            (uint32_t *)a.unique_keys, a.seg_off, a.counters);
    L.after();
    if (order) {
        L.before("tbe_rle_zero");
        zero_words_kernel<<<(nwin + 255) / 256, 256, 0, L.stream>>>(win, nwin);
        L.after();
    }
    RouteParams p;
    p.seg_off = a.seg_off;
    p.unique_keys = a.unique_keys;
    p.key64 = a.key_bytes == 8;
    p.vals = a.sorted_vals;
    p.bag_of = a.bag_of;
    p.table_offset = a.table_offset;
    p.B = a.B;
    p.T = a.T;
    p.payload_pos = a.payload_pos;
    p.wshift = wshift;
    p.counters = a.counters;
    p.long_run = a.long_run;
    p.long_chunk_base = a.long_chunk_base;
    p.chunk_desc = a.chunk_desc;
    p.owner = a.chunk_order;   // overwritten by the order kernel after its last use
    p.arrive = a.arrive;
    p.win = win;
    p.sl_threshold = a.sl_threshold;
    p.chunk = a.chunk;
    int grid = (int)((a.N + 255) / 256);
    if (grid > L.num_sms * 8) grid = L.num_sms * 8;
    L.before("tbe_route");
    route_kernel<<<grid, 256, 0, L.stream>>>(p);
    L.after();
    int cg = (int)((a.N / 256 + 255) / 256);
    if (cg > L.num_sms * 4) cg = L.num_sms * 4;
    if (cg < 1) cg = 1;
    L.before("tbe_chunk_desc");
    chunk_desc_kernel<<<cg, 256, 0, L.stream>>>(p);
    L.after();
    if (order) {
        L.before("tbe_chunk_window_scan");
        chunk_window_scan_kernel<<<1, 1024, 0, L.stream>>>(win, nwin);
        L.after();
        L.before("tbe_chunk_order");
        chunk_order_kernel<<<cg, 256, 0, L.stream>>>(a.chunk_desc, a.counters, win, a.chunk_order);
        L.after();
    }
    return TBE_OK;
}

}  // namespace tbe
