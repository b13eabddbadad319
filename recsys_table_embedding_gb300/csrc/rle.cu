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

size_t rle_workspace_bytes(int64_t N) {
    const int64_t ntiles = (N + RLE_TILE - 1) / RLE_TILE;
    return (size_t)(ntiles + 1) * 4 + 256;
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

__global__ void __launch_bounds__(RLE_THREADS) rle_count_kernel(const uint32_t *__restrict__ k,
                                                                int64_t N, uint32_t sentinel,
                                                                int32_t *tile_heads,
                                                                int32_t *counters) {
    __shared__ int tot[RLE_THREADS / 32];
    const int64_t base = (int64_t)blockIdx.x * RLE_TILE + threadIdx.x * RLE_IPT;
    int heads = 0;
    uint32_t prev = base > 0 && base - 1 < N ? __ldg(k + base - 1) : 0xffffffffu;
#pragma unroll
    for (int i = 0; i < RLE_IPT; ++i) {
        const int64_t pos = base + i;
        if (pos < N) {
            const uint32_t cur = __ldg(k + pos);
            const bool first = pos == 0 || cur != prev;
            if (first && cur != sentinel) ++heads;
            if (cur == sentinel && first) counters[C_N_VALID] = (int32_t)pos;
            if (pos == N - 1 && cur != sentinel) counters[C_N_VALID] = (int32_t)N;
            prev = cur;
        }
    }
    int total;
    block_excl_scan(heads, tot, total);
    if (threadIdx.x == 0) tile_heads[blockIdx.x] = total;
}

// One CTA of 1024 threads: exclusive scan of the tile head counts in place.
__global__ void __launch_bounds__(1024) rle_scan_kernel(int32_t *tile_heads, int64_t ntiles,
                                                        int32_t *counters) {
    __shared__ int tot[32];
    __shared__ int carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    for (int64_t b0 = 0; b0 < ntiles; b0 += 1024) {
        const int64_t i = b0 + threadIdx.x;
        const int x = i < ntiles ? tile_heads[i] : 0;
        int total;
        const int ex = block_excl_scan(x, tot, total);
        const int c = carry;
        if (i < ntiles) tile_heads[i] = c + ex;
        __syncthreads();
        if (threadIdx.x == 0) carry = c + total;
        __syncthreads();
    }
    if (threadIdx.x == 0) counters[C_NUM_UNIQUE] = carry;
}

__global__ void __launch_bounds__(RLE_THREADS) rle_write_kernel(
    const uint32_t *__restrict__ k, int64_t N, uint32_t sentinel,
    const int32_t *__restrict__ tile_base, uint32_t *unique_keys, int32_t *seg_off,
    const int32_t *counters) {
    __shared__ int tot[RLE_THREADS / 32];
    const int64_t base = (int64_t)blockIdx.x * RLE_TILE + threadIdx.x * RLE_IPT;
    uint32_t kk[RLE_IPT];
    unsigned headmask = 0;
    uint32_t prev = base > 0 && base - 1 < N ? __ldg(k + base - 1) : 0xffffffffu;
#pragma unroll
    for (int i = 0; i < RLE_IPT; ++i) {
        const int64_t pos = base + i;
        kk[i] = pos < N ? __ldg(k + pos) : sentinel;
        if (pos < N && (pos == 0 || kk[i] != prev) && kk[i] != sentinel) headmask |= 1u << i;
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
// Each chunk slot also gets a descriptor -- its position range, key, table,
// long run, the run's first slot and chunk count -- so the long-run kernel
// reads one 32-byte record per chunk instead of chasing the run tables.
__global__ void __launch_bounds__(256) route_kernel(const int32_t *__restrict__ seg_off,
                                                    const uint32_t *__restrict__ unique_keys,
                                                    const int64_t *__restrict__ table_offset,
                                                    int T, int32_t *counters, int32_t *long_run,
                                                    int32_t *long_chunk_base,
                                                    int32_t *chunk_owner, int32_t *chunk_desc,
                                                    int32_t *arrive, int sl_threshold, int chunk) {
    const int U = counters[C_NUM_UNIQUE];
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < U; r += gridDim.x * blockDim.x) {
        const int32_t rs = seg_off[r], re = seg_off[r + 1];
        const int len = re - rs;
        if (len < sl_threshold) continue;
        const int nch = (len + chunk - 1) / chunk;
        const int l = atomicAdd(counters + C_NUM_LONG, 1);
        const int cb = atomicAdd(counters + C_NUM_CHUNKS, nch);
        const uint32_t key = unique_keys[r];
        const int t = table_of_key(table_offset, T, key);
        long_run[l] = r;
        long_chunk_base[l] = cb;
        arrive[l] = 0;
        for (int c = 0; c < nch; ++c) {
            chunk_owner[cb + c] = l;
            const int32_t s = rs + c * chunk;
            int4 *d = reinterpret_cast<int4 *>(chunk_desc + (int64_t)(cb + c) * 8);
            d[0] = make_int4(s, min(s + chunk, re), (int)key, t);
            d[1] = make_int4(l, cb, nch, 0);
        }
    }
}

__global__ void zero_counters_kernel(int32_t *counters) {
    if (threadIdx.x < C_COUNT) counters[threadIdx.x] = 0;
}

__global__ void zero_first_kernel(int32_t *p) { p[0] = 0; }

tbe_status launch_rle(Launch &L, const uint32_t *sorted_keys, int64_t N, uint32_t sentinel,
                      uint32_t *unique_keys, int32_t *seg_off, int32_t *counters,
                      int32_t *long_run, int32_t *long_chunk_base, int32_t *chunk_owner,
                      int32_t *chunk_desc, int32_t *arrive, const int64_t *table_offset, int T,
                      int sl_threshold, int chunk, void *ws) {
    L.before("tbe_rle_zero");
    zero_counters_kernel<<<1, 32, 0, L.stream>>>(counters);
    L.after();
    if (N == 0) {
        // seg_off[0] = 0 for an empty batch
        L.before("tbe_rle_zero");
        zero_first_kernel<<<1, 1, 0, L.stream>>>(seg_off);
        L.after();
        return TBE_OK;
    }
    const int64_t ntiles = (N + RLE_TILE - 1) / RLE_TILE;
    int32_t *tile_heads = (int32_t *)ws;
    L.before("tbe_rle_count");
    rle_count_kernel<<<(unsigned)ntiles, RLE_THREADS, 0, L.stream>>>(sorted_keys, N, sentinel,
                                                                     tile_heads, counters);
    L.after();
    L.before("tbe_rle_scan");
    rle_scan_kernel<<<1, 1024, 0, L.stream>>>(tile_heads, ntiles, counters);
    L.after();
    L.before("tbe_rle_write");
    rle_write_kernel<<<(unsigned)ntiles, RLE_THREADS, 0, L.stream>>>(
        sorted_keys, N, sentinel, tile_heads, unique_keys, seg_off, counters);
    L.after();
    int grid = (int)((N + 255) / 256);
    if (grid > L.num_sms * 8) grid = L.num_sms * 8;
    L.before("tbe_route");
    route_kernel<<<grid, 256, 0, L.stream>>>(seg_off, unique_keys, table_offset, T, counters,
                                             long_run, long_chunk_base, chunk_owner, chunk_desc,
                                             arrive, sl_threshold, chunk);
    L.after();
    return TBE_OK;
}

}  // namespace tbe
