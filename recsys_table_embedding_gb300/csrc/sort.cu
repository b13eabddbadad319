// Stable LSD radix sort of (key, payload) pairs: the sort step of the batch
// inversion (FBTriton TBE redesign, accesspath.com, "transpose_embedding_input";
// decision checklist item 6: int32 keys halve the sort-key width).  Keys are
// 32-bit, or 64-bit when the linearised range reaches 2^31.  Only the
// significant key bits are sorted, in ceil(key_bits / 9) passes of at most
// 9 bits (512 buckets): 26-bit keys take 3 passes, 32-bit keys 4.
//
// Design (onesweep: one read and one write of the pairs per pass, digit
// prefixes across tiles by decoupled look-back):
//  1. one histogram kernel counts every pass's digits at once and zeroes the
//     look-back state; a 512-thread kernel per pass turns counts into bucket
//     starts;
//  2. per pass, CTAs take tiles in ticket order (an atomic counter, so a
//     CTA only ever waits for tiles that CTAs already running hold).  A tile
//     of 4096 pairs is ranked stably inside the CTA (per-warp match_any
//     ranking in input order, then warp prefixes), each digit's tile count is
//     published, and thread d (one per bucket) looks back over earlier
//     tiles for digit d's running prefix, reading LOOKBACK predecessors per
//     round trip.  The tile is reordered by digit in shared memory and
//     written out, so each digit's run of pairs lands contiguously.
//  The look-back status word packs a 2-bit state and a 30-bit count (so
//  N < 2^30).  Every wait is bounded: after WAIT_LIMIT_NS of polling the CTA
//  sets TBE_FLAG_SORT_TIMEOUT in the status word and carries on (the sort
//  output is then invalid, which the flag reports).
#include <type_traits>

#include "tbe_internal.cuh"

namespace tbe {

constexpr int MAX_DIGIT_BITS = 9;
constexpr int RADIX = 1 << MAX_DIGIT_BITS;   // buckets per pass (digits use <= 9 bits)
constexpr int SORT_THREADS = 512;
constexpr int SORT_WARPS = SORT_THREADS / 32;
// Pairs per thread for 32-bit keys, and whether payloads are read only when
// they are scattered (not held in registers through the ranking).  Measured
// on the large workload (84M pairs, 26-bit keys, 3 passes): 8 pairs per
// thread 0.690 ms per pass; 16 with late payloads 0.553 ms (tile overheads
// -- counter zeroing, 512-digit scans and look-back -- spread over twice the
// pairs, still two 512-thread CTAs per SM).
#ifndef TBE_SORT_IPT
#define TBE_SORT_IPT 16
#endif
#ifndef TBE_SORT_LATE_VALS
#define TBE_SORT_LATE_VALS 1
#endif
// pairs per thread and per tile: 64-bit keys keep 8 per thread (registers)
template <typename KeyT> struct SortShape {
    static constexpr int IPT = sizeof(KeyT) == 8 ? 8 : TBE_SORT_IPT;
    static constexpr int TILE = SORT_THREADS * IPT;
};
constexpr int MIN_TILE = SORT_THREADS * 8;   // the workspace is sized for the smallest tile
constexpr uint32_t ST_AGG = 1u << 30;
constexpr uint32_t ST_INC = 2u << 30;
constexpr uint32_t ST_MASK = (1u << 30) - 1;
constexpr int MAX_PASSES = 8;   // 64-bit keys: at most 7 passes of 9 bits
#ifndef TBE_SORT_LOOKBACK
#define TBE_SORT_LOOKBACK 8
#endif
// predecessors read per look-back round trip (large workload, 16 pairs per
// thread: 0.545 ms per pass at 8, 0.584 at 16, 0.637 at 32; one CTA per SM
// instead of two, for a shorter look-back: 0.827; persistent CTAs taking
// the next ticket during the current tile instead of a CTA per tile: 0.648)
constexpr int LOOKBACK = TBE_SORT_LOOKBACK;

static int num_passes(int key_bits) { return (key_bits + MAX_DIGIT_BITS - 1) / MAX_DIGIT_BITS; }
static int digit_bits(int key_bits) {
    const int p = num_passes(key_bits);
    return p > 0 ? (key_bits + p - 1) / p : 0;
}

struct SortWs {
    uint32_t *hist;        // [MAX_PASSES][RADIX] digit counts, then bucket starts
    uint32_t *tickets;     // [MAX_PASSES] tile tickets
    uint32_t *status;      // [MAX_PASSES][ntiles][RADIX] look-back words
    int64_t ntiles;
};

static SortWs carve(void *ws, int64_t N, int tile) {
    SortWs s;
    s.ntiles = (N + tile - 1) / tile;
    char *p = (char *)ws;
    s.hist = (uint32_t *)p;
    p += MAX_PASSES * RADIX * 4;
    s.tickets = (uint32_t *)p;
    p += 256;
    s.status = (uint32_t *)p;
    return s;
}

size_t sort_workspace_bytes(int64_t N, int key_bits) {
    const int64_t ntiles = (N + MIN_TILE - 1) / MIN_TILE;
    int passes = num_passes(key_bits);
    if (passes < 1) passes = 1;
    return MAX_PASSES * RADIX * 4 + 256 + (size_t)passes * ntiles * RADIX * 4 + 256;
}

// 16-byte vector of keys
template <typename KeyT> struct KeyVec;
template <> struct KeyVec<uint32_t> {
    static constexpr int K = 4;
    static __device__ __forceinline__ void load(const uint32_t *p, int64_t i, uint32_t (&k)[4]) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p) + i);
        k[0] = v.x; k[1] = v.y; k[2] = v.z; k[3] = v.w;
    }
};
template <> struct KeyVec<uint64_t> {
    static constexpr int K = 2;
    static __device__ __forceinline__ void load(const uint64_t *p, int64_t i, uint64_t (&k)[2]) {
        const ulonglong2 v = __ldg(reinterpret_cast<const ulonglong2 *>(p) + i);
        k[0] = v.x; k[1] = v.y;
    }
};

template <typename KeyT>
__global__ void __launch_bounds__(256) radix_hist_kernel(const KeyT *__restrict__ keys, int64_t N,
                                                         int passes, int bits, uint32_t *hist,
                                                         uint32_t *zero, int64_t zero_words) {
    constexpr int K = KeyVec<KeyT>::K;
    const uint32_t mask = (1u << bits) - 1;
    __shared__ uint32_t sh[MAX_PASSES * RADIX];
    for (int i = threadIdx.x; i < MAX_PASSES * RADIX; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t NV = N / K;
    for (int64_t i = tid; i < NV; i += stride) {
        KeyT kk[K];
        KeyVec<KeyT>::load(keys, i, kk);
#pragma unroll
        for (int e = 0; e < K; ++e)
            for (int ps = 0; ps < passes; ++ps)
                atomicAdd(&sh[ps * RADIX + (uint32_t)((kk[e] >> (ps * bits)) & mask)], 1u);
    }
    for (int64_t i = NV * K + tid; i < N; i += stride) {
        const KeyT k = __ldg(keys + i);
        for (int ps = 0; ps < passes; ++ps)
            atomicAdd(&sh[ps * RADIX + (uint32_t)((k >> (ps * bits)) & mask)], 1u);
    }
    for (int64_t i = tid; i < zero_words; i += stride) zero[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < passes * RADIX; i += blockDim.x)
        if (sh[i]) atomicAdd(&hist[i], sh[i]);
}

// Exclusive scan of one pass's RADIX digit counts into bucket starts, in place.
__global__ void __launch_bounds__(RADIX) radix_bucket_kernel(uint32_t *hist) {
    __shared__ uint32_t s[RADIX];
    uint32_t *h = hist + blockIdx.x * RADIX;
    const int d = threadIdx.x;
    s[d] = h[d];
    __syncthreads();
    for (int off = 1; off < RADIX; off <<= 1) {
        uint32_t v = d >= off ? s[d - off] : 0;
        __syncthreads();
        s[d] += v;
        __syncthreads();
    }
    h[d] = s[d] - h[d];
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// per-warp digit counts, then exclusive warp prefixes within the tile: both
// below 2^16 (a tile holds at most 16384 pairs), so 16-bit counters suffice
#ifndef TBE_SORT_CNT16
#define TBE_SORT_CNT16 1   // 0.546 vs 0.554 ms per pass with 32-bit counters
#endif
using WarpCnt = std::conditional_t<TBE_SORT_CNT16 != 0, uint16_t, uint32_t>;
template <typename KeyT> struct PassSmem {
    KeyT keys[SortShape<KeyT>::TILE];
    uint32_t vals[SortShape<KeyT>::TILE];
    WarpCnt warp_cnt[SORT_WARPS][RADIX];   // counts, then exclusive warp prefixes
    uint32_t count[RADIX];
    uint32_t local_off[RADIX];
    uint32_t global_base[RADIX];
    uint32_t warp_tot[RADIX / 32];
    uint32_t tile;
};

template <typename KeyT>
__global__ void __launch_bounds__(SORT_THREADS, 2)
radix_onesweep_kernel(const KeyT *__restrict__ keys_in, const uint32_t *__restrict__ vals_in,
                      KeyT *__restrict__ keys_out, uint32_t *__restrict__ vals_out, int64_t N,
                      int shift, uint32_t mask, const uint32_t *__restrict__ bucket, uint32_t *status,
                      uint32_t *ticket, int32_t *err) {
    constexpr int IPT = SortShape<KeyT>::IPT;
    constexpr int TILE = SortShape<KeyT>::TILE;
    constexpr bool LATE = TBE_SORT_LATE_VALS != 0;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    PassSmem<KeyT> &S = *reinterpret_cast<PassSmem<KeyT> *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) S.tile = atomicAdd(ticket, 1u);
    static_assert(SortShape<KeyT>::TILE <= 16384, "16-bit warp counters");
    for (int i = tid; i < (int)(sizeof(S.warp_cnt) / 4); i += SORT_THREADS)
        reinterpret_cast<uint32_t *>(&S.warp_cnt[0][0])[i] = 0;
    __syncthreads();
    const int64_t tile = S.tile;
    const int64_t tile_base = tile * TILE;

    // warp-striped load: item i of lane l in warp w sits at tile position
    // w*32*IPT + i*32 + l, so (i, lane) order within a warp is input order
    KeyT k[IPT];
    uint32_t v[LATE ? 1 : IPT], rank[IPT];
#pragma unroll
    for (int i = 0; i < IPT; ++i) {
        const int64_t pos = tile_base + warp * 32 * IPT + i * 32 + lane;
        const bool ok = pos < N;
        k[i] = ok ? __ldg(keys_in + pos) : ~KeyT(0);
        if constexpr (!LATE) v[i] = ok ? __ldg(vals_in + pos) : 0u;
    }
    const unsigned lt = lanemask_lt();
#pragma unroll
    for (int i = 0; i < IPT; ++i) {
        const int64_t pos = tile_base + warp * 32 * IPT + i * 32 + lane;
        const uint32_t d = pos < N ? (uint32_t)((k[i] >> shift) & mask) : RADIX;   // RADIX = padding
        // (per-bit ballots instead measured 0.625 vs 0.552 ms per pass)
        const unsigned peers = __match_any_sync(FULL, d);
        const int leader = __ffs(peers) - 1;
        uint32_t base = 0;
        if (lane == leader && d < RADIX) {
            base = S.warp_cnt[warp][d];
            S.warp_cnt[warp][d] = (WarpCnt)(base + __popc(peers));
        }
        base = __shfl_sync(FULL, base, leader);
        rank[i] = base + __popc(peers & lt);
        __syncwarp();
    }
    __syncthreads();

    // per digit (thread d < RADIX): tile count and exclusive prefix over warps,
    // then the look-back for the digit's prefix over earlier tiles
    const int d = tid;
    uint32_t sum = 0, x = 0;
    if (d < RADIX) {
#pragma unroll
        for (int w = 0; w < SORT_WARPS; ++w) {
            const uint32_t c = S.warp_cnt[w][d];
            S.warp_cnt[w][d] = (WarpCnt)sum;
            sum += c;
        }
        S.count[d] = sum;

        uint32_t excl = 0;
        uint32_t *st = status + tile * RADIX + d;
        if (tile == 0) {
            st_relaxed_u32(st, ST_INC | sum);
        } else {
            st_relaxed_u32(st, ST_AGG | sum);
            // look back LOOKBACK predecessors per round trip: add aggregates
            // in order until an inclusive prefix (or tile 0); stop at the
            // first tile that has published nothing yet and poll it again
            int64_t j = tile - 1;
            uint64_t t0 = 0;
            while (true) {
                uint32_t sv[LOOKBACK];
#pragma unroll
                for (int q = 0; q < LOOKBACK; ++q)
                    sv[q] = j - q >= 0 ? ld_relaxed_u32(status + (j - q) * RADIX + d) : 0u;
                int used = 0;
                bool done = false;
#pragma unroll
                for (int q = 0; q < LOOKBACK; ++q) {
                    if (done || used < q) break;
                    const uint32_t f = sv[q] & ~ST_MASK;
                    if (f == 0) break;
                    excl += sv[q] & ST_MASK;
                    used = q + 1;
                    done = f == ST_INC || j - q == 0;
                }
                if (done) break;
                j -= used;
                if (used == 0) {
                    const uint64_t now = global_ns();
                    if (t0 == 0) t0 = now;
                    else if (now - t0 > WAIT_LIMIT_NS) {
                        atomicOr(err, TBE_FLAG_SORT_TIMEOUT);
                        break;
                    }
                    __nanosleep(64);
                }
            }
            st_relaxed_u32(st, ST_INC | (excl + sum));
        }
        S.global_base[d] = __ldg(bucket + d) + excl;

        // exclusive scan of the tile's digit counts (warp scans + warp totals)
        x = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(FULL, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) S.warp_tot[warp] = x;
    }
    __syncthreads();
    if (d < RADIX) {
        uint32_t wp = 0;
        for (int w = 0; w < warp; ++w) wp += S.warp_tot[w];
        S.local_off[d] = wp + x - sum;
    }
    __syncthreads();

    // reorder the tile by digit in shared memory
#pragma unroll
    for (int i = 0; i < IPT; ++i) {
        const int64_t pos = tile_base + warp * 32 * IPT + i * 32 + lane;
        if (pos < N) {
            const uint32_t d = (uint32_t)((k[i] >> shift) & mask);
            const uint32_t lp = S.local_off[d] + S.warp_cnt[warp][d] + rank[i];
            S.keys[lp] = k[i];
            if constexpr (LATE) S.vals[lp] = __ldg(vals_in + pos);
            else S.vals[lp] = v[i];
        }
    }
    __syncthreads();

    const int64_t rem = N - tile_base;
    const int n = rem < TILE ? (int)rem : TILE;
    for (int j = tid; j < n; j += SORT_THREADS) {
        const KeyT key = S.keys[j];
        const uint32_t d = (uint32_t)((key >> shift) & mask);
        const uint32_t gp = S.global_base[d] + (j - S.local_off[d]);
        if ((int64_t)gp < N) {   // always true unless a look-back gave up (flagged)
            keys_out[gp] = key;
            vals_out[gp] = S.vals[j];
        }
    }
}

__global__ void fill_u32_kernel(uint32_t *p, int64_t n, uint32_t v) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        p[i] = v;
}

template <typename KeyT>
static void sort_passes(Launch &L, KeyT *keys_a, uint32_t *vals_a, KeyT *keys_b, uint32_t *vals_b,
                        int64_t N, int passes, int bits, const SortWs &s, int32_t *status) {
    const int64_t zero_words = (int64_t)passes * s.ntiles * RADIX;
    L.before("tbe_sort_zero");
    fill_u32_kernel<<<1, 256, 0, L.stream>>>(s.hist, MAX_PASSES * RADIX + 64, 0u);
    L.after();

    const int64_t nvec = N / KeyVec<KeyT>::K;
    int hist_grid = (int)((nvec + 255) / 256);
    if (hist_grid > L.num_sms * 4) hist_grid = L.num_sms * 4;
    if (hist_grid < 1) hist_grid = 1;
    L.before("tbe_sort_histogram");
    radix_hist_kernel<KeyT><<<hist_grid, 256, 0, L.stream>>>(keys_a, N, passes, bits, s.hist, s.status,
                                                             zero_words);
    L.after();
    L.before("tbe_sort_buckets");
    radix_bucket_kernel<<<passes, RADIX, 0, L.stream>>>(s.hist);
    L.after();

    const size_t smem = sizeof(PassSmem<KeyT>);
    static_assert(sizeof(PassSmem<uint64_t>) * 2 < 227 * 1024 && sizeof(PassSmem<uint32_t>) * 2 < 227 * 1024,
                  "two pass CTAs per SM");
    cached_smem_attr(L.dev, (const void *)radix_onesweep_kernel<KeyT>, smem);
    const KeyT *ki = keys_a;
    const uint32_t *vi = vals_a;
    KeyT *ko = keys_b;
    uint32_t *vo = vals_b;
    for (int ps = 0; ps < passes; ++ps) {
        L.before("tbe_sort_onesweep");
        radix_onesweep_kernel<KeyT><<<(unsigned)s.ntiles, SORT_THREADS, smem, L.stream>>>(
            ki, vi, ko, vo, N, ps * bits, (1u << bits) - 1, s.hist + ps * RADIX,
            s.status + (int64_t)ps * s.ntiles * RADIX, s.tickets + ps, status + 1);
        L.after();
        const KeyT *tk = ko;
        const uint32_t *tv = vo;
        ko = const_cast<KeyT *>(ki);
        vo = const_cast<uint32_t *>(vi);
        ki = tk;
        vi = tv;
    }
}

tbe_status launch_sort(Launch &L, void *keys_a, uint32_t *vals_a, void *keys_b, uint32_t *vals_b,
                       int64_t N, int key_bits, int key_bytes, void *ws, int32_t *status,
                       bool *in_b) {
    const int passes = num_passes(key_bits);
    const int bits = digit_bits(key_bits);
    *in_b = (passes & 1) != 0;
    if (N == 0 || passes == 0) {
        *in_b = false;
        return TBE_OK;
    }
    if (passes > MAX_PASSES) return TBE_ERR_KEY_RANGE;
    const SortWs s = carve(ws, N, key_bytes == 8 ? SortShape<uint64_t>::TILE : SortShape<uint32_t>::TILE);
    if (key_bytes == 8)
        sort_passes<uint64_t>(L, (uint64_t *)keys_a, vals_a, (uint64_t *)keys_b, vals_b, N, passes, bits,
                              s, status);
    else
        sort_passes<uint32_t>(L, (uint32_t *)keys_a, vals_a, (uint32_t *)keys_b, vals_b, N, passes, bits,
                              s, status);
    return TBE_OK;
}

// ---------------------------------------------------------------------------
// Self-test of the look-back's time limit.  Two tiles of zero keys; the tile
// ticket starts at 1, so the one CTA launched takes tile 1 and looks back at
// tile 0, which no CTA will ever publish.  After WAIT_LIMIT_NS the CTA sets
// TBE_FLAG_SORT_TIMEOUT and finishes its tile (every write stays inside the
// two-tile buffers; the output is invalid, as the flag says).  No copy is in
// flight during the wait.

constexpr int64_t SELFTEST_N = 2 * SortShape<uint32_t>::TILE;

size_t sort_selftest_bytes() {
    return (size_t)4 * SELFTEST_N * 4 + RADIX * 4 + 2 * RADIX * 4 + 256;
}

__global__ void sort_selftest_init_kernel(uint32_t *words, int64_t n, uint32_t *ticket) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        words[i] = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 1;
}

tbe_status launch_sort_selftest(Launch &L, void *ws, int32_t *status) {
    uint32_t *w = (uint32_t *)ws;
    uint32_t *keys_in = w, *vals_in = w + SELFTEST_N, *keys_out = w + 2 * SELFTEST_N,
             *vals_out = w + 3 * SELFTEST_N;
    uint32_t *bucket = w + 4 * SELFTEST_N;
    uint32_t *look = bucket + RADIX;
    uint32_t *ticket = look + 2 * RADIX;
    const int64_t words = 4 * SELFTEST_N + 3 * RADIX;
    L.before("tbe_selftest_init");
    sort_selftest_init_kernel<<<8, 256, 0, L.stream>>>(w, words, ticket);
    L.after();
    const size_t smem = sizeof(PassSmem<uint32_t>);
    cached_smem_attr(L.dev, (const void *)radix_onesweep_kernel<uint32_t>, smem);
    L.before("tbe_sort_onesweep");
    radix_onesweep_kernel<uint32_t><<<1, SORT_THREADS, smem, L.stream>>>(
        keys_in, vals_in, keys_out, vals_out, SELFTEST_N, 0, RADIX - 1, bucket, look, ticket,
        status + 1);
    L.after();
    return TBE_OK;
}

}  // namespace tbe
