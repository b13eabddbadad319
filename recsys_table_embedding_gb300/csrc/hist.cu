// Small-table histogram path on the 5th-generation tensor cores.
//
// FBTriton TBE redesign (accesspath.com), "Forward state reuse and
// preprocessing": the forward saves per-bag histogram counts; the backward
// uses those counts for a compensated FP16 high/low GEMM to FP32, then applies
// the optimizer; forward and backward stay separate launches and only the
// counts are reused.  Decision checklist item 2: the path covers E <= 64,
// 64 <= D <= 128, L >= 64, FP16 weights and no per-sample weights.
//
// Forward (per CTA: a contiguous range of 128-bag tiles of the tables):
//   the tile's lookups, one contiguous CSR range, are read warp by warp (a
//   warp takes 4 bags at a time, its lanes consecutive lookups of each) and
//   counted into shared memory (H[b][e], b < 128, e < 64), the counts are
//   written to the A operand as FP16 (exact: counts <= 2048) in the 128-byte
//   swizzled K-major layout and saved to global memory, and one tcgen05.mma
//   chain (M = 128 bags, N = D, K = 64 rows, FP32 accumulation in TMEM)
//   computes out_t = H_t * W_t with W_t^T staged as the B operand.  The
//   accumulator is read back with tcgen05.ld and stored to out[b, t*D + d].
// Backward (per CTA: one table and one slice of its bags; K-split):
//   gW_t^T = G_t^T * H_t with G split into hi = fp16(G), lo = fp16(G - hi):
//   both products accumulate into one FP32 TMEM accumulator (M = 128 >= D,
//   N = 64 rows, K = 64 bags per step), with the next step's operands staged
//   into the other shared-memory buffer while the tensor core runs.  The
//   slice's partial and its per-row counts go to the workspace; the CTA that
//   arrives last for a table (device-scope fence + arrival counter) sums the
//   slices in order and applies exact rowwise Adagrad to every row with a
//   nonzero count.
//
// Every mbarrier wait is bounded; on a timeout the CTA flags
// TBE_FLAG_MMA_TIMEOUT, stops issuing work, and still frees its TMEM.
#include <algorithm>

#include "tbe_internal.cuh"

namespace tbe {

constexpr int HE = 64;          // rows per table covered (K of the forward)
constexpr int HT_BAGS = 128;    // bags per forward tile (M)
#ifndef TBE_HIST_CB
#define TBE_HIST_CB 8   // bags a warp counts at a time (0.99 ms vs 1.08 at 4, 1.25 at 16)
#endif
#ifndef TBE_HIST_CU
#define TBE_HIST_CU 1   // 32-lookup loads per bag and lane in flight
#endif
constexpr int HF_THREADS = 256;
constexpr int HB_THREADS = 256;
constexpr int HB_KBAGS = 64;    // bags per backward K step
constexpr int CNT_STRIDE = HE / 2 + 1;   // 16-bit count pairs per bag, +1 word against bank conflicts

// ------------------------------------------------------------ PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// bounded wait on the phase with the given parity; false on timeout
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    return mbar_wait_bounded(smem_u32(bar), parity);
}
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16, one CTA
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on `bar` when all previously issued tcgen05.mma of this thread complete
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}
// 32 lanes x 8 consecutive 32-bit columns
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes (64 FP16 along K), 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address, 16-byte units
    d |= (uint64_t)1 << 16;                      // leading byte offset (unused when swizzled)
    d |= (uint64_t)(1024 >> 4) << 32;            // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;                      // descriptor version for this architecture
    d |= (uint64_t)2 << 61;                      // 128-byte swizzle
    return d;
}
// Instruction descriptor: FP16 x FP16 -> FP32, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// byte offset of element (row, k) in a [rows][64] FP16 K-major SW128 tile
__device__ __forceinline__ uint32_t sw128_off(int row, int k) {
    return (uint32_t)(row * 128 + ((((k >> 3) ^ (row & 7))) << 4) + (k & 7) * 2);
}

// ------------------------------------------------------------ forward

struct HistFwdParams {
    const __half *W;
    const int64_t *table_offset;
    const void *indices;  // IdxT [N]
    const void *offsets;  // IdxT [T*B+1]
    float *out;
    uint16_t *hist;       // nullable
    int32_t *status;
    int32_t *counters;    // nullable: C_MALFORMED / C_DECREASING
    int64_t B;
    int64_t N;
    int T;
    int D;
    int64_t tiles_per_table;
    int64_t tiles_total;
    int64_t tiles_per_cta;
    int do_mma;
};

constexpr int STG_PITCH = 36;   // floats per staged output row (32 + 4 against bank conflicts)

struct HistFwdSmem {
    // A and cnt are contiguous: after the MMA, they serve as the staging
    // buffer of the output ([128 bags][STG_PITCH] floats)
    alignas(1024) unsigned char A[HT_BAGS * 128];   // counts as FP16, [128 bags][64 rows]
    uint32_t cnt[HT_BAGS * CNT_STRIDE];             // two 16-bit counts per word
    alignas(1024) unsigned char Bm[128 * 128];      // W_t^T, [D][64 rows]
    int32_t bs[HT_BAGS], be[HT_BAGS];               // lookup range of each bag (empty if malformed)
    uint64_t mbar;
    uint32_t tmem_base;
};

template <typename IdxT>
__global__ void __launch_bounds__(HF_THREADS) tbe_hist_fwd_kernel(const HistFwdParams p) {
    extern __shared__ unsigned char smem_raw[];
    const IdxT *offsets = reinterpret_cast<const IdxT *>(p.offsets);
    const IdxT *indices = reinterpret_cast<const IdxT *>(p.indices);
    // 1024-byte alignment of the operand tiles (the swizzle pattern is anchored there)
    HistFwdSmem &S = *reinterpret_cast<HistFwdSmem *>(
        (void *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t tile0 = (int64_t)blockIdx.x * p.tiles_per_cta;
    int64_t tile1 = tile0 + p.tiles_per_cta;
    if (tile1 > p.tiles_total) tile1 = p.tiles_total;

    if (p.do_mma) {
        if (warp == 0) {
            tmem_alloc(&S.tmem_base, 128);
            tmem_relinquish();
        }
        if (tid == 0) {
            mbar_init(&S.mbar, 1);
            fence_mbar_init();
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = p.do_mma ? S.tmem_base : 0;
    const uint32_t idesc = idesc_f16_f32(128, p.D);
    uint32_t phase = 0;
    bool alive = true;
    int cur_t = -1;
    int oob = 0;
    // offsets[0] != 0 or offsets[T*B] != N leaves lookups outside every bag
    if (blockIdx.x == 0 && tid == 0 &&
        ((int64_t)__ldg(offsets) != 0 || (int64_t)__ldg(offsets + p.T * p.B) != p.N)) {
        atomicOr(p.status + 1, TBE_FLAG_BAD_OFFSETS);
        if (p.counters != nullptr) p.counters[C_MALFORMED] = 1;
    }

    for (int64_t tile = tile0; tile < tile1 && alive; ++tile) {
        const int t = (int)(tile / p.tiles_per_table);
        const int64_t b0 = (tile - (int64_t)t * p.tiles_per_table) * HT_BAGS;
        const int nb = (int)min((int64_t)HT_BAGS, p.B - b0);
        const int64_t row0 = __ldg(p.table_offset + t);
        const int64_t E = __ldg(p.table_offset + t + 1) - row0;
        const int64_t g0 = (int64_t)t * p.B + b0;

        // stage W_t^T as the B operand when the table changes
        if (p.do_mma && t != cur_t) {
            for (int i = tid; i < 128 * HE; i += HF_THREADS) {
                const int d = i % 128, e = i / 128;
                __half v = __float2half(0.f);
                if (d < p.D && e < E) v = p.W[(row0 + e) * p.D + d];
                *reinterpret_cast<__half *>(S.Bm + sw128_off(d, e)) = v;
            }
            cur_t = t;
        }
        for (int i = tid; i < HT_BAGS * CNT_STRIDE; i += HF_THREADS) S.cnt[i] = 0;
        if (tid < HT_BAGS) {
            // a well-formed bag has 0 <= start <= end <= N; any other is empty
            int64_t s0 = 0, s1 = 0;
            if (tid < nb) {
                s0 = (int64_t)__ldg(offsets + g0 + tid);
                s1 = (int64_t)__ldg(offsets + g0 + tid + 1);
                if (!(s0 <= s1 && s0 >= 0 && s1 <= p.N)) {
                    atomicOr(p.status + 1, TBE_FLAG_BAD_OFFSETS);
                    if (p.counters != nullptr) {
                        p.counters[C_MALFORMED] = 1;
                        if (s1 < s0) p.counters[C_DECREASING] = 1;
                    }
                    s0 = s1 = 0;
                }
            }
            S.bs[tid] = (int32_t)s0;
            S.be[tid] = (int32_t)s1;
        }
        __syncthreads();
        // count the tile's lookups: a warp takes CB bags at a time and its
        // lanes read CU*32 consecutive lookups of each (CB*CU loads in flight
        // per lane); every lookup adds one to its bag's 16-bit row counter
        // (16-byte vector reads of the indices measured slower: 1.29 vs
        // 1.00 ms on the histogram workload)
        {
            constexpr int CB = TBE_HIST_CB, CU = TBE_HIST_CU;
            constexpr int NW = HF_THREADS / 32;
            for (int r0 = warp * CB; r0 < nb; r0 += NW * CB) {
                int32_t bs[CB], be[CB];
                int32_t maxlen = 0;
#pragma unroll
                for (int j = 0; j < CB; ++j) {
                    const int r = r0 + j;
                    bs[j] = r < nb ? S.bs[r] : 0;
                    be[j] = r < nb ? S.be[r] : 0;
                    maxlen = max(maxlen, be[j] - bs[j]);
                }
                for (int32_t k = 0; k < maxlen; k += 32 * CU) {
                    IdxT v[CB][CU];
#pragma unroll
                    for (int j = 0; j < CB; ++j)
#pragma unroll
                        for (int u = 0; u < CU; ++u) {
                            const int32_t pos = bs[j] + k + u * 32 + lane;
                            v[j][u] = pos < be[j] ? __ldg(indices + pos) : IdxT(0);
                        }
#pragma unroll
                    for (int j = 0; j < CB; ++j)
#pragma unroll
                        for (int u = 0; u < CU; ++u) {
                            const int32_t pos = bs[j] + k + u * 32 + lane;
                            if (pos >= be[j]) continue;
                            const IdxT idx = v[j][u];
                            if (idx >= 0 && (int64_t)idx < E)
                                atomicAdd(&S.cnt[(r0 + j) * CNT_STRIDE + (int)(idx >> 1)],
                                          1u << ((int)(idx & 1) * 16));
                            else
                                ++oob;
                        }
                }
            }
        }
        __syncthreads();
        // counts -> FP16 A operand (+ saved histogram); thread = (row r, half h)
        {
            const int r = tid & (HT_BAGS - 1), h = tid >> 7;
            // a 16-bit count could wrap only in a bag of more than 65535 lookups
            int over = h == 0 && r < nb && S.be[r] - S.bs[r] > 65535;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int c = h * 4 + cc;
                uint32_t packed[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t pair = S.cnt[r * CNT_STRIDE + c * 4 + q];
                    const uint32_t c0 = pair & 0xFFFFu, c1 = pair >> 16;
                    over |= (c0 > 2048u) | (c1 > 2048u);
                    __half2 hv = __halves2half2(__uint2half_rn(c0), __uint2half_rn(c1));
                    packed[q] = *reinterpret_cast<uint32_t *>(&hv);
                }
                const uint4 v = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                if (p.do_mma)
                    *reinterpret_cast<uint4 *>(S.A + r * 128 + ((c ^ (r & 7)) << 4)) = v;
                if (p.hist != nullptr && r < nb)
                    *reinterpret_cast<uint4 *>(p.hist + (g0 + r) * HE + c * 8) = v;
            }
            if (over) atomicOr(p.status + 1, TBE_FLAG_HIST_COUNT);
        }
        if (!p.do_mma) {
            __syncthreads();
            continue;
        }
        fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t a = smem_u32(S.A), b = smem_u32(S.Bm);
#pragma unroll
            for (int k = 0; k < HE / 16; ++k)
                umma_f16(tmem, desc_sw128(a + k * 32), desc_sw128(b + k * 32), idesc, k > 0);
            umma_commit(&S.mbar);
        }
        __syncwarp();
        // block-uniform outcome of the bounded wait
        const bool done = __syncthreads_and(mbar_wait(&S.mbar, phase)) != 0;
        phase ^= 1;
        tc_fence_after();
        if (!done) {
            if (lane == 0) atomicOr(p.status + 1, TBE_FLAG_MMA_TIMEOUT);
            alive = false;
        } else {
            // epilogue, 32 columns per pass: TMEM -> shared staging (warp w
            // reads lanes 32*(w%4).. of columns +16*(w/4)), then full output
            // row segments written by consecutive threads (coalesced)
            static_assert(HT_BAGS * STG_PITCH * 4 <= HT_BAGS * 128 + HT_BAGS * CNT_STRIDE * 4,
                          "output staging fits in A + cnt");
            float *stg = reinterpret_cast<float *>(S.A);
            const int q = warp & 3, hh = warp >> 2;
            for (int pc = 0; pc * 32 < p.D; ++pc) {
                const int ncols = min(32, p.D - pc * 32);
                if (hh * 16 < ncols) {   // warp-uniform
#pragma unroll
                    for (int c8 = 0; c8 < 2; ++c8) {
                        uint32_t r[8];
                        tmem_ld8(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(pc * 32 + hh * 16 + c8 * 8), r);
                        tmem_wait_ld();
                        float4 *dst = reinterpret_cast<float4 *>(stg + (q * 32 + lane) * STG_PITCH + hh * 16 + c8 * 8);
                        dst[0] = make_float4(__uint_as_float(r[0]), __uint_as_float(r[1]),
                                             __uint_as_float(r[2]), __uint_as_float(r[3]));
                        dst[1] = make_float4(__uint_as_float(r[4]), __uint_as_float(r[5]),
                                             __uint_as_float(r[6]), __uint_as_float(r[7]));
                    }
                }
                __syncthreads();
                const int per_row = ncols / 4;
                for (int i = tid; i < HT_BAGS * per_row; i += HF_THREADS) {
                    const int row = i / per_row, c4 = i - row * per_row;
                    if (row < nb)
                        __stcs(reinterpret_cast<float4 *>(p.out + (b0 + row) * (int64_t)p.T * p.D +
                                                          (int64_t)t * p.D + pc * 32) + c4,
                               *reinterpret_cast<const float4 *>(stg + row * STG_PITCH + c4 * 4));
                }
                __syncthreads();
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    oob += __shfl_xor_sync(FULL, oob, 16);
    oob += __shfl_xor_sync(FULL, oob, 8);
    oob += __shfl_xor_sync(FULL, oob, 4);
    oob += __shfl_xor_sync(FULL, oob, 2);
    oob += __shfl_xor_sync(FULL, oob, 1);
    if (lane == 0 && oob && p.do_mma) atomicAdd(p.status, oob);
    if (p.do_mma) {
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp == 0) tmem_dealloc(tmem, 128);
    }
}

// ------------------------------------------------------------ backward

struct HistBwdParams {
    __half *W;
    float *mom;
    const float *G;
    const uint16_t *hist;
    const int64_t *table_offset;
    float *part;          // [T][S][64][D] FP32 slice partials
    float *cnt;           // [T][S][64] slice counts
    int32_t *arrive;      // [T]
    int32_t *status;
    const int32_t *counters;   // nullable: no update when C_DECREASING is set
    int64_t B;
    int T;
    int D;
    int S;
    int64_t kbags;        // bags per slice (multiple of 64)
    float lr;
    float eps;
};

struct HistBwdStage {
    alignas(1024) unsigned char Ahi[128 * 128];   // G^T hi: [128 d][64 bags]
    alignas(1024) unsigned char Alo[128 * 128];   // G^T lo
    alignas(1024) unsigned char Bh[HE * 128];     // H^T:   [64 rows][64 bags]
};
struct HistBwdSmem {
    HistBwdStage st[2];
    uint64_t mbar[2];
    uint32_t tmem_base;
    float cnt_part[HB_THREADS];
    int is_last;
};

__global__ void __launch_bounds__(HB_THREADS) tbe_hist_bwd_kernel(const HistBwdParams p) {
    extern __shared__ unsigned char smem_raw[];
    HistBwdSmem &S = *reinterpret_cast<HistBwdSmem *>(
        (void *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t = blockIdx.x / p.S, s = blockIdx.x % p.S;
    const int64_t bb = (int64_t)s * p.kbags;
    int64_t be = bb + p.kbags;
    if (be > p.B) be = p.B;
    const int nsteps = be > bb ? (int)((be - bb + HB_KBAGS - 1) / HB_KBAGS) : 0;
    const int64_t TD = (int64_t)p.T * p.D;
    // offsets that decrease leave lookups in two bags: no backward update
    if (p.counters != nullptr && __ldg(p.counters + C_DECREASING) != 0) return;

    if (warp == 0) {
        tmem_alloc(&S.tmem_base, 64);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&S.mbar[0], 1);
        mbar_init(&S.mbar[1], 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    const uint32_t idesc = idesc_f16_f32(128, HE);
    uint32_t ph[2] = {0, 0};
    bool alive = true;
    float mycnt = 0.f;
    int over = 0;

    // Operands of one K step held in registers: 32 gradient values of one
    // column d (8-bag chunks jc, jc+2, jc+4, jc+6) and 16 counts of one row e
    // (chunks je, je+4).  The next step's loads are issued before this step's
    // barrier and MMA issue, so their latency overlaps them.
    const int gd = tid & 127, gjc = tid >> 7;
    const int he = tid & 63, hjc = tid >> 6;
    float gv[32];
    uint16_t hv[16];
    auto load_step = [&](int i) {
        const int64_t k0 = bb + (int64_t)i * HB_KBAGS;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
            for (int z = 0; z < 8; ++z) {
                const int64_t b = k0 + (gjc + 2 * cc) * 8 + z;
                gv[cc * 8 + z] = (gd < p.D && b < be) ? __ldg(p.G + b * TD + (int64_t)t * p.D + gd) : 0.f;
            }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
            for (int z = 0; z < 8; ++z) {
                const int64_t b = k0 + (hjc + 4 * cc) * 8 + z;
                hv[cc * 8 + z] = b < be ? __ldg(p.hist + ((int64_t)t * p.B + b) * HE + he) : (uint16_t)0;
            }
    };
    if (nsteps > 0) load_step(0);
    for (int i = 0; i < nsteps && alive; ++i) {
        const int st = i & 1;
        HistBwdStage &SG = S.st[st];
        if (i >= 2) {   // the MMAs of step i-2 read this stage
            if (!__syncthreads_and(mbar_wait(&S.mbar[st], ph[st]))) {
                alive = false;   // block-uniform
                if (tid == 0) atomicOr(p.status + 1, TBE_FLAG_MMA_TIMEOUT);
                break;
            }
            ph[st] ^= 1;
            tc_fence_after();
        }
        // G^T hi/lo into the A tiles: 8 consecutive bags per 16-byte chunk
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int c = gjc + 2 * cc;
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float g0 = gv[cc * 8 + 2 * q], g1 = gv[cc * 8 + 2 * q + 1];
                over |= (fabsf(g0) > 65504.f) | (fabsf(g1) > 65504.f);
                const __half h0 = __float2half_rn(g0), h1 = __float2half_rn(g1);
                const __half l0 = __float2half_rn(g0 - __half2float(h0));
                const __half l1 = __float2half_rn(g1 - __half2float(h1));
                __half2 hh = __halves2half2(h0, h1), ll = __halves2half2(l0, l1);
                hw[q] = *reinterpret_cast<uint32_t *>(&hh);
                lw[q] = *reinterpret_cast<uint32_t *>(&ll);
            }
            const uint32_t off = (uint32_t)(gd * 128 + ((c ^ (gd & 7)) << 4));
            *reinterpret_cast<uint4 *>(SG.Ahi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4 *>(SG.Alo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        // H^T into the B tile; counts summed per row
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int c = hjc + 4 * cc;
            const uint16_t *h8 = hv + cc * 8;
#pragma unroll
            for (int z = 0; z < 8; ++z) mycnt += __half2float(__ushort_as_half(h8[z]));
            uint4 v;
            v.x = h8[0] | ((uint32_t)h8[1] << 16);
            v.y = h8[2] | ((uint32_t)h8[3] << 16);
            v.z = h8[4] | ((uint32_t)h8[5] << 16);
            v.w = h8[6] | ((uint32_t)h8[7] << 16);
            *reinterpret_cast<uint4 *>(SG.Bh + he * 128 + ((c ^ (he & 7)) << 4)) = v;
        }
        if (i + 1 < nsteps) load_step(i + 1);
        fence_async_smem();
        __syncthreads();
        if (tid == 0 && alive) {
            tc_fence_after();
            const uint32_t ah = smem_u32(SG.Ahi), al = smem_u32(SG.Alo), bh = smem_u32(SG.Bh);
#pragma unroll
            for (int k = 0; k < HB_KBAGS / 16; ++k) {
                umma_f16(tmem, desc_sw128(ah + k * 32), desc_sw128(bh + k * 32), idesc,
                         (i > 0 || k > 0) ? 1u : 0u);
                umma_f16(tmem, desc_sw128(al + k * 32), desc_sw128(bh + k * 32), idesc, 1u);
            }
            umma_commit(&S.mbar[st]);
        }
        __syncwarp();
    }
    if (over) atomicOr(p.status + 1, TBE_FLAG_FP16_OVERFLOW);
    // wait for the last step's MMAs (the commit covers all earlier ones)
    if (nsteps > 0 && alive) {
        const int st = (nsteps - 1) & 1;
        if (!__syncthreads_and(mbar_wait(&S.mbar[st], ph[st]))) {
            alive = false;   // block-uniform
            if (tid == 0) atomicOr(p.status + 1, TBE_FLAG_MMA_TIMEOUT);
        }
        tc_fence_after();
    }
    // slice partial: TMEM [128 lanes = d][64 columns = e] -> part[t][s][e][d]
    float *part = p.part + ((int64_t)t * p.S + s) * HE * p.D;
    {
        const int q = warp & 3, half = warp >> 2;
        const int d = q * 32 + lane;
#pragma unroll
        for (int c8 = 0; c8 < 4; ++c8) {
            uint32_t r[8];
            if (nsteps > 0 && alive) {
                tmem_ld8(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * 32 + c8 * 8), r);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int z = 0; z < 8; ++z) r[z] = 0;
            }
            if (d < p.D)
#pragma unroll
                for (int z = 0; z < 8; ++z)
                    part[(int64_t)(half * 32 + c8 * 8 + z) * p.D + d] = __uint_as_float(r[z]);
        }
    }
    S.cnt_part[tid] = mycnt;
    __syncthreads();
    if (tid < HE)
        p.cnt[((int64_t)t * p.S + s) * HE + tid] =
            S.cnt_part[tid] + S.cnt_part[tid + 64] + S.cnt_part[tid + 128] + S.cnt_part[tid + 192];
    // last slice of table t to arrive applies the update
    __threadfence();
    __syncthreads();
    if (tid == 0) S.is_last = atomicAdd(p.arrive + t, 1) == p.S - 1;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 64);
    if (!S.is_last) return;
    __threadfence();
    const int64_t row0 = __ldg(p.table_offset + t);
    const int64_t E = __ldg(p.table_offset + t + 1) - row0;
    for (int e = warp; e < HE; e += HB_THREADS / 32) {
        if (e >= E) break;
        float c = 0.f;
        for (int z = 0; z < p.S; ++z) c += __ldcg(p.cnt + ((int64_t)t * p.S + z) * HE + e);
        if (c == 0.f) continue;   // untouched row: no update
        float g[4] = {0.f, 0.f, 0.f, 0.f};
        const int d0 = lane * 4;
        if (d0 < p.D)
            for (int z = 0; z < p.S; ++z) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                    p.part + (((int64_t)t * p.S + z) * HE + e) * p.D + d0));
                g[0] += v.x; g[1] += v.y; g[2] += v.z; g[3] += v.w;
            }
        float ss = g[0] * g[0] + g[1] * g[1] + g[2] * g[2] + g[3] * g[3];
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) ss += __shfl_xor_sync(FULL, ss, sh);
        const int64_t row = row0 + e;
        const float m_new = p.mom[row] + ss / (float)p.D;
        const float den = __fadd_rn(__fsqrt_rn(m_new), p.eps);
        if (d0 < p.D) {
            __half *wr = p.W + row * p.D + d0;
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                const float w = __half2float(wr[z]);
                wr[z] = __float2half_rn(__fsub_rn(w, __fdiv_rn(__fmul_rn(p.lr, g[z]), den)));
            }
        }
        __syncwarp();
        if (lane == 0) p.mom[row] = m_new;
    }
    if (tid == 0) p.arrive[t] = 0;
}

__global__ void hist_zero_kernel(int32_t *p, int n) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) p[i] = 0;
}

// ------------------------------------------------------------ host side

bool hist_shape_ok(const tbe_tables *tab, const tbe_batch *bt, int64_t max_rows) {
    return tab->dtype == TBE_F16 && bt->per_sample_weights == nullptr && max_rows <= HE &&
           tab->D >= 64 && tab->D <= 128 && tab->D % 16 == 0;
}

// K slices per table: enough for TBE_HIST_WAVES waves of the GPU's resident
// CTA slots, rounded up.  Short slices balance better than one wave of long
// ones: T = 64, B = 65536 on 152 SMs, 0.99 ms at 1 wave (5 slices), 0.77 at
// 3, 0.75 at 6, 0.73 at 8 (the workspace grows with the slice count).
#ifndef TBE_HIST_WAVES
#define TBE_HIST_WAVES 6
#endif
static int hist_slices(const tbe_tables *tab, const tbe_batch *bt, int slots) {
    int S = (TBE_HIST_WAVES * slots + tab->T - 1) / tab->T;
    const int64_t max_s = (bt->B + HB_KBAGS - 1) / HB_KBAGS;
    if (S > max_s) S = (int)max_s;
    if (S < 1) S = 1;
    return S;
}

size_t hist_workspace_bytes(const tbe_tables *tab, const tbe_batch *bt) {
    // sized for the largest slice count any GPU of this family uses (<= 4*160 CTAs a wave)
    const int64_t S = (TBE_HIST_WAVES * 4 * 160 + tab->T - 1) / tab->T + 1;
    return (size_t)tab->T * S * HE * tab->D * 4 + (size_t)tab->T * S * HE * 4 + (size_t)tab->T * 4 +
           1024;
}

static size_t fwd_smem() { return sizeof(HistFwdSmem) + 1024; }
static size_t bwd_smem() { return sizeof(HistBwdSmem) + 1024; }

static tbe_status hist_fwd_launch(Launch &L, const tbe_tables *tab, const tbe_batch *bt,
                                  float *out, uint16_t *hist, int32_t *status, int32_t *counters,
                                  int do_mma) {
    if (bt->B == 0) return TBE_OK;
    HistFwdParams p;
    p.counters = counters;
    p.W = reinterpret_cast<const __half *>(tab->weights);
    p.table_offset = tab->table_offset;
    p.indices = bt->indices;
    p.offsets = bt->offsets;
    p.out = out;
    p.hist = hist;
    p.status = status;
    p.B = bt->B;
    p.N = bt->N;
    p.T = tab->T;
    p.D = tab->D;
    p.tiles_per_table = (bt->B + HT_BAGS - 1) / HT_BAGS;
    p.tiles_total = p.tiles_per_table * tab->T;
    p.do_mma = do_mma;
    const size_t smem = fwd_smem();
    auto kern = bt->index_type == TBE_INDEX_I64 ? tbe_hist_fwd_kernel<int64_t> : tbe_hist_fwd_kernel<int32_t>;
    cached_smem_attr(L.dev, (const void *)kern, smem);
    // CTAs per SM: shared memory (227 KB usable, 1 KB reserved per CTA) and
    // TMEM (512 columns, 128 per CTA) both allow 4 (64 registers x 256 threads allow 4)
    int per_sm = (int)((227 * 1024) / (smem + 1024));
    if (per_sm > 4) per_sm = 4;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)L.num_sms * per_sm;
    if (grid > p.tiles_total) grid = p.tiles_total;
    p.tiles_per_cta = (p.tiles_total + grid - 1) / grid;
    grid = (p.tiles_total + p.tiles_per_cta - 1) / p.tiles_per_cta;
    L.before(do_mma ? "tbe_hist_fwd_umma" : "tbe_hist_count");
    kern<<<(unsigned)grid, HF_THREADS, smem, L.stream>>>(p);
    L.after();
    return TBE_OK;
}

tbe_status launch_hist_forward(Launch &L, const tbe_tables *tab, const tbe_batch *bt, float *out,
                               uint16_t *hist, int32_t *status, int32_t *counters) {
    return hist_fwd_launch(L, tab, bt, out, hist, status, counters, 1);
}

tbe_status launch_hist_count(Launch &L, const tbe_tables *tab, const tbe_batch *bt, uint16_t *hist,
                             int32_t *status, int32_t *counters) {
    return hist_fwd_launch(L, tab, bt, nullptr, hist, status, counters, 0);
}

tbe_status launch_hist_backward(Launch &L, const tbe_tables *tab, const tbe_batch *bt,
                                const uint16_t *hist, float *momentum, const float *grad_out,
                                float lr, float eps, void *ws, int32_t *status,
                                const int32_t *counters) {
    if (bt->B == 0) return TBE_OK;
    HistBwdParams p;
    p.counters = counters;
    p.W = reinterpret_cast<__half *>(tab->weights);
    p.mom = momentum;
    p.G = grad_out;
    p.hist = hist;
    p.table_offset = tab->table_offset;
    p.status = status;
    p.B = bt->B;
    p.T = tab->T;
    p.D = tab->D;
    const size_t smem = bwd_smem();
    cached_smem_attr(L.dev, (const void *)tbe_hist_bwd_kernel, smem);
    // resident CTAs per SM (at most 4 per wave: the workspace is sized for that)
    const int per_sm = std::min(4, std::max(1, cached_blocks_per_sm(L.dev, (const void *)tbe_hist_bwd_kernel,
                                                                    HB_THREADS, smem)));
    p.S = hist_slices(tab, bt, per_sm * L.num_sms);
    const int64_t steps = (bt->B + HB_KBAGS - 1) / HB_KBAGS;
    p.kbags = ((steps + p.S - 1) / p.S) * HB_KBAGS;
    p.S = (int)((bt->B + p.kbags - 1) / p.kbags);
    char *w = (char *)ws;
    p.part = (float *)w;
    w += (size_t)tab->T * p.S * HE * tab->D * 4;
    p.cnt = (float *)w;
    w += (size_t)tab->T * p.S * HE * 4;
    p.arrive = (int32_t *)w;
    p.lr = lr;
    p.eps = eps;
    L.before("tbe_hist_zero");
    hist_zero_kernel<<<1, 256, 0, L.stream>>>(p.arrive, tab->T);
    L.after();
    L.before("tbe_hist_bwd_umma");
    tbe_hist_bwd_kernel<<<(unsigned)(tab->T * p.S), HB_THREADS, smem, L.stream>>>(p);
    L.after();
    return TBE_OK;
}

}  // namespace tbe
