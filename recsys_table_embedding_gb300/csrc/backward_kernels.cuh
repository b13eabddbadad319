// Backward kernels: per-unique-row gradient reduction with one fused exact
// rowwise Adagrad update per touched row.  Templates only: backward_f32.cu,
// backward_f16.cu and backward_bf16.cu instantiate them per weight dtype
// (compiled in parallel), backward.cu dispatches.
//
// FBTriton TBE redesign (accesspath.com), "Backward kernels: three paths by
// segment length":
//   short_run      (SL < 256): one owner reduces the whole run, applies the
//                  optimizer and stores with plain stores (no atomics);
//   grad_accum + apply (SL >= 256): runs are cut into 256-lookup chunks,
//                  partial sums go to a workspace, a second kernel applies;
//   fused          (SL >= 256): same chunks, a device-scope fence lets the
//                  last-arriving chunk apply the update in the same launch;
//   weighted tables scale each gradient row by its per-sample weight first.
// Decision checklist item 1: FP32 accumulation for FP16/BF16 weights, FP64
// for FP32 weights.  TorchEasyRec analysis (39.107.221.112 article 1724244),
// section 4: the optimizer update is fused into the backward (one read and
// one write of each touched row).
//
// Design.  Gradient rows are float32 [B, T*D].
//   * Long runs: a warp per 256-lookup chunk, chunks taken in (table, bag
//     window) order; rows arrive through a per-warp ring of bulk copies
//     (cp.async.bulk into shared memory, mbarrier completion) that streams
//     across chunk boundaries.  Partials of chunk slot c live at
//     partials[c*D ...] in the accumulator type.  The long-run sum always
//     adds the chunk partials in chunk order c = 0..k-1, so the two-kernel
//     and the fused modes give bit-identical weights and momentum.  The fused
//     mode needs no waiting: each chunk stores its partial, fences, and bumps
//     the run's arrival counter; only the warp that sees k-1 reads the
//     partials (through L2) and applies, then re-arms the counter.
//   * Short runs, unweighted batches (and rows under 512 bytes): a group of
//     lanes per run reads rows as float4 vectors from global memory, with the
//     weight slice and momentum loaded ahead.
//   * Short runs, weighted batches with rows of 512 bytes and more: a warp
//     streams the rows of consecutive runs through a bulk-copy ring and
//     applies each run's update from weight rows prefetched per task.
#pragma once

#include "tbe_internal.cuh"

namespace tbe {

struct BwdParams {
    void *W;
    float *mom;
    const float *G;
    const int64_t *table_offset;
    const tbe_table_layout *layout;     // nullable: uniform tables
    const tbe_bag_layout *bag_layout;   // nullable: uniform bags and gradient rows
    int cls_dtype;                      // with a layout: this launch's class (D is p.D)
    int64_t part_stride;                // bytes from one chunk slot's partial to the next
    const uint32_t *vals;
    const int32_t *bag_of;
    const float *psw;
    const uint8_t *weighted;
    const void *unique_keys;      // uint32 or uint64 (key64)
    int key64;
    const int32_t *seg_off;
    const int32_t *counters;
    const int32_t *long_run;
    const int32_t *long_chunk_base;
    const int32_t *chunk_order;   // null: slot c is taken c-th
    const int32_t *chunk_desc;
    void *partials;
    int32_t *arrive;
    int32_t *status;
    int64_t B;
    int T;
    int D;
    float lr;
    float eps;
    int sl_threshold;
    int chunk;
    int payload_pos;
};

// unique key r (a row of the weight array)
__device__ __forceinline__ int64_t load_key(const BwdParams &p, int64_t r) {
    return p.key64 ? (int64_t)__ldg(reinterpret_cast<const unsigned long long *>(p.unique_keys) + r)
                   : (int64_t)__ldg(reinterpret_cast<const uint32_t *>(p.unique_keys) + r);
}

// weight row of linearised row `key` of table t (row length p.D); `layout`
// is p.layout, or a null constant where a kernel is built without layouts
template <typename WT>
__device__ __forceinline__ WT *wrow_of(const BwdParams &p, const tbe_table_layout *layout, int t,
                                       int64_t key) {
    return reinterpret_cast<WT *>(reinterpret_cast<char *>(p.W) +
                                  weight_byte(layout, p.table_offset, t, key, p.D, (int)sizeof(WT)));
}
template <typename WT> __device__ __forceinline__ WT *wrow_of(const BwdParams &p, int t, int64_t key) {
    return wrow_of<WT>(p, p.layout, t, key);
}

// bag within table t of a sorted payload: the bag itself (unweighted
// batches) or, for a lookup position, its CSR bag less the table's first
__device__ __forceinline__ int64_t payload_bag(const BwdParams &p, const tbe_bag_layout *bags,
                                               uint32_t v, int t) {
    if (!p.payload_pos) return (int64_t)v;
    return (int64_t)__ldg(p.bag_of + v) - bag_base(bags, p.B, t);
}
__device__ __forceinline__ int64_t payload_bag(const BwdParams &p, uint32_t v, int t) {
    return payload_bag(p, p.bag_layout, v, t);
}

// bags of table t
__device__ __forceinline__ int64_t bags_of(const BwdParams &p, const tbe_bag_layout *bags, int t) {
    return bags == nullptr ? p.B : __ldg(&bags[t].B);
}
__device__ __forceinline__ int64_t bags_of(const BwdParams &p, int t) { return bags_of(p, p.bag_layout, t); }

__device__ __forceinline__ void acc4(double (&a)[4], const float4 x, float w) {
    a[0] = fma((double)w, (double)x.x, a[0]);
    a[1] = fma((double)w, (double)x.y, a[1]);
    a[2] = fma((double)w, (double)x.z, a[2]);
    a[3] = fma((double)w, (double)x.w, a[3]);
}
__device__ __forceinline__ void acc4(float (&a)[4], const float4 x, float w) {
    a[0] = fmaf(w, x.x, a[0]);
    a[1] = fmaf(w, x.y, a[1]);
    a[2] = fmaf(w, x.z, a[2]);
    a[3] = fmaf(w, x.w, a[3]);
}

__device__ __forceinline__ void ld4(const float *p, float (&w)[4]) {
    const float4 v = *reinterpret_cast<const float4 *>(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
}
__device__ __forceinline__ void st4(float *p, const float (&w)[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void ld4(const __half *p, float (&w)[4]) {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&v.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&v.y));
    w[0] = a.x; w[1] = a.y; w[2] = b.x; w[3] = b.y;
}
__device__ __forceinline__ void st4(__half *p, const float (&w)[4]) {
    __half2 a = __halves2half2(__float2half_rn(w[0]), __float2half_rn(w[1]));
    __half2 b = __halves2half2(__float2half_rn(w[2]), __float2half_rn(w[3]));
    uint2 v;
    v.x = *reinterpret_cast<uint32_t *>(&a);
    v.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = v;
}
__device__ __forceinline__ void ld4(const __nv_bfloat16 *p, float (&w)[4]) {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    const float2 a = bf16x2_to_float2(v.x);
    const float2 b = bf16x2_to_float2(v.y);
    w[0] = a.x; w[1] = a.y; w[2] = b.x; w[3] = b.y;
}
__device__ __forceinline__ void st4(__nv_bfloat16 *p, const float (&w)[4]) {
    __nv_bfloat162 a = __halves2bfloat162(__float2bfloat16_rn(w[0]), __float2bfloat16_rn(w[1]));
    __nv_bfloat162 b = __halves2bfloat162(__float2bfloat16_rn(w[2]), __float2bfloat16_rn(w[3]));
    uint2 v;
    v.x = *reinterpret_cast<uint32_t *>(&a);
    v.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = v;
}

// partial storage in the accumulator type
__device__ __forceinline__ void st_part(double *p, const double (&a)[4]) {
    reinterpret_cast<double2 *>(p)[0] = make_double2(a[0], a[1]);
    reinterpret_cast<double2 *>(p)[1] = make_double2(a[2], a[3]);
}
__device__ __forceinline__ void st_part(float *p, const float (&a)[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(a[0], a[1], a[2], a[3]);
}
template <bool L2ONLY>
__device__ __forceinline__ void ld_part(double (&a)[4], const double *p) {
    const double2 x = L2ONLY ? __ldcg(reinterpret_cast<const double2 *>(p))
                             : __ldg(reinterpret_cast<const double2 *>(p));
    const double2 y = L2ONLY ? __ldcg(reinterpret_cast<const double2 *>(p) + 1)
                             : __ldg(reinterpret_cast<const double2 *>(p) + 1);
    a[0] = x.x; a[1] = x.y; a[2] = y.x; a[3] = y.y;
}
template <bool L2ONLY>
__device__ __forceinline__ void ld_part(float (&a)[4], const float *p) {
    const float4 x = L2ONLY ? __ldcg(reinterpret_cast<const float4 *>(p))
                            : __ldg(reinterpret_cast<const float4 *>(p));
    a[0] = x.x; a[1] = x.y; a[2] = x.z; a[3] = x.w;
}

// acc += partials of chunk slots cb .. cb+nch-1, added strictly in chunk
// order; PB slots are loaded ahead so that many loads are in flight.
// partial of chunk slot `slot` (stride bytes apart)
template <typename ACC> __device__ __forceinline__ ACC *part_of(void *partials, int64_t stride, int64_t slot) {
    return reinterpret_cast<ACC *>(reinterpret_cast<char *>(partials) + slot * stride);
}

// (PB only sets how many loads are in flight, not the order of the additions)
template <bool L2ONLY, typename ACC, int LPR, int NV, int PB = (NV >= 2 ? 2 : 4)>
__device__ __forceinline__ void sum_partials(ACC (&acc)[NV][4], void *partials, int64_t stride, int cb,
                                             int nch, int li) {
    for (int c0 = 0; c0 < nch; c0 += PB) {
        ACC v[PB][NV][4];
#pragma unroll
        for (int j = 0; j < PB; ++j)
            if (c0 + j < nch)
#pragma unroll
                for (int q = 0; q < NV; ++q)
                    ld_part<L2ONLY>(v[j][q], part_of<ACC>(partials, stride, cb + c0 + j) + li * 4 + q * LPR * 4);
#pragma unroll
        for (int j = 0; j < PB; ++j)
            if (c0 + j < nch)
#pragma unroll
                for (int q = 0; q < NV; ++q)
#pragma unroll
                    for (int x = 0; x < 4; ++x) acc[q][x] += v[j][q][x];
    }
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
// ---- bulk-copy gather ------------------------------------------------------
// One lane issues a cp.async.bulk (the TMA engine's non-tensor copy) per
// gradient row into a per-warp ring of STAGES stages of 4 KB; each stage's
// mbarrier completes when all its bytes have landed.  Lanes then read their
// own 16-byte vectors of each row from shared memory.

#ifndef TBE_BWD_STAGES
#define TBE_BWD_STAGES 2   // more warps beat deeper rings: 3.20 ms at 2 stages vs 3.96 at 3
#endif
#ifndef TBE_CHUNK_THREADS
#define TBE_CHUNK_THREADS 128
#endif
#ifndef TBE_CHUNK_UB
#define TBE_CHUNK_UB 8   // rows of a full long-run stage read before they are added: 2.51 ms vs 2.67 row by row
#endif
constexpr int STAGES = TBE_BWD_STAGES;
constexpr int STAGE_BYTES = 4096;
#ifndef TBE_CHUNK_STAGE_BYTES
#define TBE_CHUNK_STAGE_BYTES 4096   // large workload: 2.67 ms; 2048: 3.67, 6144: 3.25, 8192: 2.89
#endif
constexpr int CSTAGE_BYTES = TBE_CHUNK_STAGE_BYTES;   // stage of the long-run ring (>= the widest row)
static_assert(CSTAGE_BYTES >= 2048 && CSTAGE_BYTES % 2048 == 0, "long-run stages hold whole rows");
// 4 warps: at chunk 256, five blocks fit an SM for unweighted batches, four
// with the weight buffer
constexpr int CHUNK_THREADS = TBE_CHUNK_THREADS;
constexpr int PV = 8;                // payloads a lane prefetches in registers

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// global -> shared bulk copy of `bytes` (multiple of 16, both ends 16-byte aligned)
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// shared memory of one warp: STAGES x CSTAGE_BYTES ring, STAGES mbarriers,
// then two buffers (current and next chunk) of the gradient-row offset and,
// for weighted batches, the weight of each lookup
__host__ __device__ constexpr int warp_smem_bytes(int chunk, bool weighted) {
    return (STAGES * CSTAGE_BYTES + 64 + 2 * chunk * (weighted ? 8 : 4) + 127) / 128 * 128;
}
// a lookup whose bag lies outside its run's table (only malformed offsets
// can make one) is marked in the offset buffer; its copy reads a row of
// zeros (never written, so zero from module load), so it adds nothing
constexpr uint32_t NO_ROW = 0xFFFFFFFFu;
static __device__ __align__(128) float g_zero_row[512];   // the widest gradient row

// One chunk of a long run, as the route kernel describes it.
struct Chunk {
    int32_t s, e;      // sorted positions [s, e)
    int64_t key;
    int t, l, cb, nch; // table, long run, its first chunk slot and chunk count
    int slot;          // chunk slot (index of its descriptor and its partial)
    bool skip;         // a table of another launch's class: nothing to do here
};

// the chunk taken ci-th: slot chunk_order[ci], or ci without an order
__device__ __forceinline__ Chunk load_chunk(const BwdParams &p, const tbe_table_layout *layout, int ci) {
    const int slot = p.chunk_order != nullptr ? __ldg(p.chunk_order + ci) : ci;
    const int4 a = __ldg(reinterpret_cast<const int4 *>(p.chunk_desc) + 2 * (int64_t)slot);
    const int4 b = __ldg(reinterpret_cast<const int4 *>(p.chunk_desc) + 2 * (int64_t)slot + 1);
    Chunk c;
    c.s = a.x; c.e = a.y;
    c.key = (int64_t)(((uint64_t)(uint32_t)a.w << 32) | (uint32_t)a.z);
    c.t = table_of_key(p.table_offset, p.T, c.key);
    c.l = b.x; c.cb = b.y; c.nch = b.z;
    c.slot = slot;
    c.skip = !in_class(layout, c.t, p.D, p.cls_dtype);
    if (c.skip) c.e = c.s;
    return c;
}
// Exact rowwise Adagrad arithmetic, m += mean_d(g^2); w -= lr*g/(sqrt(m)+eps),
// in the accumulator's precision: FP64 for FP32 tables, from the FP64 row
// gradient (decision checklist item 1's FP64 accumulation carried through the
// update, so the stored weight is the correctly rounded result), FP32 for
// FP16/BF16 tables.  The new momentum is rounded to FP32 (its stored type)
// before it enters the denominator.
template <typename ACC> struct Adagrad;
template <> struct Adagrad<double> {
    using G = double;   // type the row gradient enters the update in
    static __device__ __forceinline__ G grad(double a) { return a; }
    static __device__ __forceinline__ float mom(float m_old, double ss, int D) {
        return (float)((double)m_old + ss / (double)D);
    }
    static __device__ __forceinline__ double den(float m_new, float eps) {
        return sqrt((double)m_new) + (double)eps;
    }
    static __device__ __forceinline__ float step(float w, double g, float lr, double den) {
        return (float)((double)w - (double)lr * g / den);
    }
};
template <> struct Adagrad<float> {
    using G = float;
    static __device__ __forceinline__ G grad(float a) { return a; }
    static __device__ __forceinline__ float mom(float m_old, float ss, int D) {
        return __fadd_rn(m_old, __fdiv_rn(ss, (float)D));
    }
    static __device__ __forceinline__ float den(float m_new, float eps) {
        return __fadd_rn(__fsqrt_rn(m_new), eps);
    }
    static __device__ __forceinline__ float step(float w, float g, float lr, float den) {
        return __fsub_rn(w, __fdiv_rn(__fmul_rn(lr, g), den));
    }
};

// Exact rowwise Adagrad on row `row` from the reduced gradient in acc.  Only
// lanes of sub-group 0 hold meaningful values; every lane takes part in the
// shuffles.
template <typename WT, typename ACC, int LPR, int NV>
__device__ __forceinline__ void adagrad_apply(const ACC (&acc)[NV][4], const BwdParams &p,
                                              const tbe_table_layout *layout, int t, int64_t row,
                                              int lane, int sub, int li) {
    using A = Adagrad<ACC>;
    ACC ss = ACC(0);
#pragma unroll
    for (int q = 0; q < NV; ++q)
#pragma unroll
        for (int x = 0; x < 4; ++x) ss += acc[q][x] * acc[q][x];
#pragma unroll
    for (int sh = 1; sh < LPR; sh <<= 1) ss += __shfl_xor_sync(FULL, ss, sh);
    if (sub != 0) return;
    const float m_new = A::mom(p.mom[row], ss, p.D);
    const auto den = A::den(m_new, p.eps);
    WT *wr = wrow_of<WT>(p, layout, t, row) + li * 4;
#pragma unroll
    for (int q = 0; q < NV; ++q) {
        float w[4];
        ld4(wr + q * LPR * 4, w);
#pragma unroll
        for (int x = 0; x < 4; ++x) w[x] = A::step(w[x], acc[q][x], p.lr, den);
        st4(wr + q * LPR * 4, w);
    }
    if (lane == 0) p.mom[row] = m_new;
}

// Raw weight slices held between the prefetch and the update.
template <typename WT> struct WRaw;
template <> struct WRaw<float> { using t = float4; };
template <> struct WRaw<__half> { using t = uint2; };
template <> struct WRaw<__nv_bfloat16> { using t = uint2; };

template <typename WT>
__device__ __forceinline__ typename WRaw<WT>::t ld_wraw(const WT *p) {
    return *reinterpret_cast<const typename WRaw<WT>::t *>(p);
}
__device__ __forceinline__ void unpack_w(const float4 r, float (&w)[4]) {
    w[0] = r.x; w[1] = r.y; w[2] = r.z; w[3] = r.w;
}
__device__ __forceinline__ void unpack_w(const uint2 r, float (&w)[4], __half) {
    const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
    const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
    w[0] = a.x; w[1] = a.y; w[2] = b.x; w[3] = b.y;
}
__device__ __forceinline__ void unpack_w(const uint2 r, float (&w)[4], __nv_bfloat16) {
    const float2 a = bf16x2_to_float2(r.x);
    const float2 b = bf16x2_to_float2(r.y);
    w[0] = a.x; w[1] = a.y; w[2] = b.x; w[3] = b.y;
}
template <typename WT>
__device__ __forceinline__ void unpack(const typename WRaw<WT>::t r, float (&w)[4]) {
    if constexpr (sizeof(WT) == 4) unpack_w(r, w);
    else unpack_w(r, w, WT());
}

// Short runs (SL < sl_threshold): a group of GL lanes owns one run, so a warp
#ifndef TBE_SHORT_PREFETCH
#define TBE_SHORT_PREFETCH 1   // load the next run's range and key one iteration ahead
#endif
#ifndef TBE_SHORT_MINB
#define TBE_SHORT_MINB 3       // 256-thread blocks per SM the register budget must allow
#endif
// (FP64 accumulators of FP32 tables take twice the registers: two blocks)
#ifndef TBE_SHORT_THREADS
#define TBE_SHORT_THREADS 256   // threads of a short-run block (128, 7 per SM at 72 registers: 2.21 vs 2.19 ms)
#endif
template <typename WT> constexpr int short_min_blocks() { return sizeof(WT) == 4 ? 2 : TBE_SHORT_MINB; }
#ifndef TBE_SHORT_U
#define TBE_SHORT_U 0          // gradient rows in flight per run step (0: 2 or 4 by row width; 6 or 8 at two blocks per SM: 3.3-3.5 ms)
#endif

// works on 32/GL runs at once.  Lane gl of a group holds vectors
// gl + q*GL (q < NV) of the row (float4 of the gradient, 4 weights).  The
// weight slice and the momentum are loaded before the gather so their
// latency overlaps it; U gradient rows of the run are in flight per step.
template <typename WT, int GL, int NV, int U, bool LAY>
__global__ void __launch_bounds__(TBE_SHORT_THREADS, short_min_blocks<WT>()) tbe_bwd_short_kernel(const BwdParams p) {
    using ACC = typename WTraits<WT>::acc;
    // LAY: tables or bags with layouts; without, the layout code folds away
    const tbe_table_layout *layout = LAY ? p.layout : nullptr;
    const tbe_bag_layout *bag_layout = LAY ? p.bag_layout : nullptr;
    constexpr int GPW = 32 / GL;
    const int lane = threadIdx.x & 31, grp = lane / GL, gl = lane % GL;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int U_runs = p.counters[C_NUM_UNIQUE];
    const int64_t TD = (int64_t)p.T * p.D;
    // range and key of the group's next run, loaded one iteration ahead so
    // their latency overlaps the current run's gather
    int32_t s_n = 0, e_n = 0;
    int64_t key_n = 0;
    auto meta = [&](int r) {
        if (r < U_runs) {
            s_n = __ldg(p.seg_off + r);
            e_n = __ldg(p.seg_off + r + 1);
            key_n = load_key(p, r);
        }
    };
    // (wide lane vectors keep their registers for the gather instead; the
    // next run's first payloads loaded one iteration ahead as well measured
    // slower, 2.45 vs 2.19 ms on the large workload)
    constexpr bool PF = TBE_SHORT_PREFETCH && NV <= 2;
    if (PF) meta(warp * GPW + grp);
    for (int rb = warp * GPW; rb < U_runs; rb += nwarps * GPW) {
        const int r = rb + grp;
        if (!PF) meta(r);
        const int32_t s = s_n, e = e_n;
        const int64_t key = key_n;
        if (PF) meta(r + nwarps * GPW);
        bool mine = r < U_runs && e - s < p.sl_threshold;
        int t = 0;
        if (layout != nullptr) {   // the run's table decides its class first
            if (mine) t = table_of_key(p.table_offset, p.T, key);
            mine = mine && in_class(layout, t, p.D, p.cls_dtype);
        }
        ACC acc[NV][4];
#pragma unroll
        for (int q = 0; q < NV; ++q)
#pragma unroll
            for (int x = 0; x < 4; ++x) acc[q][x] = ACC(0);
        typename WRaw<WT>::t wraw[NV];
        float m_old = 0.f;
        // uniform tables: the weight row follows from the key alone, so its
        // loads are issued before the table lookup
        WT *wr = layout != nullptr ? (mine ? wrow_of<WT>(p, layout, t, key) : nullptr)
                                   : reinterpret_cast<WT *>(p.W) + key * p.D;
        if (mine) {
#pragma unroll
            for (int q = 0; q < NV; ++q) wraw[q] = ld_wraw(wr + (gl + q * GL) * 4);
            m_old = p.mom[key];
            if (layout == nullptr) t = table_of_key(p.table_offset, p.T, key);
            const bool wt = p.psw != nullptr && (p.weighted == nullptr || __ldg(p.weighted + t) != 0);
            // gradient row of bag b: G + g0 + b * gs
            const float *Gt = p.G + (bag_layout ? __ldg(&bag_layout[t].out_offset) : (int64_t)t * p.D) +
                              gl * 4;
            const int64_t gs = bag_layout ? __ldg(&bag_layout[t].out_stride) : TD;
            const int Bt = (int)bags_of(p, bag_layout, t);
            for (int32_t i = s; i < e; i += U) {
                int bk[U];
                float wk[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    bk[u] = -1;
                    wk[u] = 1.f;
                    if (i + u < e) {
                        const uint32_t v = __ldg(p.vals + i + u);
                        const int b = (int)payload_bag(p, bag_layout, v, t);
                        if (p.payload_pos && wt) wk[u] = __ldg(p.psw + v);
                        // only malformed (overlapping) offsets can give a bag
                        // outside the run's table; such a lookup adds nothing
                        bk[u] = (b >= 0 && b < Bt) ? b : -1;
                    }
                }
                float4 x[U][NV];
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (bk[u] >= 0)
#pragma unroll
                        for (int q = 0; q < NV; ++q)
                            x[u][q] = __ldg(reinterpret_cast<const float4 *>(Gt + (int64_t)bk[u] * gs + q * GL * 4));
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (bk[u] >= 0)
#pragma unroll
                        for (int q = 0; q < NV; ++q) acc4(acc[q], x[u][q], wk[u]);
            }
        }
        // exact rowwise Adagrad: m += mean_d g^2; w -= lr * g / (sqrt(m) + eps)
        using A = Adagrad<ACC>;
        ACC ss = ACC(0);
#pragma unroll
        for (int q = 0; q < NV; ++q)
#pragma unroll
            for (int x = 0; x < 4; ++x) ss += acc[q][x] * acc[q][x];
#pragma unroll
        for (int o = 1; o < GL; o <<= 1) ss += __shfl_xor_sync(FULL, ss, o);
        if (mine) {
            const float m_new = A::mom(m_old, ss, p.D);
            const auto den = A::den(m_new, p.eps);
#pragma unroll
            for (int q = 0; q < NV; ++q) {
                float w[4];
                unpack<WT>(wraw[q], w);
#pragma unroll
                for (int x = 0; x < 4; ++x) w[x] = A::step(w[x], acc[q][x], p.lr, den);
                st4(wr + (gl + q * GL) * 4, w);
            }
            if (gl == 0) p.mom[key] = m_new;
        }
    }
}

// Long-run chunks.  A warp takes the chunks at order positions ci,
// ci + nwarps, ... (slot chunk_order[ci]: slots grouped by the batch window
// of their first bag, so warps working at the same time read gradient rows
// of nearby bags, which L2 then serves) and treats their gradient rows as one
// stream of ring stages: while it reduces chunk j, the ring already holds
// copies of chunk j+1, whose lookups were staged in the second buffer, so
// neither the chunk's metadata, its payload loads nor the fused tail leave
// the copy engine idle.  A stage never spans two chunks.  The partial of a
// chunk slot is the sum over its range in sorted order, so results do not
// depend on the order or on which warp took which chunk.
template <typename WT, int LPR, int NV, bool FUSED, bool LAY, bool WGT>
__global__ void __launch_bounds__(CHUNK_THREADS) tbe_bwd_chunk_kernel(const BwdParams p) {
    using ACC = typename WTraits<WT>::acc;
    constexpr int RPI = 32 / LPR;
    // LAY: tables or bags with layouts; WGT: the batch has per-sample
    // weights (a weight buffer next to the offsets); without either, its
    // code folds away
    const tbe_table_layout *layout = LAY ? p.layout : nullptr;
    const tbe_bag_layout *bag_layout = LAY ? p.bag_layout : nullptr;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31, sub = lane / LPR, li = lane % LPR;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int nchunks = p.counters[C_NUM_CHUNKS];
    int ci = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (ci >= nchunks) return;

    unsigned char *wsm = smem_raw + (threadIdx.x >> 5) * warp_smem_bytes(p.chunk, WGT);
    const uint32_t ring0 = smem_addr(wsm);
    const uint32_t bar0 = smem_addr(wsm + STAGES * CSTAGE_BYTES);
    uint32_t *offb = reinterpret_cast<uint32_t *>(wsm + STAGES * CSTAGE_BYTES + 64);  // [2][chunk], 16-B units
    float *wgt = WGT ? reinterpret_cast<float *>(offb + 2 * p.chunk) : nullptr;      // [2][chunk]
    if (lane == 0)
        for (int i = 0; i < STAGES; ++i) bar_init(bar0 + 8 * i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();

    const uint32_t row_bytes = (uint32_t)p.D * 4;
    const int R = CSTAGE_BYTES / (int)row_bytes;   // rows per stage (D <= 512)
    const float4 *G4 = reinterpret_cast<const float4 *>(p.G);

    // payload of lookups [s, s + PV*32) into registers (issued early)
    uint32_t pv[PV];
    auto fetch = [&](const Chunk &c) {
#pragma unroll
        for (int k = 0; k < PV; ++k) {
            const int32_t i = c.s + lane + 32 * k;
            pv[k] = i < c.e ? __ldg(p.vals + i) : 0u;
        }
    };
    // offset from G (in 16-byte vectors) of each lookup's gradient row and its
    // weight, for the lookups of c, into buffer buf
    auto stage = [&](const Chunk &c, int buf) {
        const bool wt = WGT && p.psw != nullptr && (p.weighted == nullptr || __ldg(p.weighted + c.t) != 0);
        const int n = c.e - c.s;
        const int64_t g0 = bag_layout ? __ldg(&bag_layout[c.t].out_offset) : (int64_t)c.t * p.D;
        const int64_t gs = bag_layout ? __ldg(&bag_layout[c.t].out_stride) : (int64_t)p.T * p.D;
        const int64_t Bt = bags_of(p, bag_layout, c.t);
        uint32_t *o = offb + buf * p.chunk;
        float *w = WGT ? wgt + buf * p.chunk : nullptr;
        auto put = [&](int i, uint32_t v) {
            const int64_t b = payload_bag(p, bag_layout, v, c.t);
            // only malformed (overlapping) offsets can give a bag outside the
            // run's table: such a lookup copies row 0 and adds nothing
            const bool ok = b >= 0 && b < Bt;
            o[i] = ok ? (uint32_t)((g0 + b * gs) >> 2) : NO_ROW;   // 16-byte units
            if constexpr (WGT) w[i] = p.payload_pos && wt ? __ldg(p.psw + v) : 1.f;
        };
#pragma unroll
        for (int k = 0; k < PV; ++k)
            if (lane + 32 * k < n) put(lane + 32 * k, pv[k]);
        for (int i = lane + 32 * PV; i < n; i += 32) put(i, __ldg(p.vals + c.s + i));
        __syncwarp();
    };

    uint32_t gprod = 0, gcons = 0, phase = 0;
    auto produce = [&](const Chunk &c, int buf, int k) {
        const int st = (int)(gprod % STAGES);
        const int rows = min(R, c.e - c.s - k * R);
        const uint32_t bar = bar0 + 8 * st;
        if (lane == 0) bar_arrive_expect_tx(bar, (uint32_t)rows * row_bytes);
        __syncwarp();
        const uint32_t *o = offb + buf * p.chunk + k * R;
        const uint32_t dst0 = ring0 + st * CSTAGE_BYTES;
        for (int j = lane; j < rows; j += 32) {
            const uint32_t oj = o[j];
            bulk_g2s(dst0 + j * row_bytes, oj != NO_ROW ? (const void *)(G4 + oj) : (const void *)g_zero_row,
                     row_bytes, bar);
        }
        ++gprod;
    };

    Chunk cur = load_chunk(p, layout, ci);
    fetch(cur);
    stage(cur, 0);
    int buf = 0;
    int ni = ci + nwarps;
    bool has_next = ni < nchunks;
    Chunk nxt = cur;
    if (has_next) nxt = load_chunk(p, layout, ni);
    int cur_nst = (cur.e - cur.s + R - 1) / R;
    int pk = 0;              // next stage to issue of the chunk being issued
    bool p_next = false;     // issuing into nxt already
    bool next_staged = false;
    auto refill = [&]() {
        while (gprod - gcons < (uint32_t)STAGES) {
            if (!p_next) {
                if (pk < cur_nst) { produce(cur, buf, pk++); continue; }
                if (!has_next || !next_staged) break;
                p_next = true;
                pk = 0;
            }
            if (pk < (nxt.e - nxt.s + R - 1) / R) produce(nxt, buf ^ 1, pk++);
            else break;
        }
    };
    refill();

    for (;;) {
        next_staged = false;
        if (has_next) fetch(nxt);   // latency overlaps the first stage below
        ACC acc[NV][4];
#pragma unroll
        for (int q = 0; q < NV; ++q)
#pragma unroll
            for (int x = 0; x < 4; ++x) acc[q][x] = ACC(0);
        const float *w = WGT ? wgt + buf * p.chunk : nullptr;
        for (int k = 0; k < cur_nst; ++k) {
            const int st = (int)(gcons % STAGES);
            if (!mbar_wait_bounded(bar0 + 8 * st, (phase >> st) & 1u)) {
                // stop issuing: give the copies still in flight one more
                // bounded wait each, flag the failure, end the warp's work
                for (uint32_t g = gcons + 1; g < gprod; ++g)
                    mbar_wait_bounded(bar0 + 8 * (g % STAGES), (phase >> (g % STAGES)) & 1u);
                if (lane == 0) atomicOr(p.status + 1, TBE_FLAG_COPY_TIMEOUT);
                return;
            }
            phase ^= 1u << st;
            const int rows = min(R, cur.e - cur.s - k * R);
            const unsigned char *sp = wsm + st * CSTAGE_BYTES;
            // a full stage: its rows' vectors are read UBE at a time before
            // they are added (same order of additions as the loop below)
            constexpr int RC = CSTAGE_BYTES / (LPR * NV * 16);   // rows of a full stage
            constexpr int IT = RC / RPI;                          // rows of a full stage per lane
            constexpr int UBE = TBE_CHUNK_UB < IT ? TBE_CHUNK_UB : IT;
            static_assert(IT % UBE == 0, "full stages split into equal batches");
            if (UBE > 1 && rows == RC) {
#pragma unroll
                for (int j0 = 0; j0 < IT; j0 += UBE) {
                    float4 v[UBE][NV];
                    float xw[UBE];
#pragma unroll
                    for (int u = 0; u < UBE; ++u) {
                        const int j = sub + (j0 + u) * RPI;
                        const float4 *src = reinterpret_cast<const float4 *>(sp + j * row_bytes) + li;
#pragma unroll
                        for (int q = 0; q < NV; ++q) v[u][q] = src[q * LPR];
                        xw[u] = WGT ? w[k * R + j] : 1.f;
                    }
#pragma unroll
                    for (int u = 0; u < UBE; ++u)
#pragma unroll
                        for (int q = 0; q < NV; ++q) acc4(acc[q], v[u][q], xw[u]);
                }
            } else {
                for (int j = sub; j < rows; j += RPI) {
                    const float4 *src = reinterpret_cast<const float4 *>(sp + j * row_bytes) + li;
                    if constexpr (WGT) {
                        const float x = w[k * R + j];
#pragma unroll
                        for (int q = 0; q < NV; ++q) acc4(acc[q], src[q * LPR], x);
                    } else {
#pragma unroll
                        for (int q = 0; q < NV; ++q) acc4(acc[q], src[q * LPR], 1.f);
                    }
                }
            }
            ++gcons;
            __syncwarp();   // the stage is read before it is refilled
            if (!next_staged && has_next) {
                stage(nxt, buf ^ 1);
                next_staged = true;
            }
            refill();
        }
        if (!next_staged && has_next) {
            stage(nxt, buf ^ 1);
            next_staged = true;
            refill();
        }
#pragma unroll
        for (int sh = LPR; sh < 32; sh <<= 1)
#pragma unroll
            for (int q = 0; q < NV; ++q)
#pragma unroll
                for (int x = 0; x < 4; ++x) acc[q][x] += __shfl_xor_sync(FULL, acc[q][x], sh);
        ACC *part = part_of<ACC>(p.partials, p.part_stride, cur.slot) + li * 4;
        if (sub == 0 && !cur.skip)
#pragma unroll
            for (int q = 0; q < NV; ++q) st_part(part + q * LPR * 4, acc[q]);
        if (FUSED && !cur.skip) {
            __threadfence();
            __syncwarp();
            int old = 0;
            if (lane == 0) old = atomicAdd(p.arrive + cur.l, 1);
            old = __shfl_sync(FULL, old, 0);
            if (old == cur.nch - 1) {
                __threadfence();
#pragma unroll
                for (int q = 0; q < NV; ++q)
#pragma unroll
                    for (int x = 0; x < 4; ++x) acc[q][x] = ACC(0);
                if (sub == 0)
                    sum_partials<true, ACC, LPR, NV>(acc, p.partials, p.part_stride, cur.cb, cur.nch, li);
                adagrad_apply<WT, ACC, LPR, NV>(acc, p, layout, cur.t, cur.key, lane, sub, li);
                if (lane == 0) p.arrive[cur.l] = 0;
            }
        }
        if (!has_next) break;
        // the next chunk becomes current; stages already issued for it stay
        cur = nxt;
        buf ^= 1;
        cur_nst = (cur.e - cur.s + R - 1) / R;
        if (!p_next) pk = 0;
        p_next = false;
        ni += nwarps;
        has_next = ni < nchunks;
        if (has_next) nxt = load_chunk(p, layout, ni);
        next_staged = false;
        refill();
    }
}

// ---- streaming short runs (gradient rows of 512 bytes and more) -----------
// A warp takes tasks of RT consecutive runs (lane i: run r0 + i), skips the
// long ones, and streams the gradient rows of the short ones, in sorted
// order, through the same kind of bulk-copy ring as the long-run kernel.
// The lookups of a task are staged 32 at a time into a table (offset,
// weight, run slot, last-of-run flag); each run's weight row is copied into a
// per-task shared buffer and its momentum loaded when the task starts, so the
// Adagrad update of a run is applied as soon as its last gradient row has
// been added, without a round trip to memory.  The ring, the tables and the
// weight buffers are double-buffered across blocks and tasks, so metadata,
// payload and weight loads overlap the rows in flight.

#ifndef TBE_SHORT_STREAM
#define TBE_SHORT_STREAM 1   // 0: the register kernel for every batch
#endif
#ifndef TBE_SHORT_STAGES
#define TBE_SHORT_STAGES 1   // mid workload: 1.93 ms at 1 stage, 2.18 at 2, 2.59 at 3 (more warps win)
#endif
constexpr int SS_STAGES = TBE_SHORT_STAGES;
constexpr int SS_WARPS = 2;          // warps per CTA
#ifndef TBE_SHORT_WBUF
#define TBE_SHORT_WBUF 2048   // mid workload: 2.02 ms at 2 KB vs 2.18 at 4 KB (2 stages)
#endif
constexpr int SS_WBUF = TBE_SHORT_WBUF;   // weight-row buffer per task
constexpr int SS_BLK = 32;           // lookups per staged table
constexpr uint32_t SS_LAST = 0x100u; // tag flag: last lookup of its run

__host__ __device__ constexpr int ss_warp_bytes() {
    return (SS_STAGES * STAGE_BYTES + 2 * SS_WBUF + 3 * 2 * SS_BLK * 4 + 8 * (SS_STAGES + 2) + 127) /
           128 * 128;
}
// runs per task: as many weight rows as fit the buffer, at most 32
__host__ __device__ inline int ss_runs_per_task(int wrow_bytes) {
    const int r = SS_WBUF / wrow_bytes;
    return r < 1 ? 1 : (r > 32 ? 32 : r);
}

// One task as its lanes hold it (lane i: run r0 + i).
struct SsTask {
    int q;          // task index (-1: none)
    int nr;         // runs in the task
    int32_t s;      // first sorted position of the lane's run
    int32_t e;
    int64_t key;
    int len;        // lookups of the lane's run if short, else 0
    int pre;        // exclusive prefix of len over the lanes
    int total;      // short-run lookups of the task
    int t;          // table of the lane's run
    float mom;      // momentum of the lane's row
};

// 2-byte weights with one vector per lane: registers for 12 CTAs per SM
// (shared memory allows 12; the kernel is latency-bound), no spill
template <typename WT, int NV> constexpr int ss_min_blocks() { return sizeof(WT) == 2 && NV == 1 ? 12 : 1; }

template <typename WT, int NV, bool LAY>
__global__ void __launch_bounds__(SS_WARPS * 32, ss_min_blocks<WT, NV>()) tbe_bwd_short_stream_kernel(const BwdParams p) {
    using ACC = typename WTraits<WT>::acc;
    // LAY: tables or bags with layouts; without, the layout code folds away
    const tbe_table_layout *layout = LAY ? p.layout : nullptr;
    const tbe_bag_layout *bag_layout = LAY ? p.bag_layout : nullptr;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int U_runs = p.counters[C_NUM_UNIQUE];
    const int wrow = p.D * (int)sizeof(WT);
    const int RT = ss_runs_per_task(wrow);
    const int ntasks = (U_runs + RT - 1) / RT;
    const int q0 = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (q0 >= ntasks) return;

    unsigned char *wsm = smem_raw + (threadIdx.x >> 5) * ss_warp_bytes();
    unsigned char *ring = wsm;
    unsigned char *wbuf = ring + SS_STAGES * STAGE_BYTES;                  // [2][SS_WBUF]
    uint32_t *tab_off = reinterpret_cast<uint32_t *>(wbuf + 2 * SS_WBUF);  // [2][32], 16-B units
    float *tab_w = reinterpret_cast<float *>(tab_off + 2 * SS_BLK);        // [2][32]
    uint32_t *tab_tag = reinterpret_cast<uint32_t *>(tab_w + 2 * SS_BLK);  // [2][32]
    const uint32_t bar0 = smem_addr(tab_tag + 2 * SS_BLK);                 // ring stages
    const uint32_t wbar0 = bar0 + 8 * SS_STAGES;                            // weight buffers
    if (lane == 0)
        for (int i = 0; i < SS_STAGES + 2; ++i) bar_init(bar0 + 8 * i, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();

    const uint32_t row_bytes = (uint32_t)p.D * 4;
    const int R = STAGE_BYTES / (int)row_bytes;   // gradient rows per stage (1..8)
    const int64_t TD = (int64_t)p.T * p.D;
    const float4 *G4 = reinterpret_cast<const float4 *>(p.G);

    // phase A: run bounds and keys of task q (loads only; lane i: run q*RT + i)
    auto task_load = [&](int q, SsTask &T) {
        T.q = q < ntasks ? q : -1;
        T.nr = T.q >= 0 ? min(RT, U_runs - q * RT) : 0;
        T.s = T.e = 0;
        T.key = 0;
        T.len = T.pre = T.total = T.t = 0;
        T.mom = 0.f;
        if (lane < T.nr) {
            T.s = __ldg(p.seg_off + q * RT + lane);
            T.e = __ldg(p.seg_off + q * RT + lane + 1);
            T.key = load_key(p, (int64_t)q * RT + lane);
        }
    };
    // phase B: lengths of the short runs, prefixes, tables, momentum; the
    // weight rows of the short runs are copied into weight buffer wb
    uint32_t wphase = 0;   // bit k: parity of weight buffer k's next completion
    auto task_prepare = [&](SsTask &T, int wb) {
        bool mine = T.q >= 0 && lane < T.nr && T.e - T.s < p.sl_threshold;
        int tt = 0;
        if (layout != nullptr) {   // the run's table decides its class first
            if (mine) tt = table_of_key(p.table_offset, p.T, T.key);
            mine = mine && in_class(layout, tt, p.D, p.cls_dtype);
        }
        T.len = mine ? T.e - T.s : 0;
        int x = T.len;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(FULL, x, o);
            if (lane >= o) x += y;
        }
        T.total = __shfl_sync(FULL, x, 31);
        T.pre = x - T.len;
        T.mom = mine ? p.mom[T.key] : 0.f;
        T.t = !mine ? 0 : (layout != nullptr ? tt : table_of_key(p.table_offset, p.T, T.key));
        const unsigned m = __ballot_sync(FULL, mine);
        if (m) {
            const uint32_t bar = wbar0 + 8 * wb;
            if (lane == 0) bar_arrive_expect_tx(bar, (uint32_t)__popc(m) * (uint32_t)wrow);
            __syncwarp();
            if (mine)
                bulk_g2s(smem_addr(wbuf + wb * SS_WBUF + lane * wrow), wrow_of<WT>(p, layout, T.t, T.key),
                         (uint32_t)wrow, bar);
        }
    };
    // table of block blk of task T (its lookups blk*32 + lane) into buffer tb
    auto stage_block = [&](const SsTask &T, int blk, int tb) {
        const int k = blk * SS_BLK + lane;
        // the lookup's run slot: the largest lane whose prefix is <= k (a
        // zero-length slot is never the largest such lane for k < total)
        int slot = 0;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1) {
            const int c = slot + step;
            const int pre_c = __shfl_sync(FULL, T.pre, c & 31);
            if (c < 32 && pre_c <= k) slot = c;
        }
        const int32_t s_sl = __shfl_sync(FULL, T.s, slot);
        const int pre_sl = __shfl_sync(FULL, T.pre, slot);
        const int len_sl = __shfl_sync(FULL, T.len, slot);
        const int t_sl = __shfl_sync(FULL, T.t, slot);
        if (k < T.total) {
            const uint32_t v = __ldg(p.vals + s_sl + (k - pre_sl));
            const int64_t b = payload_bag(p, bag_layout, v, t_sl);
            float x = 1.f;
            if (p.payload_pos && p.psw != nullptr &&
                (p.weighted == nullptr || __ldg(p.weighted + t_sl) != 0))
                x = __ldg(p.psw + v);
            // only malformed (overlapping) offsets can give a bag outside the
            // run's table: such a lookup copies row 0 with weight 0
            const bool ok = b >= 0 && b < bags_of(p, bag_layout, t_sl);
            const int64_t g0 = bag_layout ? __ldg(&bag_layout[t_sl].out_offset) : (int64_t)t_sl * p.D;
            const int64_t gs = bag_layout ? __ldg(&bag_layout[t_sl].out_stride) : TD;
            tab_off[tb * SS_BLK + lane] = ok ? (uint32_t)((g0 + b * gs) >> 2) : 0u;
            tab_w[tb * SS_BLK + lane] = ok ? x : 0.f;
            tab_tag[tb * SS_BLK + lane] = (uint32_t)slot | (k == pre_sl + len_sl - 1 ? SS_LAST : 0u);
        }
        __syncwarp();
    };
    auto nblocks = [&](const SsTask &T) { return (T.total + SS_BLK - 1) / SS_BLK; };

    uint32_t gprod = 0, gcons = 0, phase = 0;
    auto produce = [&](const SsTask &T, int blk, int tb, int sb) {
        const int st = (int)(gprod % SS_STAGES);
        const int rows = min(R, T.total - blk * SS_BLK - sb * R);
        const uint32_t bar = bar0 + 8 * st;
        if (lane == 0) bar_arrive_expect_tx(bar, (uint32_t)rows * row_bytes);
        __syncwarp();
        const uint32_t dst0 = smem_addr(ring + st * STAGE_BYTES);
        for (int j = lane; j < rows; j += 32)
            bulk_g2s(dst0 + j * row_bytes, G4 + tab_off[tb * SS_BLK + sb * R + j], row_bytes, bar);
        ++gprod;
    };

    // Tasks: cur (consumed now, weight buffer cw), nxt (prepared: weight rows
    // copied into buffer cw ^ 1), nn (run bounds loaded).  Moving on makes nxt
    // current and prepares the task after it into the buffer just released.
    SsTask cur, nxt, nn;
    int cw = 0;
    task_load(q0, cur);
    task_load(q0 + nwarps, nxt);
    task_load(q0 + 2 * nwarps, nn);
    task_prepare(cur, 0);
    task_prepare(nxt, 1);
    auto advance = [&]() {
        cur = nxt;
        cw ^= 1;
        nxt = nn;
        task_load(cur.q >= 0 ? cur.q + 2 * nwarps : ntasks, nn);
        task_prepare(nxt, cw ^ 1);
    };
    while (cur.q >= 0 && cur.total == 0) advance();
    if (cur.q < 0) return;

    // Blocks are numbered in consumption order; block n uses table buffer n&1.
    // consumer: block cn = block cblk of task cur
    // staged:   the newest block whose table is staged (cn or cn + 1)
    // producer: block pn (cn or cn + 1), next stage psb
    int cblk = 0;
    uint32_t cn = 0, staged = 0, pn = 0;
    int psb = 0;
    stage_block(cur, 0, 0);

    auto refill = [&]() {
        while (gprod - gcons < (uint32_t)SS_STAGES && pn <= staged) {
            const bool in_cur = pn == cn || cblk + 1 < nblocks(cur);
            const SsTask &T = in_cur ? cur : nxt;
            const int blk = pn == cn ? cblk : (in_cur ? cblk + 1 : 0);
            const int nsb = (min(SS_BLK, T.total - blk * SS_BLK) + R - 1) / R;
            if (psb < nsb) {
                produce(T, blk, (int)(pn & 1), psb++);
                continue;
            }
            if (pn != cn) break;   // at most one block ahead of the consumer
            ++pn;
            psb = 0;
        }
    };
    refill();

    ACC acc[NV][4];
#pragma unroll
    for (int q = 0; q < NV; ++q)
#pragma unroll
        for (int x = 0; x < 4; ++x) acc[q][x] = ACC(0);
    bool wready = false;   // the current task's weight rows have landed

    for (;;) {
        // stage the table of the block after the consumer's
        if (staged == cn) {
            if (cblk + 1 < nblocks(cur)) {
                stage_block(cur, cblk + 1, (int)((cn + 1) & 1));
                staged = cn + 1;
            } else if (nxt.q >= 0 && nxt.total > 0) {
                stage_block(nxt, 0, (int)((cn + 1) & 1));
                staged = cn + 1;
            }
        }
        refill();
        const int tb = (int)(cn & 1);
        const int rows_blk = min(SS_BLK, cur.total - cblk * SS_BLK);
        const int nsb = (rows_blk + R - 1) / R;
        for (int sb = 0; sb < nsb; ++sb) {
            const int st = (int)(gcons % SS_STAGES);
            if (!mbar_wait_bounded(bar0 + 8 * st, (phase >> st) & 1u)) {
                // stop issuing: give the copies still in flight one more
                // bounded wait each, flag the failure, end the warp's work
                for (uint32_t g = gcons + 1; g < gprod; ++g)
                    mbar_wait_bounded(bar0 + 8 * (g % SS_STAGES), (phase >> (g % SS_STAGES)) & 1u);
                if (lane == 0) atomicOr(p.status + 1, TBE_FLAG_COPY_TIMEOUT);
                return;
            }
            phase ^= 1u << st;
            const int rows = min(R, rows_blk - sb * R);
            const unsigned char *sp = ring + st * STAGE_BYTES;
            for (int j = 0; j < rows; ++j) {
                const int e = tb * SS_BLK + sb * R + j;
                const float x = tab_w[e];
                const uint32_t tag = tab_tag[e];
                const float4 *src = reinterpret_cast<const float4 *>(sp + j * row_bytes) + lane;
#pragma unroll
                for (int q = 0; q < NV; ++q) acc4(acc[q], src[q * 32], x);
                if (!(tag & SS_LAST)) continue;
                // the run in slot (tag & 31) is complete: exact rowwise Adagrad
                //   m += mean_d(g^2);  w -= lr * g / (sqrt(m) + eps)
                if (!wready) {
                    if (!mbar_wait_bounded(wbar0 + 8 * cw, (wphase >> cw) & 1u)) {
                        for (uint32_t g = gcons + 1; g < gprod; ++g)
                            mbar_wait_bounded(bar0 + 8 * (g % SS_STAGES), (phase >> (g % SS_STAGES)) & 1u);
                        if (lane == 0) atomicOr(p.status + 1, TBE_FLAG_COPY_TIMEOUT);
                        return;
                    }
                    wphase ^= 1u << cw;
                    wready = true;
                }
                const int slot = (int)(tag & 31u);
                using A = Adagrad<ACC>;
                ACC g[NV][4];
                ACC ss = ACC(0);
#pragma unroll
                for (int q = 0; q < NV; ++q)
#pragma unroll
                    for (int x2 = 0; x2 < 4; ++x2) {
                        g[q][x2] = acc[q][x2];
                        ss += g[q][x2] * g[q][x2];
                        acc[q][x2] = ACC(0);
                    }
#pragma unroll
                for (int sh = 1; sh < 32; sh <<= 1) ss += __shfl_xor_sync(FULL, ss, sh);
                const float m_old = __shfl_sync(FULL, cur.mom, slot);
                const int64_t key = __shfl_sync(FULL, cur.key, slot);
                const int tk = __shfl_sync(FULL, cur.t, slot);
                const float m_new = A::mom(m_old, ss, p.D);
                const auto den = A::den(m_new, p.eps);
                const WT *wsrc = reinterpret_cast<const WT *>(wbuf + cw * SS_WBUF + slot * wrow) + lane * 4;
                WT *wdst = wrow_of<WT>(p, layout, tk, key) + lane * 4;
#pragma unroll
                for (int q = 0; q < NV; ++q) {
                    float w[4];
                    ld4(wsrc + q * 128, w);
#pragma unroll
                    for (int x2 = 0; x2 < 4; ++x2) w[x2] = A::step(w[x2], g[q][x2], p.lr, den);
                    st4(wdst + q * 128, w);
                }
                if (lane == 0) p.mom[key] = m_new;
            }
            ++gcons;
            __syncwarp();   // the stage is read before it is refilled
            refill();
        }
        if (cblk + 1 < nblocks(cur)) {
            ++cblk;
            ++cn;
            continue;
        }
        // task done: the next task with short-run lookups becomes current
        do {
            advance();
        } while (cur.q >= 0 && cur.total == 0);
        if (cur.q < 0) break;
        wready = false;
        cblk = 0;
        ++cn;
        if (staged < cn) {   // empty tasks were skipped: the table is not staged yet
            stage_block(cur, 0, (int)(cn & 1));
            staged = cn;
        }
        if (pn < cn) {
            pn = cn;
            psb = 0;
        }
    }
}

template <typename WT, int LPR, int NV>
__global__ void __launch_bounds__(256) tbe_bwd_apply_kernel(const BwdParams p) {
    using ACC = typename WTraits<WT>::acc;
    const int lane = threadIdx.x & 31, sub = lane / LPR, li = lane % LPR;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int nlong = p.counters[C_NUM_LONG];
    for (int l = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; l < nlong; l += nwarps) {
        const int r = __ldg(p.long_run + l);
        const int cb = __ldg(p.long_chunk_base + l);
        const int32_t rs = __ldg(p.seg_off + r), re = __ldg(p.seg_off + r + 1);
        const int nch = (re - rs + p.chunk - 1) / p.chunk;
        const int64_t key = load_key(p, r);
        const int t = table_of_key(p.table_offset, p.T, key);
        if (!in_class(p.layout, t, p.D, p.cls_dtype)) continue;   // warp-uniform
        ACC acc[NV][4];
#pragma unroll
        for (int q = 0; q < NV; ++q)
#pragma unroll
            for (int x = 0; x < 4; ++x) acc[q][x] = ACC(0);
        // (16 partial rows in flight instead of 4 measured the same)
        if (sub == 0) sum_partials<false, ACC, LPR, NV>(acc, p.partials, p.part_stride, cb, nch, li);
        adagrad_apply<WT, ACC, LPR, NV>(acc, p, p.layout, t, key, lane, sub, li);
    }
}


// ---------------------------------------------------------------------------

template <typename K>
inline int persistent_grid(const Launch &L, K kernel, size_t smem = 0, int threads = 256) {
    return L.num_sms * cached_blocks_per_sm(L.dev, (const void *)kernel, threads, smem);
}

// lanes per run of the short-run kernel, for a gradient row of V 16-byte
// vectors (V a power of two up to 32, or 64, 96, 128): the whole row up to
// 16 lanes, 16 lanes for 32 vectors, else 32 lanes.  Measured: 4-vector rows
// (demo workload) 0.195 ms in 4-lane groups vs 0.252 in 2-lane and 0.406 in
// 1-lane groups; 32-vector rows (large workload) 2.19 ms in 16-lane groups vs
// 2.62 in 8-lane and 3.00 in 32-lane groups.
static constexpr int short_group_lanes(int V) { return V <= 16 ? V : V <= 32 ? 16 : 32; }

#ifndef TBE_CHUNK_MAXB
#define TBE_CHUNK_MAXB 0   // cap on long-run blocks per SM (0: as many as fit; a cap of 4: 3.64 vs 3.30 ms)
#endif
template <typename WT, int LPR, int NV, bool FUSED>
inline void chunk_launch(Launch &L, const BwdParams &p) {
    const bool lay = p.layout != nullptr || p.bag_layout != nullptr;
    const bool wgt = p.psw != nullptr;
    auto kc = lay ? (wgt ? tbe_bwd_chunk_kernel<WT, LPR, NV, FUSED, true, true>
                         : tbe_bwd_chunk_kernel<WT, LPR, NV, FUSED, true, false>)
                  : (wgt ? tbe_bwd_chunk_kernel<WT, LPR, NV, FUSED, false, true>
                         : tbe_bwd_chunk_kernel<WT, LPR, NV, FUSED, false, false>);
    const size_t csm = (size_t)(CHUNK_THREADS / 32) * warp_smem_bytes(p.chunk, wgt);
    cached_smem_attr(L.dev, (const void *)kc, csm);
    L.before(FUSED ? "tbe_bwd_fused_long" : "tbe_bwd_grad_accum");
    int grid = persistent_grid(L, kc, csm, CHUNK_THREADS);
    if (TBE_CHUNK_MAXB > 0 && grid > L.num_sms * TBE_CHUNK_MAXB) grid = L.num_sms * TBE_CHUNK_MAXB;
    kc<<<grid, CHUNK_THREADS, csm, L.stream>>>(p);
    L.after();
}

template <typename WT, int LPR, int NV>
inline void bwd_launch(Launch &L, const BwdParams &p, int long_mode) {
    if (long_mode == TBE_LONG_TWO_KERNEL) chunk_launch<WT, LPR, NV, false>(L, p);
    else chunk_launch<WT, LPR, NV, true>(L, p);
    bool stream = false;
    if constexpr (LPR == 32 && TBE_SHORT_STREAM) stream = p.payload_pos != 0;
    if (stream) {
        // weighted batch, gradient rows of 512 bytes and more: short runs
        // streamed through a bulk-copy ring, one row per warp step; staging
        // 32 lookups at a time amortises the dependent bag lookup of a
        // position payload (2.60 vs 2.82 ms on the mid workload, while the
        // register kernel stays ahead on unweighted batches, 2.55 vs 2.80 ms
        // on the large one)
        auto ks = (p.layout != nullptr || p.bag_layout != nullptr) ? tbe_bwd_short_stream_kernel<WT, NV, true>
                                                                   : tbe_bwd_short_stream_kernel<WT, NV, false>;
        const size_t ssm = (size_t)SS_WARPS * ss_warp_bytes();
        cached_smem_attr(L.dev, (const void *)ks, ssm);
        L.before("tbe_bwd_short_run");
        ks<<<persistent_grid(L, ks, ssm, SS_WARPS * 32), SS_WARPS * 32, ssm, L.stream>>>(p);
        L.after();
    }
    if (!stream) {
        // short runs: GL lanes per run, 4 gradient vectors per lane where the row allows
        constexpr int V = LPR * NV;                       // float4 vectors per gradient row
        constexpr int SGL = short_group_lanes(V);
        constexpr int SNV = V / SGL;
        static_assert(SGL >= 1 && SGL <= 32 && (32 % SGL) == 0 && SNV * SGL == V && SNV <= 4,
                      "short-run lane groups");
        constexpr int SU = TBE_SHORT_U > 0 ? TBE_SHORT_U : SNV >= 3 ? 2 : 4;
        auto ks = (p.layout != nullptr || p.bag_layout != nullptr) ? tbe_bwd_short_kernel<WT, SGL, SNV, SU, true>
                                                                   : tbe_bwd_short_kernel<WT, SGL, SNV, SU, false>;
        L.before("tbe_bwd_short_run");
        ks<<<persistent_grid(L, ks, 0, TBE_SHORT_THREADS), TBE_SHORT_THREADS, 0, L.stream>>>(p);
        L.after();
    }
    if (long_mode == TBE_LONG_TWO_KERNEL) {
        auto ka = tbe_bwd_apply_kernel<WT, LPR, NV>;
        L.before("tbe_bwd_apply");
        ka<<<persistent_grid(L, ka), 256, 0, L.stream>>>(p);
        L.after();
    }
}

template <typename WT>
inline bool bwd_dispatch(Launch &L, const BwdParams &p, RowPlan rp, int long_mode) {
    switch (rp.lpr * 10 + rp.nv) {
    case 11: bwd_launch<WT, 1, 1>(L, p, long_mode); return true;
    case 21: bwd_launch<WT, 2, 1>(L, p, long_mode); return true;
    case 41: bwd_launch<WT, 4, 1>(L, p, long_mode); return true;
    case 81: bwd_launch<WT, 8, 1>(L, p, long_mode); return true;
    case 161: bwd_launch<WT, 16, 1>(L, p, long_mode); return true;
    case 321: bwd_launch<WT, 32, 1>(L, p, long_mode); return true;
    case 322: bwd_launch<WT, 32, 2>(L, p, long_mode); return true;
    case 323: bwd_launch<WT, 32, 3>(L, p, long_mode); return true;
    case 324: bwd_launch<WT, 32, 4>(L, p, long_mode); return true;
    default: return false;
    }
}

}  // namespace tbe
