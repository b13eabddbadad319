// Forward pooled-sum gather with fused bounds check, and the linearize step
// of the batch inversion.
//
// FBTriton TBE redesign (accesspath.com): "Backward kernels" (notation T, E,
// D, L, B), decision checklist items 1 (FP32 accumulation for FP16/BF16
// weights, FP64 for FP32 weights), 5 (bounds check fused into the lookup)
// and 6 (int32 linearised keys); "Forward state reuse and preprocessing"
// (the linearize/sort/RLE work may run inside the forward).  TorchEasyRec
// analysis (39.107.221.112 article 1724244), section 1: one fused lookup over
// the KeyedJagged CSR input of all tables.
//
// Design: one warp per bag, persistent grid-stride over the T*B bags.  A row
// of D elements is read as 16-byte vectors by LPR lanes (NV vectors each), so
// a warp gathers 32/LPR rows per step and keeps U steps of loads in flight
// before accumulating.  Sub-group partial sums are combined with shuffles and
// the pooled row is written once.  When preprocessing runs in the forward,
// the same pass writes the linearised key and the sort payload of every
// lookup (coalesced, in position order).  Indices and offsets are int32 or
// int64 (kernels templated on the index type IdxT); keys are written here
// only when they are 32-bit, the 64-bit keys of row ranges of 2^31 and more
// come from the linearize kernel.
#include <string.h>

#include <algorithm>
#include <type_traits>

#include "tbe_internal.cuh"

namespace tbe {

// Tables of one launch: with layouts, a launch serves the tables of one
// (D, dtype) class, at most FWD_TLIST per launch.
constexpr int FWD_TLIST = 256;

struct FwdParams {
    const void *W;
    const int64_t *table_offset;
    const tbe_table_layout *layout;     // nullable: uniform tables
    const tbe_bag_layout *bag_layout;   // nullable: uniform bags and output rows
    int ntl;                            // tables of this launch (0: all, uniform bags)
    int32_t tlist[FWD_TLIST];           // their ids
    int64_t tcum[FWD_TLIST + 1];        // their bags, cumulative
    const void *indices;   // IdxT [N]
    const void *offsets;   // IdxT [NB+1]
    const float *psw;
    const uint8_t *weighted;
    float *out;
    void *keys;            // KeyT [N] (uint32 in the forward kernel)
    uint32_t *vals;
    int32_t *bag_of;
    int32_t *status;
    int32_t *counters;   // nullable: C_MALFORMED / C_DECREASING
    int64_t B;
    int64_t NB;
    int64_t N;
    int T;
    int D;
    uint64_t sentinel;
    int payload_pos;
};

// A VB-byte vector of a weight row (VB = 8 or 16) as 32-bit words.
template <int VB> struct Vec {
    uint32_t v[VB / 4];
};
template <int VB> __device__ __forceinline__ Vec<VB> ldg_vec(const void *p) {
    Vec<VB> r;
    if constexpr (VB == 16) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(p));
        r.v[0] = q.x; r.v[1] = q.y; r.v[2] = q.z; r.v[3] = q.w;
    } else {
        const uint2 q = __ldg(reinterpret_cast<const uint2 *>(p));
        r.v[0] = q.x; r.v[1] = q.y;
    }
    return r;
}

#ifndef TBE_FWD_MIXED_ADD
#define TBE_FWD_MIXED_ADD 1
#endif
// a += element 0, b += element 1 of two packed 16-bit values: one FP32 add
// per element that takes the 16-bit operand directly (its widening to FP32
// is exact, so the sum is the FP32 sum of the widened values)
template <typename WT> __device__ __forceinline__ void add2(float &a, float &b, uint32_t x) {
    if constexpr (std::is_same<WT, __half>::value)
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
            : "+f"(a), "+f"(b) : "r"(x));
    else
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
            : "+f"(a), "+f"(b) : "r"(x));
}

// acc[e] += w * element e of the vector (FP64 accumulators for FP32 tables);
// UNIT: w is 1 (unweighted), so 16-bit elements are added without a multiply
template <typename WT, int VB, bool UNIT = false, typename ACC>
__device__ __forceinline__ void accum(ACC (&a)[VB / sizeof(WT)], const Vec<VB> &x, float w) {
    constexpr int NW = VB / 4;
    if constexpr (sizeof(WT) == 2 && UNIT && TBE_FWD_MIXED_ADD) {
#pragma unroll
        for (int e = 0; e < NW; ++e) add2<WT>(a[2 * e], a[2 * e + 1], x.v[e]);
    } else if constexpr (sizeof(WT) == 4) {
#pragma unroll
        for (int e = 0; e < NW; ++e) a[e] = fma((double)w, (double)__uint_as_float(x.v[e]), a[e]);
    } else {
#pragma unroll
        for (int e = 0; e < NW; ++e) {
            float2 f;
            if constexpr (std::is_same<WT, __half>::value)
                f = __half22float2(*reinterpret_cast<const __half2 *>(&x.v[e]));
            else
                f = bf16x2_to_float2(x.v[e]);
            a[2 * e] = fmaf(w, f.x, a[2 * e]);
            a[2 * e + 1] = fmaf(w, f.y, a[2 * e + 1]);
        }
    }
}

template <int VEC, typename ACC> __device__ __forceinline__ void store_out(float *o, const ACC (&a)[VEC]) {
    if constexpr (VEC % 4 == 0) {
#pragma unroll
        for (int i = 0; i < VEC / 4; ++i)
            __stcs(reinterpret_cast<float4 *>(o) + i,
                   make_float4((float)a[4 * i], (float)a[4 * i + 1], (float)a[4 * i + 2], (float)a[4 * i + 3]));
    } else {
        __stcs(reinterpret_cast<float2 *>(o), make_float2((float)a[0], (float)a[1]));
    }
}

template <typename IdxT> __device__ __forceinline__ int64_t ld_off(const FwdParams &p, int64_t g) {
    return (int64_t)__ldg(reinterpret_cast<const IdxT *>(p.offsets) + g);
}

// Lookup range of bag g.  Well-formed: 0 <= start <= end <= N; a malformed
// bag is made empty, flagged in the status word and recorded in the
// counters (if any).
template <typename IdxT>
__device__ __forceinline__ void read_bag(const FwdParams &p, int64_t g, bool leader, int32_t &start,
                                         int32_t &end) {
    const int64_t s = ld_off<IdxT>(p, g), e = ld_off<IdxT>(p, g + 1);
    start = (int32_t)s;
    end = (int32_t)e;
    if (s <= e && s >= 0 && e <= p.N) return;
    if (leader) {
        atomicOr(p.status + 1, TBE_FLAG_BAD_OFFSETS);
        if (p.counters != nullptr) {
            p.counters[C_MALFORMED] = 1;
            if (e < s) p.counters[C_DECREASING] = 1;
        }
    }
    start = end = 0;
}

// offsets[0] != 0 or offsets[T*B] != N leaves lookups outside every bag
template <typename IdxT> __device__ __forceinline__ void check_span(const FwdParams &p) {
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    if (ld_off<IdxT>(p, 0) != 0 || ld_off<IdxT>(p, p.NB) != p.N) {
        atomicOr(p.status + 1, TBE_FLAG_BAD_OFFSETS);
        if (p.counters != nullptr) p.counters[C_MALFORMED] = 1;
    }
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) v += __shfl_xor_sync(FULL, v, s);
    return v;
}

// The kernel is issue-bound (most row reads hit L2), so the inner loop is
// kept short: full steps of 32/LPR*U rows whose lookups are all in range run
// without predicates or branches; the rest of a 32-lookup block (and any
// block with an out-of-range index) goes one 32/LPR-row step at a time with
// per-row checks.  (t, b) of the next bag are stepped, not divided.
template <typename WT, int VB, int LPR, int NV, int U, bool WEIGHTED, typename IdxT, bool LAY>
__global__ void __launch_bounds__(256) tbe_fwd_kernel(const __grid_constant__ FwdParams p) {
    // LAY: tables or bags with layouts, one class of tables per launch;
    // without, the layout code folds away
    const int ntl = LAY ? p.ntl : 0;
    const tbe_table_layout *layout = LAY ? p.layout : nullptr;
    const tbe_bag_layout *bag_layout = LAY ? p.bag_layout : nullptr;
    using ACC = typename WTraits<WT>::acc;
    constexpr int VEC = VB / (int)sizeof(WT);   // elements per lane vector
    constexpr int RPI = 32 / LPR;
    constexpr int STEP = RPI * U;               // rows of a full step
    const int lane = threadIdx.x & 31, sub = lane / LPR, li = lane % LPR;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    // work item k: bag k of all tables (uniform: (t, b) stepped without
    // division), or bag k of this launch's class tables (table found in the
    // cumulative bag counts)
    int64_t k = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nitems = ntl ? p.tcum[ntl] : p.NB;
    int t = ntl ? 0 : (int)(k / p.B);
    int64_t b = ntl ? 0 : k - (int64_t)t * p.B;
    const int tstep = ntl ? 0 : (int)(nwarps / p.B);
    const int64_t bstep = ntl ? 0 : nwarps - (int64_t)tstep * p.B;
    int oob = 0;
    check_span<IdxT>(p);
    uint32_t *keys = reinterpret_cast<uint32_t *>(p.keys);
    const IdxT *indices = reinterpret_cast<const IdxT *>(p.indices);
    for (; k < nitems; k += nwarps) {
        int64_t bag = k;
        if (ntl) {
            int lo = 0, hi = ntl;   // class table lo: tcum[lo] <= k < tcum[lo+1]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (p.tcum[mid] <= k) lo = mid; else hi = mid;
            }
            t = p.tlist[lo];
            b = k - p.tcum[lo];
            bag = bag_base(bag_layout, p.B, t) + b;
        }
        const int64_t row0 = __ldg(p.table_offset + t);
        const int64_t E = __ldg(p.table_offset + t + 1) - row0;
        int32_t start, end;
        read_bag<IdxT>(p, bag, lane == 0, start, end);
        const bool wt = WEIGHTED && (p.weighted == nullptr || __ldg(p.weighted + t) != 0);
        const WT *Wt = reinterpret_cast<const WT *>(reinterpret_cast<const char *>(p.W) +
                                                    weight_byte(layout, p.table_offset, t, row0, p.D,
                                                                (int)sizeof(WT))) + li * VEC;
        ACC acc[NV][VEC];
#pragma unroll
        for (int q = 0; q < NV; ++q)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[q][e] = ACC(0);

        for (int32_t base = start; base < end; base += 32) {
            const int n = min(32, end - base);
            IdxT idx = 0;
            float w = 1.f;
            if (lane < n) {
                idx = __ldg(indices + base + lane);
                if (wt) w = __ldg(p.psw + base + lane);
            }
            const bool valid = lane < n && idx >= 0 && (int64_t)idx < E;
            oob += (lane < n) && !valid;
            if (keys != nullptr && lane < n) {
                keys[base + lane] = valid ? (uint32_t)(row0 + idx) : (uint32_t)p.sentinel;
                p.vals[base + lane] = p.payload_pos ? (uint32_t)(base + lane) : (uint32_t)b;
                if (p.bag_of != nullptr) p.bag_of[base + lane] = (int32_t)bag;
            }
            const unsigned vmask = __ballot_sync(FULL, valid);
            // full steps while every lookup of the block is in range
            int j = 0;
            if (vmask == (n == 32 ? FULL : ((1u << n) - 1u))) {
                for (; j + STEP <= n; j += STEP) {
                    Vec<VB> v[U][NV];
                    float wv[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const IdxT ik = __shfl_sync(FULL, idx, j + u * RPI + sub);
                        wv[u] = WEIGHTED ? __shfl_sync(FULL, w, j + u * RPI + sub) : 1.f;
                        const WT *r = Wt + (int64_t)ik * p.D;
#pragma unroll
                        for (int q = 0; q < NV; ++q) v[u][q] = ldg_vec<VB>(r + q * LPR * VEC);
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int q = 0; q < NV; ++q) accum<WT, VB, !WEIGHTED>(acc[q], v[u][q], wv[u]);
                }
            }
            // the rest, one 32/LPR-row step at a time
            for (; j < n; j += RPI) {
                const int k = j + sub;
                const int src = k & 31;
                const IdxT ik = __shfl_sync(FULL, idx, src);
                const float wk = WEIGHTED ? __shfl_sync(FULL, w, src) : 1.f;
                if (k < n && ((vmask >> src) & 1u)) {
                    const WT *r = Wt + (int64_t)ik * p.D;
                    Vec<VB> v[NV];
#pragma unroll
                    for (int q = 0; q < NV; ++q) v[q] = ldg_vec<VB>(r + q * LPR * VEC);
#pragma unroll
                    for (int q = 0; q < NV; ++q) accum<WT, VB, !WEIGHTED>(acc[q], v[q], wk);
                }
            }
        }
#pragma unroll
        for (int s = LPR; s < 32; s <<= 1)
#pragma unroll
            for (int q = 0; q < NV; ++q)
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[q][e] += __shfl_xor_sync(FULL, acc[q][e], s);
        if (sub == 0) {
            float *o = p.out + out_row(bag_layout, p.T, p.D, t, b) + li * VEC;
#pragma unroll
            for (int q = 0; q < NV; ++q) store_out<VEC>(o + q * LPR * VEC, acc[q]);
        }
        if (!ntl) {
            t += tstep;
            b += bstep;
            if (b >= p.B) {
                b -= p.B;
                ++t;
            }
        }
    }
    oob = warp_sum_i(oob);
    if (lane == 0 && oob) atomicAdd(p.status, oob);
}

// 256-thread blocks per SM the register budget must allow.  Large workload:
// 8 (32 registers, a few spilled, a full SM of warps) 2.05 ms; without a
// bound the compiler's 40 registers 2.20 ms; 5 blocks 2.35 ms.  (The next
// round's index loaded with the current round's: 2.31.)
#ifndef TBE_FWD_GROUP_MINB
#define TBE_FWD_GROUP_MINB 8
#endif
// (with layouts, whose code needs more registers, 6 blocks: 40 registers)
template <bool LAY> constexpr int fwd_group_minb() { return LAY ? 6 : TBE_FWD_GROUP_MINB; }

// Rows of at most 16 lanes: one bag per group of LPR lanes, 32/LPR bags per
// warp.  Each warp instruction then serves several bags, so the per-bag work
// (offsets, table bounds, index and key traffic, output store) is shared,
// and a bag needs no cross-lane reduction.  Lookups go in rounds of LPR (one
// index per lane); within a round the groups step through their lookups
// together, U rows per step without predicates while every group has that
// many valid lookups left, then one row per step with a per-group check.
template <typename WT, int VB, int LPR, int NV, int U, bool WEIGHTED, typename IdxT, bool LAY>
__global__ void __launch_bounds__(256, fwd_group_minb<LAY>()) tbe_fwd_group_kernel(const __grid_constant__ FwdParams p) {
    static_assert(LPR <= 16, "groups of at most half a warp");
    const int ntl = LAY ? p.ntl : 0;
    const tbe_table_layout *layout = LAY ? p.layout : nullptr;
    const tbe_bag_layout *bag_layout = LAY ? p.bag_layout : nullptr;
    using ACC = typename WTraits<WT>::acc;
    constexpr int VEC = VB / (int)sizeof(WT);   // elements per lane vector
    constexpr int GPW = 32 / LPR;               // bags per warp
    const int lane = threadIdx.x & 31, grp = lane / LPR, li = lane % LPR;
    const int gbase = grp * LPR;                // first lane of the group
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t S = nwarps * GPW;             // bags per grid step
    int64_t k = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * GPW + grp;
    const int64_t nitems = ntl ? p.tcum[ntl] : p.NB;
    int t = ntl ? 0 : (int)(k / p.B);
    int64_t b = ntl ? 0 : k - (int64_t)t * p.B;
    const int tstep = ntl ? 0 : (int)(S / p.B);
    const int64_t bstep = ntl ? 0 : S - (int64_t)tstep * p.B;
    int oob = 0;
    check_span<IdxT>(p);
    uint32_t *keys = reinterpret_cast<uint32_t *>(p.keys);
    const IdxT *indices = reinterpret_cast<const IdxT *>(p.indices);
    for (;; k += S) {
        const bool active = k < nitems;
        if (!__any_sync(FULL, active)) break;
        int64_t bag = k;
        int32_t start = 0, end = 0;
        int64_t row0 = 0, E = 0;
        bool wt = false;
        if (active) {
            if (ntl) {
                int lo = 0, hi = ntl;   // class table lo: tcum[lo] <= k < tcum[lo+1]
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (p.tcum[mid] <= k) lo = mid; else hi = mid;
                }
                t = p.tlist[lo];
                b = k - p.tcum[lo];
                bag = bag_base(bag_layout, p.B, t) + b;
            }
            row0 = __ldg(p.table_offset + t);
            E = __ldg(p.table_offset + t + 1) - row0;
            read_bag<IdxT>(p, bag, li == 0, start, end);
            wt = WEIGHTED && (p.weighted == nullptr || __ldg(p.weighted + t) != 0);
        }
        const int n = end - start;
        const WT *Wt = reinterpret_cast<const WT *>(reinterpret_cast<const char *>(p.W) +
                                                    weight_byte(layout, p.table_offset, t, row0, p.D,
                                                                (int)sizeof(WT))) + li * VEC;
        ACC acc[NV][VEC];
#pragma unroll
        for (int q = 0; q < NV; ++q)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[q][e] = ACC(0);

        const int nmax = __reduce_max_sync(FULL, n);
        for (int32_t base = 0; base < nmax; base += LPR) {
            const int m = max(0, min(LPR, n - base));   // this group's lookups in the round
            const int32_t pos = start + base + li;
            IdxT idx = 0;
            float w = 1.f;
            if (li < m) {
                idx = __ldg(indices + pos);
                if (wt) w = __ldg(p.psw + pos);
            }
            const bool valid = li < m && idx >= 0 && (int64_t)idx < E;
            oob += (li < m) && !valid;
            if (keys != nullptr && li < m) {
                keys[pos] = valid ? (uint32_t)(row0 + idx) : (uint32_t)p.sentinel;
                p.vals[pos] = p.payload_pos ? (uint32_t)pos : (uint32_t)b;
                if (p.bag_of != nullptr) p.bag_of[pos] = (int32_t)bag;
            }
            const unsigned vmask = __ballot_sync(FULL, valid);
            const unsigned gmask = (vmask >> gbase) & (LPR == 32 ? FULL : ((1u << LPR) - 1u));
            // lookups every group can take without checks: a group whose
            // round is all valid offers m of them, any other none
            const bool gfull = gmask == (m >= 32 ? FULL : ((1u << m) - 1u));
            const int mfull = __reduce_min_sync(FULL, gfull ? m : 0);
            const int mrnd = __reduce_max_sync(FULL, m);
            int j = 0;
            for (; j + U <= mfull; j += U) {
                Vec<VB> v[U][NV];
                float wv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const IdxT ik = __shfl_sync(FULL, idx, gbase + j + u);
                    wv[u] = WEIGHTED ? __shfl_sync(FULL, w, gbase + j + u) : 1.f;
                    const WT *r = Wt + (int64_t)ik * p.D;
#pragma unroll
                    for (int q = 0; q < NV; ++q) v[u][q] = ldg_vec<VB>(r + q * LPR * VEC);
                }
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int q = 0; q < NV; ++q) accum<WT, VB, !WEIGHTED>(acc[q], v[u][q], wv[u]);
            }
            for (; j < mrnd; ++j) {
                const int src = gbase + j;
                const IdxT ik = __shfl_sync(FULL, idx, src);
                const float wk = WEIGHTED ? __shfl_sync(FULL, w, src) : 1.f;
                if ((vmask >> src) & 1u) {
                    const WT *r = Wt + (int64_t)ik * p.D;
                    Vec<VB> v[NV];
#pragma unroll
                    for (int q = 0; q < NV; ++q) v[q] = ldg_vec<VB>(r + q * LPR * VEC);
#pragma unroll
                    for (int q = 0; q < NV; ++q) accum<WT, VB, !WEIGHTED>(acc[q], v[q], wk);
                }
            }
        }
        if (active) {
            float *o = p.out + out_row(bag_layout, p.T, p.D, t, b) + li * VEC;
#pragma unroll
            for (int q = 0; q < NV; ++q) store_out<VEC>(o + q * LPR * VEC, acc[q]);
        }
        if (!ntl) {
            t += tstep;
            b += bstep;
            if (b >= p.B) {
                b -= p.B;
                ++t;
            }
        }
    }
    oob = warp_sum_i(oob);
    if (lane == 0 && oob) atomicAdd(p.status, oob);
}

// Linearize alone (the batch inversion's first step when it runs at the
// start of the backward, or when keys are 64-bit): one warp per bag writes
// key and payload of every lookup; out-of-range lookups get the sentinel key
// (the forward counts them).
template <typename IdxT, typename KeyT>
__global__ void __launch_bounds__(256) tbe_linearize_kernel(const __grid_constant__ FwdParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    check_span<IdxT>(p);
    KeyT *keys = reinterpret_cast<KeyT *>(p.keys);
    const IdxT *indices = reinterpret_cast<const IdxT *>(p.indices);
    for (int64_t bag = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; bag < p.NB;
         bag += nwarps) {
        const int t = table_of_bag(p.bag_layout, p.B, p.T, bag);
        const int64_t b = bag - bag_base(p.bag_layout, p.B, t);
        const int64_t row0 = __ldg(p.table_offset + t);
        const int64_t E = __ldg(p.table_offset + t + 1) - row0;
        int32_t start, end;
        read_bag<IdxT>(p, bag, lane == 0, start, end);
        for (int32_t i = start + lane; i < end; i += 32) {
            const IdxT idx = __ldg(indices + i);
            const bool valid = idx >= 0 && (int64_t)idx < E;
            keys[i] = valid ? (KeyT)(row0 + idx) : (KeyT)p.sentinel;
            p.vals[i] = p.payload_pos ? (uint32_t)i : (uint32_t)b;
            if (p.bag_of != nullptr) p.bag_of[i] = (int32_t)bag;
        }
    }
}

// Runs after the forward or linearize kernel and does nothing unless that
// kernel found the offsets malformed.  Then each lookup position p finds the
// bag that would own it -- the last bag g with offsets[g] <= p, a binary
// search that is exact while the offsets never decrease -- and, unless that
// bag is well formed and holds p, gets the sentinel key (so the sort puts it
// last and no run starts at it), payload 0 and bag -1.  When some bag ends
// before it starts, two well-formed bags can hold one lookup, and every
// lookup gets the sentinel: such a batch has no backward update.
template <typename IdxT, typename KeyT>
__global__ void __launch_bounds__(256) tbe_offsets_fixup_kernel(const __grid_constant__ FwdParams p) {
    if (__ldg(p.counters + C_MALFORMED) == 0) return;
    KeyT *keys = reinterpret_cast<KeyT *>(p.keys);
    const bool decreasing = __ldg(p.counters + C_DECREASING) != 0;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.N; i += stride) {
        bool covered = false;
        if (!decreasing) {
            // largest g in [0, NB] with offsets[g] <= i (none if offsets[0] > i)
            int64_t lo = 0, hi = p.NB + 1;   // answer in [lo - 1, hi)
            while (lo < hi) {
                const int64_t mid = (lo + hi) >> 1;
                if (ld_off<IdxT>(p, mid) <= i) lo = mid + 1; else hi = mid;
            }
            const int64_t g = lo - 1;
            covered = g >= 0 && g < p.NB && ld_off<IdxT>(p, g) >= 0 && ld_off<IdxT>(p, g + 1) <= p.N;
        }
        if (!covered) {
            keys[i] = (KeyT)p.sentinel;
            p.vals[i] = 0u;
            if (p.bag_of != nullptr) p.bag_of[i] = -1;
        }
    }
}

// ---------------------------------------------------------------------------

RowPlan row_plan(int D, int bytes_per_elem) {
    RowPlan r{0, 0, false};
    const int64_t bytes = (int64_t)D * bytes_per_elem;
    if (D <= 0 || bytes % 16) return r;
    const int V = (int)(bytes / 16);
    if (V <= 32 && (V & (V - 1)) == 0) {
        r.lpr = V;
        r.nv = 1;
        r.ok = true;
    } else if (V % 32 == 0 && V / 32 <= 4) {
        r.lpr = 32;
        r.nv = V / 32;
        r.ok = true;
    }
    return r;
}

template <typename K>
static int grid_for(const Launch &L, K kernel, int threads, int64_t work_warps) {
    const int per_sm = cached_blocks_per_sm(L.dev, (const void *)kernel, threads, 0);
    const int64_t want = (work_warps * 32 + threads - 1) / threads;
    int64_t g = (int64_t)L.num_sms * per_sm;
    if (want < g) g = want;
    return (int)(g < 1 ? 1 : g);
}

#ifndef TBE_FWD_ROWS
#define TBE_FWD_ROWS 4   // weight rows of a full step per warp for short bags
#endif
#ifndef TBE_FWD_LONG_BAG
#define TBE_FWD_LONG_BAG 26   // from this mean bag length on, full steps take twice the rows
#endif

// steps of `rows` weight rows: 32/LPR per warp instruction, U of them, with
// at most 32 registers of loaded data per lane
template <int LPR, int NV, int VB> constexpr int fwd_unroll(int rows) {
    return (32 / LPR >= rows ? 1 : rows / (32 / LPR)) * (NV * VB / 4) > 32
               ? (32 / (NV * VB / 4) > 0 ? 32 / (NV * VB / 4) : 1)
               : (32 / LPR >= rows ? 1 : rows / (32 / LPR));
}

// Rows of at most 16 lanes take the grouped kernel: on the large workload
// (bf16 D=128, ~20 lookups per bag) 2.18 ms vs 2.74 ms for a warp per bag;
// demo (f32 D=16) 0.037 vs 0.103 ms.
#ifndef TBE_FWD_GROUPED
#define TBE_FWD_GROUPED 1
#endif
#ifndef TBE_FWD_GROUP_U
#define TBE_FWD_GROUP_U 2   // rows in flight per group in a full step (twice that for long bags)
#endif

template <int NV, int VB> constexpr int group_unroll(int u) {
    return u * NV * VB / 4 > 32 ? (32 / (NV * VB / 4) > 0 ? 32 / (NV * VB / 4) : 1) : u;
}

template <typename WT, int VB, int LPR, int NV, typename IdxT>
static void fwd_group_launch(Launch &L, const FwdParams &p) {
    constexpr int US = group_unroll<NV, VB>(TBE_FWD_GROUP_U);
    constexpr int UL = group_unroll<NV, VB>(2 * TBE_FWD_GROUP_U);
    const bool long_bags = p.N >= (int64_t)TBE_FWD_LONG_BAG * p.NB;
    const bool lay = p.ntl != 0;
    auto k = p.psw != nullptr
                 ? (long_bags ? (lay ? tbe_fwd_group_kernel<WT, VB, LPR, NV, UL, true, IdxT, true>
                                     : tbe_fwd_group_kernel<WT, VB, LPR, NV, UL, true, IdxT, false>)
                              : (lay ? tbe_fwd_group_kernel<WT, VB, LPR, NV, US, true, IdxT, true>
                                     : tbe_fwd_group_kernel<WT, VB, LPR, NV, US, true, IdxT, false>))
                 : (long_bags ? (lay ? tbe_fwd_group_kernel<WT, VB, LPR, NV, UL, false, IdxT, true>
                                     : tbe_fwd_group_kernel<WT, VB, LPR, NV, UL, false, IdxT, false>)
                              : (lay ? tbe_fwd_group_kernel<WT, VB, LPR, NV, US, false, IdxT, true>
                                     : tbe_fwd_group_kernel<WT, VB, LPR, NV, US, false, IdxT, false>));
    const int64_t items = p.ntl ? p.tcum[p.ntl] : p.NB;
    const int grid = grid_for(L, k, 256, (items + 32 / LPR - 1) / (32 / LPR));
    L.before("tbe_fwd_gather");
    k<<<grid, 256, 0, L.stream>>>(p);
    L.after();
}

template <typename WT, int VB, int LPR, int NV, typename IdxT>
static void fwd_launch(Launch &L, const FwdParams &p) {
    if constexpr (LPR <= 16 && TBE_FWD_GROUPED) {
        fwd_group_launch<WT, VB, LPR, NV, IdxT>(L, p);
        return;
    }
    // measured on bf16 D=128 tables: 4-row steps 3.12 ms vs 8-row 3.43 ms for
    // bags of ~20 lookups; 8-row steps 0.57 ms vs 4-row 0.70 ms for ~32
    constexpr int US = fwd_unroll<LPR, NV, VB>(TBE_FWD_ROWS);
    constexpr int UL = fwd_unroll<LPR, NV, VB>(2 * TBE_FWD_ROWS);
    const bool long_bags = p.N >= (int64_t)TBE_FWD_LONG_BAG * p.NB;
    const bool lay = p.ntl != 0;
    auto k = p.psw != nullptr
                 ? (long_bags ? (lay ? tbe_fwd_kernel<WT, VB, LPR, NV, UL, true, IdxT, true>
                                     : tbe_fwd_kernel<WT, VB, LPR, NV, UL, true, IdxT, false>)
                              : (lay ? tbe_fwd_kernel<WT, VB, LPR, NV, US, true, IdxT, true>
                                     : tbe_fwd_kernel<WT, VB, LPR, NV, US, true, IdxT, false>))
                 : (long_bags ? (lay ? tbe_fwd_kernel<WT, VB, LPR, NV, UL, false, IdxT, true>
                                     : tbe_fwd_kernel<WT, VB, LPR, NV, UL, false, IdxT, false>)
                              : (lay ? tbe_fwd_kernel<WT, VB, LPR, NV, US, false, IdxT, true>
                                     : tbe_fwd_kernel<WT, VB, LPR, NV, US, false, IdxT, false>));
    const int grid = grid_for(L, k, 256, p.ntl ? p.tcum[p.ntl] : p.NB);
    L.before("tbe_fwd_gather");
    k<<<grid, 256, 0, L.stream>>>(p);
    L.after();
}

// Rows are read as 16-byte lane vectors: a warp instruction covers 512 bytes
// (fewer, larger requests measured faster than 8-byte vectors on this path).
template <typename WT, typename IdxT>
static bool fwd_dispatch(Launch &L, const FwdParams &p, int row_bytes) {
    const RowPlan rp = row_plan(row_bytes / (int)sizeof(WT), (int)sizeof(WT));
    switch (rp.lpr * 10 + rp.nv) {
    case 11: fwd_launch<WT, 16, 1, 1, IdxT>(L, p); return true;
    case 21: fwd_launch<WT, 16, 2, 1, IdxT>(L, p); return true;
    case 41: fwd_launch<WT, 16, 4, 1, IdxT>(L, p); return true;
    case 81: fwd_launch<WT, 16, 8, 1, IdxT>(L, p); return true;
    case 161: fwd_launch<WT, 16, 16, 1, IdxT>(L, p); return true;
    case 321: fwd_launch<WT, 16, 32, 1, IdxT>(L, p); return true;
    case 322: fwd_launch<WT, 16, 32, 2, IdxT>(L, p); return true;
    case 323: fwd_launch<WT, 16, 32, 3, IdxT>(L, p); return true;
    case 324: fwd_launch<WT, 16, 32, 4, IdxT>(L, p); return true;
    default: return false;
    }
}

template <typename IdxT>
static bool fwd_dtype(Launch &L, const FwdParams &p, int dtype, int D) {
    switch (dtype) {
    case TBE_F32: return fwd_dispatch<float, IdxT>(L, p, D * 4);
    case TBE_F16: return fwd_dispatch<__half, IdxT>(L, p, D * 2);
    case TBE_BF16: return fwd_dispatch<__nv_bfloat16, IdxT>(L, p, D * 2);
    default: return false;
    }
}

static FwdParams make_params(const tbe_tables *tab, const tbe_batch *bt, float *out, void *keys,
                             uint32_t *vals, int32_t *bag_of, uint64_t sentinel, int32_t *status,
                             int32_t *counters) {
    FwdParams p;
    memset(&p, 0, sizeof(p));
    p.W = tab->weights;
    p.table_offset = tab->table_offset;
    p.indices = bt->indices;
    p.offsets = bt->offsets;
    p.psw = bt->per_sample_weights;
    p.weighted = bt->weighted_tables;
    p.out = out;
    p.keys = keys;
    p.vals = vals;
    p.bag_of = bag_of;
    p.status = status;
    p.counters = counters;
    p.B = bt->B;
    // with a bag layout the bags are counted per table (B is ignored)
    p.NB = (int64_t)tab->T * bt->B;
    if (bt->bag_layout_host != nullptr) {
        p.NB = 0;
        for (int t = 0; t < tab->T; ++t) p.NB += bt->bag_layout_host[t].B;
    }
    p.N = bt->N;
    p.T = tab->T;
    p.D = tab->D;
    p.sentinel = sentinel;
    p.payload_pos = bt->per_sample_weights != nullptr ? 1 : 0;
    p.layout = tab->layout;
    p.bag_layout = bt->bag_layout;
    p.ntl = 0;
    return p;
}

tbe_status launch_forward(Launch &L, const tbe_tables *tab, const tbe_batch *bt, float *out,
                          uint32_t *keys, uint32_t *vals, int32_t *bag_of, uint64_t sentinel,
                          int32_t *status, int32_t *counters, const TableClasses &cls) {
    FwdParams p = make_params(tab, bt, out, keys, vals, bag_of, sentinel, status, counters);
    if (p.NB == 0) return TBE_OK;
    const bool i64 = bt->index_type == TBE_INDEX_I64;
    if (bt->bag_layout == nullptr && tab->layout == nullptr) {   // uniform: one launch
        const bool ok = i64 ? fwd_dtype<int64_t>(L, p, tab->dtype, tab->D)
                            : fwd_dtype<int32_t>(L, p, tab->dtype, tab->D);
        return ok ? TBE_OK : TBE_ERR_UNSUPPORTED_DIM;
    }
    // one launch per (D, dtype) class and per FWD_TLIST of its tables
    for (const TableClass &c : cls.classes) {
        for (size_t i0 = 0; i0 < c.tables.size(); i0 += FWD_TLIST) {
            const size_t n = std::min(c.tables.size() - i0, (size_t)FWD_TLIST);
            p.D = c.D;
            p.ntl = (int)n;
            p.tcum[0] = 0;
            for (size_t i = 0; i < n; ++i) {
                const int t = c.tables[i0 + i];
                p.tlist[i] = t;
                p.tcum[i + 1] = p.tcum[i] + cls.B[t];
            }
            if (p.tcum[n] == 0) continue;
            const bool ok = i64 ? fwd_dtype<int64_t>(L, p, c.dtype, c.D) : fwd_dtype<int32_t>(L, p, c.dtype, c.D);
            if (!ok) return TBE_ERR_UNSUPPORTED_DIM;
        }
    }
    return TBE_OK;
}

template <typename IdxT, typename KeyT> static void linearize_launch(Launch &L, const FwdParams &p) {
    auto k = tbe_linearize_kernel<IdxT, KeyT>;
    const int grid = grid_for(L, k, 256, p.ntl ? p.tcum[p.ntl] : p.NB);
    L.before("tbe_linearize");
    k<<<grid, 256, 0, L.stream>>>(p);
    L.after();
}

tbe_status launch_linearize(Launch &L, const tbe_tables *tab, const tbe_batch *bt, void *keys,
                            int key_bytes, uint32_t *vals, int32_t *bag_of, uint64_t sentinel,
                            int32_t *status, int32_t *counters) {
    FwdParams p = make_params(tab, bt, nullptr, keys, vals, bag_of, sentinel, status, counters);
    if (p.NB == 0) return TBE_OK;
    const bool i64 = bt->index_type == TBE_INDEX_I64;
    if (key_bytes == 8) {
        if (i64) linearize_launch<int64_t, uint64_t>(L, p);
        else linearize_launch<int32_t, uint64_t>(L, p);
    } else {
        if (i64) linearize_launch<int64_t, uint32_t>(L, p);
        else linearize_launch<int32_t, uint32_t>(L, p);
    }
    return TBE_OK;
}

template <typename IdxT, typename KeyT> static void fixup_launch(Launch &L, const FwdParams &p) {
    int64_t grid = (p.N + 255) / 256;
    if (grid > (int64_t)L.num_sms * 4) grid = (int64_t)L.num_sms * 4;
    L.before("tbe_offsets_fixup");
    tbe_offsets_fixup_kernel<IdxT, KeyT><<<(unsigned)grid, 256, 0, L.stream>>>(p);
    L.after();
}

tbe_status launch_offsets_fixup(Launch &L, const tbe_tables *tab, const tbe_batch *bt, void *keys,
                                int key_bytes, uint32_t *vals, int32_t *bag_of, uint64_t sentinel,
                                const int32_t *counters) {
    FwdParams p = make_params(tab, bt, nullptr, keys, vals, bag_of, sentinel, nullptr,
                              const_cast<int32_t *>(counters));
    if (p.N == 0) return TBE_OK;
    const bool i64 = bt->index_type == TBE_INDEX_I64;
    if (key_bytes == 8) {
        if (i64) fixup_launch<int64_t, uint64_t>(L, p);
        else fixup_launch<int32_t, uint64_t>(L, p);
    } else {
        if (i64) fixup_launch<int64_t, uint32_t>(L, p);
        else fixup_launch<int32_t, uint32_t>(L, p);
    }
    return TBE_OK;
}

}  // namespace tbe
