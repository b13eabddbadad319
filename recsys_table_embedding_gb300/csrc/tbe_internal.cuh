// Internal declarations shared by the CUDA translation units of the library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "tbe.h"

namespace tbe {

constexpr unsigned FULL = 0xffffffffu;

// Indices into meta->counters (device int32).  C_MALFORMED is set when the
// batch's offsets are malformed in any way (a bag not 0 <= start <= end <= N,
// or offsets[0] != 0, or offsets[T*B] != N); C_DECREASING when some bag has
// end < start.  Both are zeroed before the forward or linearize kernel runs.
enum Counter {
    C_NUM_UNIQUE = 0,
    C_N_VALID = 1,
    C_NUM_LONG = 2,
    C_NUM_CHUNKS = 3,
    C_MALFORMED = 4,
    C_DECREASING = 5,
    C_COUNT = 8
};

// Weight element traits: the 16-byte vector of a row, and the accumulator
// precision (FBTriton TBE redesign, decision checklist item 1: FP32 for
// FP16/BF16 weights, FP64 for FP32 weights).
template <typename WT> struct WTraits;
template <> struct WTraits<float> {
    using acc = double;
    static constexpr int VEC = 4;   // elements per 16-byte vector
};
template <> struct WTraits<__half> {
    using acc = float;
    static constexpr int VEC = 8;
};
template <> struct WTraits<__nv_bfloat16> {
    using acc = float;
    static constexpr int VEC = 8;
};

// Two bf16 values packed in a 32-bit word (element 0 in the low half) as
// floats.  A bf16 value is the high half of the float with the same value,
// so widening is a shift or a mask of the bits (exact for every value).
#ifndef TBE_BF16_WIDEN_BITS
#define TBE_BF16_WIDEN_BITS 1
#endif
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
#if TBE_BF16_WIDEN_BITS
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
#else
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
#endif
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename WT> __device__ __forceinline__ WT from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __half from_f32<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ uint4 ldg_v4(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// Relaxed GPU-scope accesses for flag/status words that carry their own data.
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Every device-side wait in this library gives up after this long (wall
// clock, from the %globaltimer nanosecond counter), sets a status flag and
// stops issuing work.  Waits normally end within microseconds.
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

#ifndef TBE_MBAR_SUSPEND_NS
#define TBE_MBAR_SUSPEND_NS 20000
#endif
// Bounded wait for the completion of the mbarrier phase with the given parity
// (shared-memory address `bar`).  Each try_wait may suspend the thread for up
// to TBE_MBAR_SUSPEND_NS until the phase completes, so a waiting warp does
// not spin through issue slots the other warps need.  False if WAIT_LIMIT_NS
// passed first.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "n"(TBE_MBAR_SUSPEND_NS)
            : "memory");
        if (ok) return true;
        const uint64_t now = global_ns();
        if (i == 0) t0 = now;
        else if (now - t0 > WAIT_LIMIT_NS) return false;
    }
}

// Table of a linearised key: largest t with table_offset[t] <= key (T small).
__device__ __forceinline__ int table_of_key(const int64_t *table_offset, int T, int64_t key) {
    int lo = 0, hi = T;   // answer in [lo, hi)
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (__ldg(table_offset + mid) <= key) lo = mid; else hi = mid;
    }
    return lo;
}

// ---- addressing of tables, bags and output rows ---------------------------
// Uniform problems (no layouts): table t's rows are rows table_offset[t].. of
// one [rows_total, D] array, bag (t,b) is CSR bag t*B+b and its output row
// starts at (b*T + t)*D.  With layouts (tables of different D/dtype, or a
// different B per table) these come from the caller's per-table records.

// byte offset in the weights of element 0 of linearised row `row` of table t
// (D and esize: the row length and element size of t)
__device__ __forceinline__ int64_t weight_byte(const tbe_table_layout *layout,
                                               const int64_t *table_offset, int t, int64_t row,
                                               int D, int esize) {
    if (layout == nullptr) return row * D * esize;
    return __ldg(&layout[t].weights_byte_offset) + (row - __ldg(table_offset + t)) * D * esize;
}

// float index in out / grad_out of bag b of table t
__device__ __forceinline__ int64_t out_row(const tbe_bag_layout *bags, int T, int D, int t,
                                           int64_t b) {
    if (bags == nullptr) return (b * T + t) * (int64_t)D;
    return __ldg(&bags[t].out_offset) + b * __ldg(&bags[t].out_stride);
}

// first CSR bag of table t
__device__ __forceinline__ int64_t bag_base(const tbe_bag_layout *bags, int64_t B, int t) {
    return bags == nullptr ? (int64_t)t * B : __ldg(&bags[t].bag_offset);
}

// table of CSR bag g
__device__ __forceinline__ int table_of_bag(const tbe_bag_layout *bags, int64_t B, int T, int64_t g) {
    if (bags == nullptr) return (int)(g / B);
    int lo = 0, hi = T;   // largest t with bag_offset[t] <= g
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (__ldg(&bags[mid].bag_offset) <= g) lo = mid; else hi = mid;
    }
    return lo;
}

// whether table t has the row length and dtype of this launch's class
__device__ __forceinline__ bool in_class(const tbe_table_layout *layout, int t, int D, int dtype) {
    return layout == nullptr || (__ldg(&layout[t].D) == D && __ldg(&layout[t].dtype) == dtype);
}

// ---------------------------------------------------------------------------
// Host-side launch context: the caller's stream, config and optional
// per-kernel timing events.
struct Launch {
    cudaStream_t stream;
    const tbe_config *cfg;
    int used = 0;
    int dev = 0;         // current device when the entry point was called
    int num_sms = 0;
    bool capturing = false;   // `stream` is being captured into a CUDA graph
    bool failed = false;
    Launch(cudaStream_t s, const tbe_config *c);
    void before(const char *name);
    void after();
};

// Launch properties are looked up once per (device, kernel) and cached, so a
// call enqueues its kernels without per-launch driver queries:
// resident blocks per SM for `threads` threads and `smem` dynamic bytes ...
int cached_blocks_per_sm(int dev, const void *fn, int threads, size_t smem);
// ... and the dynamic shared-memory limit (with the max-shared carveout),
// raised to `smem` bytes the first time a kernel needs it on a device.
void cached_smem_attr(int dev, const void *fn, size_t smem);

// Row-vector plan for a D-element row of `bytes_per_elem`: lanes per row
// (LPR) and 16-byte vectors per lane (NV), with LPR * NV * 16 = row bytes.
struct RowPlan {
    int lpr, nv;
    bool ok;
};
RowPlan row_plan(int D, int bytes_per_elem);

// Host-side grouping of tables with layouts into launch classes of one row
// length and dtype (uniform problems: one class of all tables).
struct TableClass {
    int D, dtype;
    std::vector<int> tables;
};
struct TableClasses {
    std::vector<TableClass> classes;
    std::vector<int64_t> B;   // bags of each table
};

// --- forward.cu
// `counters` (nullable) receives C_MALFORMED / C_DECREASING.  `keys`
// (nullable) are 32-bit: 64-bit keys come from launch_linearize.  Tables
// with layouts are gathered one class per launch.
tbe_status launch_forward(Launch &L, const tbe_tables *tab, const tbe_batch *bt, float *out,
                          uint32_t *keys, uint32_t *vals, int32_t *bag_of, uint64_t sentinel,
                          int32_t *status, int32_t *counters, const TableClasses &cls);
tbe_status launch_linearize(Launch &L, const tbe_tables *tab, const tbe_batch *bt, void *keys,
                            int key_bytes, uint32_t *vals, int32_t *bag_of, uint64_t sentinel,
                            int32_t *status, int32_t *counters);
// After the forward or linearize kernel: when counters[C_MALFORMED] is set,
// every lookup outside a well-formed bag gets the sentinel key (all lookups
// when counters[C_DECREASING] is set), so that only lookups of well-formed
// bags reach the backward.  Does nothing on well-formed batches.
tbe_status launch_offsets_fixup(Launch &L, const tbe_tables *tab, const tbe_batch *bt, void *keys,
                                int key_bytes, uint32_t *vals, int32_t *bag_of, uint64_t sentinel,
                                const int32_t *counters);
// zero meta->counters (all C_COUNT words)
void launch_zero_counters(Launch &L, int32_t *counters);

// --- sort.cu: stable LSD radix sort of (key, val) pairs over the low
// `key_bits` bits (keys of key_bytes = 4 or 8); result lands in (keys_a,
// vals_a) when the number of passes is even, else in (keys_b, vals_b);
// returns which via *in_b.
size_t sort_workspace_bytes(int64_t N, int key_bits);
tbe_status launch_sort(Launch &L, void *keys_a, uint32_t *vals_a, void *keys_b, uint32_t *vals_b,
                       int64_t N, int key_bits, int key_bytes, void *ws, int32_t *status,
                       bool *in_b);

// Self-test of the look-back's time limit (scratch of sort_selftest_bytes()).
size_t sort_selftest_bytes();
tbe_status launch_sort_selftest(Launch &L, void *ws, int32_t *status);

// --- rle.cu: run-length encode sorted keys, route long runs into chunks.
size_t rle_workspace_bytes(int64_t N);
// Long-run chunk slots are taken in order of (table, batch window of 2^wshift
// bags of their first lookup) when the batch has at least CHUNK_ORDER_MIN_B
// bags per table and at most CHUNK_WINDOWS_MAX tables, so that concurrently
// reduced chunks share gradient rows.
#ifndef TBE_CHUNK_ORDER_MIN_B
#define TBE_CHUNK_ORDER_MIN_B 4096
#endif
constexpr int64_t CHUNK_ORDER_MIN_B = TBE_CHUNK_ORDER_MIN_B;
constexpr int CHUNK_WINDOWS_MAX = 4096;
bool chunk_order_on(int64_t B, int T);
int chunk_window_shift(int64_t B, int T);

struct RleArgs {
    const void *sorted_keys;
    const uint32_t *sorted_vals;
    const int32_t *bag_of;
    int64_t N, B;
    uint64_t sentinel;
    int key_bytes;
    int payload_pos;
    void *unique_keys;
    int32_t *seg_off;
    int32_t *counters;
    int32_t *long_run;
    int32_t *long_chunk_base;
    int32_t *chunk_order;
    int32_t *chunk_desc;
    int32_t *arrive;
    const int64_t *table_offset;
    int T;
    int sl_threshold;
    int chunk;
    bool order_ok;   // chunk ordering by bag window applies (every table has B bags)
};
tbe_status launch_rle(Launch &L, const RleArgs &a, void *ws);

// --- backward.cu
struct BwdArgs {
    const tbe_tables *tab;
    const tbe_batch *bt;
    const tbe_meta *meta;
    float *momentum;
    const float *grad_out;
    float lr, eps;
    void *partials;          // [max_chunks, D] accumulator type
    int32_t *arrive;         // [max_long]
    int32_t *status;         // caller's device status words
    int64_t max_chunks, max_long;
    int sl_threshold, chunk, long_mode;
    const TableClasses *classes;   // the launch classes (one for uniform problems)
    int64_t part_stride;           // bytes between chunk slots' partials
};
size_t bwd_partials_bytes(int64_t max_chunks, int D, int dtype);
tbe_status launch_backward(Launch &L, const BwdArgs &a);
// Self-test of the bulk-copy wait's time limit.
tbe_status launch_copy_wait_selftest(Launch &L, int32_t *status);

// --- hist.cu: small-table histogram path on the tensor cores
bool hist_shape_ok(const tbe_tables *tab, const tbe_batch *bt, int64_t max_rows);
size_t hist_workspace_bytes(const tbe_tables *tab, const tbe_batch *bt);
// `counters` (nullable; the meta's) receives C_MALFORMED / C_DECREASING in
// the forward and count kernels; the backward applies no update when
// counters[C_DECREASING] is set.
tbe_status launch_hist_forward(Launch &L, const tbe_tables *tab, const tbe_batch *bt, float *out,
                               uint16_t *hist, int32_t *status, int32_t *counters);
tbe_status launch_hist_count(Launch &L, const tbe_tables *tab, const tbe_batch *bt,
                             uint16_t *hist, int32_t *status, int32_t *counters);
tbe_status launch_hist_backward(Launch &L, const tbe_tables *tab, const tbe_batch *bt,
                                const uint16_t *hist, float *momentum, const float *grad_out,
                                float lr, float eps, void *ws, int32_t *status,
                                const int32_t *counters);

}  // namespace tbe
