// Backward entry: fills the kernels' parameters and runs one set of launches
// per (D, dtype) class (kernels in backward_kernels.cuh, instantiated per
// weight dtype in backward_f32.cu / backward_f16.cu / backward_bf16.cu).
#include "backward_kernels.cuh"

namespace tbe {

bool bwd_dispatch_f32(Launch &L, const BwdParams &p, RowPlan rp, int long_mode);
bool bwd_dispatch_f16(Launch &L, const BwdParams &p, RowPlan rp, int long_mode);
bool bwd_dispatch_bf16(Launch &L, const BwdParams &p, RowPlan rp, int long_mode);

size_t bwd_partials_bytes(int64_t max_chunks, int D, int dtype) {
    const size_t acc = dtype == TBE_F32 ? 8 : 4;
    return (size_t)max_chunks * (size_t)D * acc;
}

tbe_status launch_backward(Launch &L, const BwdArgs &a) {
    const tbe_meta *m = a.meta;
    BwdParams p;
    p.W = a.tab->weights;
    p.mom = a.momentum;
    p.G = a.grad_out;
    p.table_offset = a.tab->table_offset;
    p.vals = m->sorted_vals;
    p.bag_of = m->bag_of;
    p.psw = a.bt->per_sample_weights;
    p.weighted = a.bt->weighted_tables;
    p.unique_keys = m->unique_keys;
    p.key64 = m->key_bytes == 8;
    p.seg_off = m->seg_off;
    p.counters = m->counters;
    p.long_run = m->long_run;
    p.long_chunk_base = m->long_chunk_base;
    // the order the RLE built (none for batches with a bag layout)
    p.chunk_order = a.bt->bag_layout == nullptr && chunk_order_on(a.bt->B, a.tab->T) ? m->chunk_order
                                                                                      : nullptr;
    p.chunk_desc = m->chunk_desc;
    p.partials = a.partials;
    p.arrive = a.arrive;
    p.status = a.status;
    p.B = a.bt->B;
    p.T = a.tab->T;
    p.D = a.tab->D;
    p.lr = a.lr;
    p.eps = a.eps;
    p.sl_threshold = a.sl_threshold;
    p.chunk = a.chunk;
    p.payload_pos = m->payload_is_pos;
    p.layout = a.tab->layout;
    p.bag_layout = a.bt->bag_layout;
    p.part_stride = a.part_stride;
    if (a.bt->N == 0) return TBE_OK;
    // one set of launches per (D, dtype) class; with layouts each kernel
    // skips the runs and chunks of other classes' tables
    for (const TableClass &c : a.classes->classes) {
        p.D = c.D;
        p.cls_dtype = c.dtype;
        const RowPlan rp = row_plan(c.D, 4);
        bool ok = false;
        switch (c.dtype) {
        case TBE_F32: ok = bwd_dispatch_f32(L, p, rp, a.long_mode); break;
        case TBE_F16: ok = bwd_dispatch_f16(L, p, rp, a.long_mode); break;
        case TBE_BF16: ok = bwd_dispatch_bf16(L, p, rp, a.long_mode); break;
        default: return TBE_ERR_UNSUPPORTED_DTYPE;
        }
        if (!ok) return TBE_ERR_UNSUPPORTED_DIM;
    }
    return TBE_OK;
}

// ---------------------------------------------------------------------------
// Self-test of the bulk-copy wait's time limit: one warp waits on an
// mbarrier phase that nothing will complete (no copy is issued), gives up
// after WAIT_LIMIT_NS and sets TBE_FLAG_COPY_TIMEOUT, as the gradient-row
// rings do when a copy does not land.

__global__ void __launch_bounds__(32) mbar_selftest_kernel(int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) bar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();
    if (!mbar_wait_bounded(b, 0) && threadIdx.x == 0) atomicOr(status + 1, TBE_FLAG_COPY_TIMEOUT);
}

tbe_status launch_copy_wait_selftest(Launch &L, int32_t *status) {
    L.before("tbe_selftest_copy_wait");
    mbar_selftest_kernel<<<1, 32, 0, L.stream>>>(status);
    L.after();
    return TBE_OK;
}

}  // namespace tbe

