// Backward kernels instantiated for __nv_bfloat16 weights (see backward_kernels.cuh).
#include "backward_kernels.cuh"

namespace tbe {

bool bwd_dispatch_bf16(Launch &L, const BwdParams &p, RowPlan rp, int long_mode) {
    return bwd_dispatch<__nv_bfloat16>(L, p, rp, long_mode);
}

}  // namespace tbe
