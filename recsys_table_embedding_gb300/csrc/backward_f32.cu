// Backward kernels instantiated for float weights (see backward_kernels.cuh).
#include "backward_kernels.cuh"

namespace tbe {

bool bwd_dispatch_f32(Launch &L, const BwdParams &p, RowPlan rp, int long_mode) {
    return bwd_dispatch<float>(L, p, rp, long_mode);
}

}  // namespace tbe
