// Backward kernels instantiated for __half weights (see backward_kernels.cuh).
#include "backward_kernels.cuh"

namespace tbe {

bool bwd_dispatch_f16(Launch &L, const BwdParams &p, RowPlan rp, int long_mode) {
    return bwd_dispatch<__half>(L, p, rp, long_mode);
}

}  // namespace tbe
