// rms_bwd.cu -- the fused residual-add + RMSNorm backward: the RMS instantiations of the
// kernels in ln_bwd_kernels.cuh.
#include "ln_bwd_kernels.cuh"

namespace lnk {

cudaError_t plan_rms_bwd(Dtype dt, int rows, int cols, bool aligned, int path_override,
                         BwdPlan* plan) {
    return plan_bwd_t<true>(dt, rows, cols, aligned, path_override, plan);
}

cudaError_t launch_rms_bwd(Dtype dt, const BwdArgs& a, const BwdPlan& plan, cudaStream_t stream,
                           int* launches) {
    return launch_bwd_t<true>(dt, a, plan, stream, launches);
}

}  // namespace lnk
