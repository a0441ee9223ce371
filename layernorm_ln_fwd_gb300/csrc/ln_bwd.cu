// ln_bwd.cu -- the fused residual-add + LayerNorm backward: instantiations of the kernels in
// ln_bwd_kernels.cuh and the library-facing plan / launch entry points (which hand RMSNorm
// problems to rms_bwd.cu).
#include "ln_bwd_kernels.cuh"

namespace lnk {

int bwd_max_grid(int rows, int sms) { return std::max(1, std::min(rows, sms * 8)); }

cudaError_t plan_bwd(Dtype dt, bool rms, int rows, int cols, bool aligned, int path_override,
                     BwdPlan* plan) {
    if (rms) return plan_rms_bwd(dt, rows, cols, aligned, path_override, plan);
    return plan_bwd_t<false>(dt, rows, cols, aligned, path_override, plan);
}

cudaError_t launch_bwd(Dtype dt, const BwdArgs& a, const BwdPlan& plan, cudaStream_t stream,
                       int* launches) {
    if (plan.rms) return launch_rms_bwd(dt, a, plan, stream, launches);
    return launch_bwd_t<false>(dt, a, plan, stream, launches);
}

}  // namespace lnk
