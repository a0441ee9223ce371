// bdr_fwd.cu -- the LayerNorm forward with the bias + dropout + residual prologue: the
// prologue instantiations of the kernels in ln_fwd_kernels.cuh (PRO = 1: the keep decisions
// from the generator; PRO = 2: the same, also stored as bits for the backward).
#include "ln_fwd_kernels.cuh"

namespace lnk {

cudaError_t launch_bdr_fwd(Dtype dt, const FwdArgs& a, bool aligned, int path_override,
                           cudaStream_t stream, int* launches) {
    if (a.pro.keep_out) return launch_norm_fwd<false, 2>(dt, a, aligned, path_override, stream, launches);
    return launch_norm_fwd<false, 1>(dt, a, aligned, path_override, stream, launches);
}

}  // namespace lnk
