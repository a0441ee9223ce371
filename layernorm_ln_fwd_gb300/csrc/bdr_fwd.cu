// bdr_fwd.cu -- the LayerNorm forward with the bias + dropout + residual prologue: the
// prologue instantiations of the kernels in ln_fwd_kernels.cuh.
#include "ln_fwd_kernels.cuh"

namespace lnk {

cudaError_t launch_bdr_fwd(Dtype dt, const FwdArgs& a, bool aligned, int path_override,
                           cudaStream_t stream, int* launches) {
    return launch_norm_fwd<false, true>(dt, a, aligned, path_override, stream, launches);
}

}  // namespace lnk
