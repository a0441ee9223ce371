// ln_noalloc.cu -- a bf16 backward for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at the time they run the backward: a serving process
// that reserved its whole device-memory budget at start-up, or a plugin whose host framework
// owns every device allocation through its own allocator, would fail or fragment memory by
// allocating mid-run.  ln_bwd_bf16_noalloc runs the same backward kernels as ln_bwd_bf16 but
// keeps their scratch (the per-block partial sums) in a fixed array that is part of the
// library's device image, so the call allocates nothing.  The array starts zeroed (static
// device storage) and every completed backward leaves the words it used at zero again, as
// the kernels' finish requires; ln_device_check re-zeroes it after a backward gave up.
#include <map>
#include <mutex>

#include "ln.h"
#include "ln_device.cuh"
#include "ln_internal.h"

namespace {

// The scratch array.  Every GPU that loads the library holds it until the process exits.
// In host code its name is only a host-side stand-in: the device address comes from
// cudaGetSymbolAddress below, per device.
static __device__ __align__(256) unsigned char ln_noalloc_scratch[LN_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
std::map<int, void*> g_scratch_addr;  // device ordinal -> device address of the array

// Looks up (once per device, with that device current) the device address of the array.
cudaError_t scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_scratch_addr.find(dev);
    if (it == g_scratch_addr.end()) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, ln_noalloc_scratch);
        if (e != cudaSuccess) return e;
        it = g_scratch_addr.emplace(dev, p).first;
    }
    *out = it->second;
    return cudaSuccess;
}

}  // namespace

namespace lnk {
cudaError_t noalloc_scratch_clear(cudaStream_t stream) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    void* p = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_scratch_addr.find(dev);
        if (it == g_scratch_addr.end()) return cudaSuccess;  // never used on this device
        p = it->second;
    }
    e = cudaMemsetAsync(p, 0, LN_NOALLOC_SCRATCH_BYTES, stream);
    return e == cudaSuccess ? cudaStreamSynchronize(stream) : e;
}
}  // namespace lnk

extern "C" ln_status ln_bwd_bf16_noalloc(const ln_bf16* dy, const ln_bf16* x_or_res_out,
                                         const ln_bf16* gamma, const float* mean,
                                         const float* rstd, ln_bf16* dx, ln_bf16* dgamma,
                                         ln_bf16* dbeta, int64_t rows, int64_t cols,
                                         ln_stream_t stream) {
    using B = __nv_bfloat16;
    // Sizes are checked before the address lookup, so invalid calls touch no CUDA state.
    if (rows < 0 || cols <= 0) return LN_EINVAL;
    if (cols > LN_MAX_COLS || rows > LN_MAX_ROWS) return LN_EUNSUPPORTED;
    void* ws = nullptr;
    const cudaError_t e = scratch_address(&ws);
    if (e != cudaSuccess) {
        lnk::record_cuda_error(e);
        return LN_ECUDA;
    }
    // The regular backward with the fixed array as a caller-owned workspace: the same plan,
    // kernels, checks and test hooks as ln_bwd_bf16.
    const ln_status st = lnk::bwd_impl<B>(
        lnk::Dtype::BF16, false, reinterpret_cast<const B*>(dy), reinterpret_cast<const B*>(x_or_res_out),
        reinterpret_cast<const B*>(gamma), mean, rstd, reinterpret_cast<B*>(dx),
        reinterpret_cast<B*>(dgamma), reinterpret_cast<B*>(dbeta), rows, cols, ws,
        LN_NOALLOC_SCRATCH_BYTES, false, stream);
    // A problem whose partial sums do not fit the array is an unsupported size here.
    return st == LN_ENOSPACE ? LN_EUNSUPPORTED : st;
}
