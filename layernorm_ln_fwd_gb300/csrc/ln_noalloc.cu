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

ln_status fail(cudaError_t e) {
    lnk::record_cuda_error(e);
    return LN_ECUDA;
}

}  // namespace

namespace lnk {
cudaError_t noalloc_scratch_clear() {
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
    return cudaMemset(p, 0, LN_NOALLOC_SCRATCH_BYTES);
}
}  // namespace lnk

extern "C" ln_status ln_bwd_bf16_noalloc(const ln_bf16* dy, const ln_bf16* x_or_res_out,
                                         const ln_bf16* gamma, const float* mean,
                                         const float* rstd, ln_bf16* dx, ln_bf16* dgamma,
                                         ln_bf16* dbeta, int64_t rows, int64_t cols,
                                         ln_stream_t stream_) {
    using lnk::Dtype;
    if (rows < 0 || cols <= 0) return LN_EINVAL;
    if (cols > LN_MAX_COLS || rows > LN_MAX_ROWS) return LN_EUNSUPPORTED;
    if (!dgamma || !dbeta) return LN_EINVAL;
    if (rows > 0 && (!dy || !x_or_res_out || !gamma || !mean || !rstd || !dx)) return LN_EINVAL;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(e);
    const lnk::DeviceInfo& di = lnk::device_info(dev);
    if (di.cc_major != 10 || di.cc_minor != 3) return LN_EUNSUPPORTED;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (rows == 0) {  // sums over no rows
        e = cudaMemsetAsync(dgamma, 0, (size_t)cols * sizeof(ln_bf16), stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(dbeta, 0, (size_t)cols * sizeof(ln_bf16), stream);
        return e == cudaSuccess ? LN_OK : fail(e);
    }
    const void* ptrs[] = {dy, x_or_res_out, gamma, dx};
    const bool aligned = lnk::vector_ok(Dtype::BF16, (int)cols, ptrs, 4);
    lnk::BwdPlan plan;
    e = lnk::plan_bwd(Dtype::BF16, (int)rows, (int)cols, aligned, lnk::kPathAuto, &plan);
    if (e != cudaSuccess) return fail(e);
    if (lnk::bwd_workspace_bytes(plan.grid, (int)cols, lnk::bwd_plan_acc_region(plan)) >
        (size_t)LN_NOALLOC_SCRATCH_BYTES)
        return LN_EUNSUPPORTED;  // the problem's partial sums do not fit the fixed scratch
    void* ws = nullptr;
    e = scratch_address(&ws);
    if (e != cudaSuccess) return fail(e);
    lnk::BwdArgs a;
    a.dy = dy;
    a.xr = x_or_res_out;
    a.gamma = gamma;
    a.mean = mean;
    a.rstd = rstd;
    a.dx = dx;
    a.dgamma = dgamma;
    a.dbeta = dbeta;
    a.rows = (int)rows;
    a.cols = (int)cols;
    a.counters = static_cast<unsigned*>(ws);
    a.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + lnk::kWorkspaceHeader);
    a.status = lnk::status_word();
    a.wait_limit_ns = lnk::kWaitLimitNs;
    a.wait_extra = 0;
    int launches = 0;
    e = lnk::launch_bwd(Dtype::BF16, a, plan, stream, &launches);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? LN_OK : fail(e);
}
