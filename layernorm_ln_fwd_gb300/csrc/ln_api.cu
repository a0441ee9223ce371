// ln_api.cu -- the C ABI declared in include/ln.h: argument checks, kernel selection,
// backward workspaces and the per-device status word.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "ln.h"
#include "ln_device.cuh"
#include "ln_internal.h"

// One status word per device.  Kernels OR kStatusTimeout into it when a bounded wait runs
// out; ln_device_check reads and clears it.
__device__ unsigned ln_status_word_dev;

namespace lnk {
namespace {

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
std::map<int, unsigned*> g_status_ptrs;
std::map<std::tuple<int, const void*, int, size_t>, int> g_occupancy;

struct Workspace {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;

std::atomic<int> g_force_path{kPathAuto};
std::atomic<unsigned> g_wait_test_us{0};

thread_local int t_last_cuda_error = 0;
thread_local int t_last_launches = 0;

bool check_mode() {
    static const bool on = [] {
        const char* v = std::getenv("LN_CHECK");
        return v && v[0] && v[0] != '0';
    }();
    return on;
}

int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev;
}

}  // namespace

const DeviceInfo& device_info(int dev) {
    if (dev < 0) dev = current_device();
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_devices.find(dev);
    if (it != g_devices.end()) return it->second;
    DeviceInfo d;
    d.device = dev;
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev);
    cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    return g_devices.emplace(dev, d).first->second;
}

unsigned* status_word() {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_status_ptrs.find(dev);
    if (it != g_status_ptrs.end()) return it->second;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, ln_status_word_dev) != cudaSuccess) return nullptr;
    g_status_ptrs[dev] = static_cast<unsigned*>(p);
    return static_cast<unsigned*>(p);
}

int blocks_per_sm(const void* kernel, int threads, size_t smem) {
    const int dev = current_device();
    auto key = std::make_tuple(dev, kernel, threads, smem);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_occupancy.find(key);
        if (it != g_occupancy.end()) return it->second;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess)
        n = 0;
    std::lock_guard<std::mutex> lk(g_mu);
    g_occupancy[key] = n;
    return n;
}

cudaError_t launch_kernel(const void* kern, dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, void** args, bool cooperative) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cooperative) {  // every block co-resident: the driver checks it against occupancy
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelExC(&cfg, kern, args);
}

void record_cuda_error(cudaError_t e) { t_last_cuda_error = (int)e; }

bool vector_ok(Dtype dt, int cols, const void* const* ptrs, int nptrs) {
    const int esize = dt == Dtype::F32 ? 4 : 2;
    if (((size_t)cols * esize) % 16 != 0) return false;
    for (int i = 0; i < nptrs; ++i)
        if (ptrs[i] && (reinterpret_cast<uintptr_t>(ptrs[i]) & 15u) != 0) return false;
    return true;
}

namespace {

// Validation shared by all entry points; touches no CUDA state.
ln_status check_sizes(int64_t rows, int64_t cols) {
    if (rows < 0 || cols <= 0) return LN_EINVAL;
    if (cols > LN_MAX_COLS || rows > LN_MAX_ROWS) return LN_EUNSUPPORTED;
    return LN_OK;
}

ln_status cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return LN_ECUDA;
}

ln_status check_device() {
    const int dev = current_device();
    if (dev < 0) return cuda_fail(cudaGetLastError());
    const DeviceInfo& di = device_info(dev);
    if (di.cc_major != 10 || di.cc_minor != 3) return LN_EUNSUPPORTED;
    return LN_OK;
}

uint64_t wait_limit_ns() {
    const unsigned us = g_wait_test_us.load();
    return us ? (uint64_t)us * 1000ull : kWaitLimitNs;
}

ln_status finish_call(cudaError_t e, int launches, cudaStream_t stream) {
    t_last_launches = launches;
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e);
    if (check_mode()) {
        // Check mode synchronises, which a stream being captured into a graph cannot do.
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone)
            return ln_device_check(reinterpret_cast<ln_stream_t>(stream));
    }
    return LN_OK;
}

// `rms`: the RMSNorm forward (beta and mean unused, may be null; rstd receives 1 / rms).
// The dropout threshold floor(p 2^32) (p in [0, 1)).
uint32_t drop_threshold(float p) {
    const double t = std::floor((double)p * 4294967296.0);
    return t >= 4294967295.0 ? 4294967295u : (uint32_t)t;
}

// The workspace of a backward: the library's own one for `stream` (allocated, or grown, and
// zeroed on first use) when `own_ws`, else the caller's `ws` if it holds `need` bytes.
ln_status acquire_workspace(bool own_ws, void*& ws, size_t ws_bytes, size_t need,
                            cudaStream_t stream) {
    if (!own_ws) return ws_bytes < need ? LN_ENOSPACE : LN_OK;
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_mu);
    Workspace& w = g_workspaces[std::make_pair(dev, stream)];
    if (w.bytes < need) {
        cudaError_t e = cudaSuccess;
        if (w.ptr) {
            e = cudaStreamSynchronize(stream);  // the old workspace may still be in use
            if (e == cudaSuccess) e = cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
            if (e != cudaSuccess) return cuda_fail(e);
        }
        e = cudaMalloc(&w.ptr, need);
        if (e != cudaSuccess) {
            w.ptr = nullptr;
            return cuda_fail(e);
        }
        w.bytes = need;
        e = cudaMemsetAsync(w.ptr, 0, need, stream);  // zero between calls, from the start
        if (e != cudaSuccess) return cuda_fail(e);
    }
    ws = w.ptr;
    return LN_OK;
}

template <typename T>
ln_status fwd_impl(Dtype dt, bool rms, const T* x, const T* res, const T* gamma, const T* beta,
                   float eps, int64_t rows, int64_t cols, T* out, T* res_out, float* mean,
                   float* rstd, ln_stream_t stream_, const T* bias = nullptr, float p = 0.f,
                   uint64_t seed = 0, uint64_t offset = 0, uint8_t* keep_out = nullptr) {
    t_last_launches = 0;
    if (!std::isfinite(eps) || eps < 0.f) return LN_EINVAL;
    ln_status st = check_sizes(rows, cols);
    if (st != LN_OK) return st;
    if (rows == 0) return LN_OK;  // nothing is read or written
    if (!x || !gamma || (!rms && (!beta || !mean)) || !out || !rstd) return LN_EINVAL;
    st = check_device();
    if (st != LN_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const void* ptrs[] = {x, res, gamma, beta, out, res_out, bias};
    const bool aligned = vector_ok(dt, (int)cols, ptrs, 7);
    FwdArgs a;
    if (bias) {
        a.pro.bias = bias;
        a.pro.scale = 1.0f / (1.0f - p);
        a.pro.rng = DropoutRng::make(seed, offset, drop_threshold(p));
        a.pro.keep_out = keep_out;
        a.pro.keep_stride = (int)((cols + 7) / 8);
    }
    a.x = x;
    a.res = res;
    a.gamma = gamma;
    a.beta = beta;
    a.eps = eps;
    a.rows = (int)rows;
    a.cols = (int)cols;
    a.out = out;
    a.res_out = res_out;
    a.mean = mean;
    a.rstd = rstd;
    a.status = status_word();
    a.wait_limit_ns = wait_limit_ns();
    int launches = 0;
    cudaError_t e = rms    ? launch_rms_fwd(dt, a, aligned, g_force_path.load(), stream, &launches)
                    : bias ? launch_bdr_fwd(dt, a, aligned, g_force_path.load(), stream, &launches)
                           : launch_fwd(dt, a, aligned, g_force_path.load(), stream, &launches);
    return finish_call(e, launches, stream);
}

}  // namespace

template <typename T>
ln_status bwd_impl(Dtype dt, bool rms, const T* dy, const T* xr, const T* gamma,
                   const float* mean, const float* rstd, T* dx, T* dgamma, T* dbeta,
                   int64_t rows, int64_t cols, void* ws, size_t ws_bytes, bool own_ws,
                   ln_stream_t stream_) {
    t_last_launches = 0;
    ln_status st = check_sizes(rows, cols);
    if (st != LN_OK) return st;
    if (!dgamma || (!rms && !dbeta)) return LN_EINVAL;
    if (rows > 0 && (!dy || !xr || !gamma || (!rms && !mean) || !rstd || !dx)) return LN_EINVAL;
    if (!own_ws && !ws) return LN_EINVAL;
    if (!own_ws && (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return LN_EALIGN;
    st = check_device();
    if (st != LN_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const size_t esize = sizeof(T);
    if (rows == 0) {  // sums over no rows
        cudaError_t e = cudaMemsetAsync(dgamma, 0, (size_t)cols * esize, stream);
        if (e == cudaSuccess && !rms) e = cudaMemsetAsync(dbeta, 0, (size_t)cols * esize, stream);
        return finish_call(e, 0, stream);
    }
    const void* ptrs[] = {dy, xr, gamma, dx};
    const bool aligned = vector_ok(dt, (int)cols, ptrs, 4);
    BwdPlan plan;
    cudaError_t e = plan_bwd(dt, rms, (int)rows, (int)cols, aligned, g_force_path.load(), &plan);
    if (e != cudaSuccess) return cuda_fail(e);
    const size_t need = bwd_workspace_bytes(plan.grid, (int)cols, bwd_plan_acc_region(plan));
    st = acquire_workspace(own_ws, ws, ws_bytes, need, stream);
    if (st != LN_OK) return st;
    BwdArgs a;
    a.dy = dy;
    a.xr = xr;
    a.gamma = gamma;
    a.mean = mean;
    a.rstd = rstd;
    a.dx = dx;
    a.dgamma = dgamma;
    a.dbeta = dbeta;
    a.rows = (int)rows;
    a.cols = (int)cols;
    a.counters = static_cast<unsigned*>(ws);
    a.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + kWorkspaceHeader);
    a.status = status_word();
    a.wait_limit_ns = wait_limit_ns();
    a.wait_extra = g_wait_test_us.load() ? 1u : 0u;
    int launches = 0;
    e = launch_bwd(dt, a, plan, stream, &launches);
    return finish_call(e, launches, stream);
}

template ln_status bwd_impl<float>(Dtype, bool, const float*, const float*, const float*,
                                   const float*, const float*, float*, float*, float*, int64_t,
                                   int64_t, void*, size_t, bool, ln_stream_t);
template ln_status bwd_impl<__nv_bfloat16>(Dtype, bool, const __nv_bfloat16*, const __nv_bfloat16*,
                                           const __nv_bfloat16*, const float*, const float*,
                                           __nv_bfloat16*, __nv_bfloat16*, __nv_bfloat16*,
                                           int64_t, int64_t, void*, size_t, bool, ln_stream_t);

}  // namespace lnk

namespace lnk {
namespace {
template <typename T>
ln_status softmax_impl(Dtype dt, bool bwd, const T* a, const T* b, const T* mask,
                       int64_t mask_rows, float scale, int64_t rows, int64_t cols, T* out,
                       ln_stream_t stream_) {
    t_last_launches = 0;
    if (!std::isfinite(scale)) return LN_EINVAL;
    ln_status st = check_sizes(rows, cols);
    if (st != LN_OK) return st;
    if (mask && (mask_rows < 1 || mask_rows > LN_MAX_ROWS)) return LN_EINVAL;
    if (rows == 0) return LN_OK;
    if (!a || !out || (bwd && !b)) return LN_EINVAL;
    st = check_device();
    if (st != LN_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const void* ptrs[] = {a, b, mask, out};
    SoftmaxArgs s;
    s.a = a;
    s.b = b;
    s.mask = mask;
    s.mask_rows = mask ? (int)mask_rows : 1;
    s.scale = scale;
    s.rows = (int)rows;
    s.cols = (int)cols;
    s.out = out;
    s.status = status_word();
    s.wait_limit_ns = wait_limit_ns();
    int launches = 0;
    cudaError_t e = launch_softmax(dt, bwd, s, vector_ok(dt, (int)cols, ptrs, 4),
                                   g_force_path.load(), stream, &launches);
    return finish_call(e, launches, stream);
}
}  // namespace
}  // namespace lnk

namespace lnk {
namespace {
template <typename T>
ln_status xent_impl(Dtype dt, const T* logits, const int32_t* targets, int64_t rows, int64_t V,
                    float alpha, float dloss, float* losses, T* dlogits, ln_stream_t stream_) {
    t_last_launches = 0;
    if (!std::isfinite(alpha) || alpha < 0.f || alpha > 1.f || !std::isfinite(dloss))
        return LN_EINVAL;
    if (rows < 0 || V <= 0) return LN_EINVAL;
    if (rows > LN_MAX_ROWS || V > LN_XENT_MAX_V) return LN_EUNSUPPORTED;
    if (rows == 0) return LN_OK;
    if (!logits || !targets || (!losses && !dlogits)) return LN_EINVAL;
    ln_status st = check_device();
    if (st != LN_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    const void* ptrs[] = {logits, dlogits};
    XentArgs a;
    a.logits = logits;
    a.targets = targets;
    a.rows = (int)rows;
    a.V = (int)V;
    a.alpha = alpha;
    a.dloss = dloss;
    a.losses = losses;
    a.dlogits = dlogits;
    a.status = status_word();
    a.wait_limit_ns = wait_limit_ns();
    int launches = 0;
    cudaError_t e = launch_xent(dt, a, vector_ok(dt, (int)V, ptrs, 2), stream, &launches);
    return finish_call(e, launches, stream);
}
}  // namespace
}  // namespace lnk

namespace lnk {
namespace {
template <typename T>
ln_status dropout_bwd_impl(Dtype dt, const T* ds, float p, uint64_t seed, uint64_t offset,
                           int64_t rows, int64_t cols, T* dh, T* dbias, void* ws, size_t ws_bytes,
                           bool own_ws, ln_stream_t stream_, const uint8_t* keep = nullptr) {
    t_last_launches = 0;
    if (!std::isfinite(p) || p < 0.f || p >= 1.f) return LN_EINVAL;
    ln_status st = check_sizes(rows, cols);
    if (st != LN_OK) return st;
    if (!dbias || (rows > 0 && (!ds || !dh))) return LN_EINVAL;
    if (!own_ws && !ws) return LN_EINVAL;
    if (!own_ws && (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return LN_EALIGN;
    st = check_device();
    if (st != LN_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (rows == 0) return finish_call(cudaMemsetAsync(dbias, 0, (size_t)cols * sizeof(T), stream), 0, stream);
    const void* ptrs[] = {ds, dh};
    const bool vec = dropout_bwd_vector(dt, (int)cols, vector_ok(dt, (int)cols, ptrs, 2));
    const int segs = dropout_bwd_segments((int)rows, (int)cols, device_info(-1).sms,
                                          vec ? (dt == Dtype::F32 ? 4 : 8) : 1);
    const size_t need = kWorkspaceHeader + (size_t)segs * (size_t)cols * 2 * sizeof(float);
    st = acquire_workspace(own_ws, ws, ws_bytes, need, stream);
    if (st != LN_OK) return st;
    DropoutBwdArgs a;
    a.ds = ds;
    a.dh = dh;
    a.dbias = dbias;
    a.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + kWorkspaceHeader);
    a.rows = (int)rows;
    a.cols = (int)cols;
    a.segs = segs;
    a.scale = 1.0f / (1.0f - p);
    a.thr = drop_threshold(p);
    a.seed = seed;
    a.offset = offset;
    a.status = status_word();
    a.wait_limit_ns = wait_limit_ns();
    a.keep = keep;
    int launches = 0;
    cudaError_t e = launch_dropout_bwd(dt, a, vec, stream, &launches);
    return finish_call(e, launches, stream);
}
}  // namespace
}  // namespace lnk

using lnk::Dtype;

extern "C" {

ln_status ln_fwd_f32(const float* x, const float* res, const float* gamma, const float* beta,
                     float eps, int64_t rows, int64_t cols, float* out, float* res_out,
                     float* mean, float* rstd, ln_stream_t stream) {
    return lnk::fwd_impl<float>(Dtype::F32, false, x, res, gamma, beta, eps, rows, cols, out, res_out,
                                mean, rstd, stream);
}

ln_status ln_fwd_bf16(const ln_bf16* x, const ln_bf16* res, const ln_bf16* gamma,
                      const ln_bf16* beta, float eps, int64_t rows, int64_t cols, ln_bf16* out,
                      ln_bf16* res_out, float* mean, float* rstd, ln_stream_t stream) {
    using B = __nv_bfloat16;
    return lnk::fwd_impl<B>(Dtype::BF16, false, reinterpret_cast<const B*>(x),
                            reinterpret_cast<const B*>(res), reinterpret_cast<const B*>(gamma),
                            reinterpret_cast<const B*>(beta), eps, rows, cols,
                            reinterpret_cast<B*>(out), reinterpret_cast<B*>(res_out), mean, rstd,
                            stream);
}

ln_status ln_bwd_f32(const float* dy, const float* x_or_res_out, const float* gamma,
                     const float* mean, const float* rstd, float* dx, float* dgamma,
                     float* dbeta, int64_t rows, int64_t cols, ln_stream_t stream) {
    return lnk::bwd_impl<float>(Dtype::F32, false, dy, x_or_res_out, gamma, mean, rstd, dx, dgamma,
                                dbeta, rows, cols, nullptr, 0, true, stream);
}

ln_status ln_bwd_bf16(const ln_bf16* dy, const ln_bf16* x_or_res_out, const ln_bf16* gamma,
                      const float* mean, const float* rstd, ln_bf16* dx, ln_bf16* dgamma,
                      ln_bf16* dbeta, int64_t rows, int64_t cols, ln_stream_t stream) {
    using B = __nv_bfloat16;
    return lnk::bwd_impl<B>(Dtype::BF16, false, reinterpret_cast<const B*>(dy),
                            reinterpret_cast<const B*>(x_or_res_out),
                            reinterpret_cast<const B*>(gamma), mean, rstd, reinterpret_cast<B*>(dx),
                            reinterpret_cast<B*>(dgamma), reinterpret_cast<B*>(dbeta), rows, cols,
                            nullptr, 0, true, stream);
}

size_t ln_bwd_workspace_bytes(int64_t rows, int64_t cols) {
    if (lnk::check_sizes(rows, cols) != LN_OK) return 0;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const lnk::DeviceInfo& di = lnk::device_info(dev);
    if (di.sms <= 0) return 0;
    return lnk::bwd_workspace_bytes(lnk::bwd_max_grid((int)std::max<int64_t>(rows, 1), di.sms),
                                    (int)cols,
                                    !lnk::bwd_scalar_acc_in_smem((int)cols, (size_t)di.smem_optin));
}

ln_status ln_bwd_f32_ws(const float* dy, const float* x_or_res_out, const float* gamma,
                        const float* mean, const float* rstd, float* dx, float* dgamma,
                        float* dbeta, int64_t rows, int64_t cols, void* workspace,
                        size_t workspace_bytes, ln_stream_t stream) {
    return lnk::bwd_impl<float>(Dtype::F32, false, dy, x_or_res_out, gamma, mean, rstd, dx, dgamma,
                                dbeta, rows, cols, workspace, workspace_bytes, false, stream);
}

ln_status ln_bwd_bf16_ws(const ln_bf16* dy, const ln_bf16* x_or_res_out, const ln_bf16* gamma,
                         const float* mean, const float* rstd, ln_bf16* dx, ln_bf16* dgamma,
                         ln_bf16* dbeta, int64_t rows, int64_t cols, void* workspace,
                         size_t workspace_bytes, ln_stream_t stream) {
    using B = __nv_bfloat16;
    return lnk::bwd_impl<B>(Dtype::BF16, false, reinterpret_cast<const B*>(dy),
                            reinterpret_cast<const B*>(x_or_res_out),
                            reinterpret_cast<const B*>(gamma), mean, rstd, reinterpret_cast<B*>(dx),
                            reinterpret_cast<B*>(dgamma), reinterpret_cast<B*>(dbeta), rows, cols,
                            workspace, workspace_bytes, false, stream);
}

ln_status ln_rms_fwd_f32(const float* x, const float* res, const float* gamma, float eps,
                         int64_t rows, int64_t cols, float* out, float* res_out, float* rrms,
                         ln_stream_t stream) {
    return lnk::fwd_impl<float>(Dtype::F32, true, x, res, gamma, nullptr, eps, rows, cols, out,
                                res_out, nullptr, rrms, stream);
}

ln_status ln_rms_fwd_bf16(const ln_bf16* x, const ln_bf16* res, const ln_bf16* gamma, float eps,
                          int64_t rows, int64_t cols, ln_bf16* out, ln_bf16* res_out, float* rrms,
                          ln_stream_t stream) {
    using B = __nv_bfloat16;
    return lnk::fwd_impl<B>(Dtype::BF16, true, reinterpret_cast<const B*>(x),
                            reinterpret_cast<const B*>(res), reinterpret_cast<const B*>(gamma),
                            nullptr, eps, rows, cols, reinterpret_cast<B*>(out),
                            reinterpret_cast<B*>(res_out), nullptr, rrms, stream);
}

ln_status ln_rms_bwd_f32(const float* dy, const float* x_or_res_out, const float* gamma,
                         const float* rrms, float* dx, float* dgamma, int64_t rows, int64_t cols,
                         ln_stream_t stream) {
    return lnk::bwd_impl<float>(Dtype::F32, true, dy, x_or_res_out, gamma, nullptr, rrms, dx,
                                dgamma, nullptr, rows, cols, nullptr, 0, true, stream);
}

ln_status ln_rms_bwd_bf16(const ln_bf16* dy, const ln_bf16* x_or_res_out, const ln_bf16* gamma,
                          const float* rrms, ln_bf16* dx, ln_bf16* dgamma, int64_t rows,
                          int64_t cols, ln_stream_t stream) {
    using B = __nv_bfloat16;
    return lnk::bwd_impl<B>(Dtype::BF16, true, reinterpret_cast<const B*>(dy),
                            reinterpret_cast<const B*>(x_or_res_out),
                            reinterpret_cast<const B*>(gamma), nullptr, rrms,
                            reinterpret_cast<B*>(dx), reinterpret_cast<B*>(dgamma), nullptr, rows,
                            cols, nullptr, 0, true, stream);
}

ln_status ln_rms_bwd_f32_ws(const float* dy, const float* x_or_res_out, const float* gamma,
                            const float* rrms, float* dx, float* dgamma, int64_t rows,
                            int64_t cols, void* workspace, size_t workspace_bytes,
                            ln_stream_t stream) {
    return lnk::bwd_impl<float>(Dtype::F32, true, dy, x_or_res_out, gamma, nullptr, rrms, dx,
                                dgamma, nullptr, rows, cols, workspace, workspace_bytes, false,
                                stream);
}

ln_status ln_rms_bwd_bf16_ws(const ln_bf16* dy, const ln_bf16* x_or_res_out,
                             const ln_bf16* gamma, const float* rrms, ln_bf16* dx,
                             ln_bf16* dgamma, int64_t rows, int64_t cols, void* workspace,
                             size_t workspace_bytes, ln_stream_t stream) {
    using B = __nv_bfloat16;
    return lnk::bwd_impl<B>(Dtype::BF16, true, reinterpret_cast<const B*>(dy),
                            reinterpret_cast<const B*>(x_or_res_out),
                            reinterpret_cast<const B*>(gamma), nullptr, rrms,
                            reinterpret_cast<B*>(dx), reinterpret_cast<B*>(dgamma), nullptr, rows,
                            cols, workspace, workspace_bytes, false, stream);
}


ln_status ln_softmax_fwd_f32(const float* x, const float* mask, int64_t mask_rows, float scale,
                             int64_t rows, int64_t cols, float* y, ln_stream_t stream) {
    return lnk::softmax_impl<float>(Dtype::F32, false, x, nullptr, mask, mask_rows, scale, rows,
                                    cols, y, stream);
}

ln_status ln_softmax_fwd_bf16(const ln_bf16* x, const ln_bf16* mask, int64_t mask_rows,
                              float scale, int64_t rows, int64_t cols, ln_bf16* y,
                              ln_stream_t stream) {
    using B = __nv_bfloat16;
    return lnk::softmax_impl<B>(Dtype::BF16, false, reinterpret_cast<const B*>(x), nullptr,
                                reinterpret_cast<const B*>(mask), mask_rows, scale, rows, cols,
                                reinterpret_cast<B*>(y), stream);
}

ln_status ln_softmax_bwd_f32(const float* dy, const float* y, float scale, int64_t rows,
                             int64_t cols, float* dx, ln_stream_t stream) {
    return lnk::softmax_impl<float>(Dtype::F32, true, dy, y, nullptr, 1, scale, rows, cols, dx,
                                    stream);
}

ln_status ln_softmax_bwd_bf16(const ln_bf16* dy, const ln_bf16* y, float scale, int64_t rows,
                              int64_t cols, ln_bf16* dx, ln_stream_t stream) {
    using B = __nv_bfloat16;
    return lnk::softmax_impl<B>(Dtype::BF16, true, reinterpret_cast<const B*>(dy),
                                reinterpret_cast<const B*>(y), nullptr, 1, scale, rows, cols,
                                reinterpret_cast<B*>(dx), stream);
}

ln_status ln_xent_f32(const float* logits, const int32_t* targets, int64_t rows, int64_t V,
                      float alpha, float dloss, float* losses, float* dlogits,
                      ln_stream_t stream) {
    return lnk::xent_impl<float>(Dtype::F32, logits, targets, rows, V, alpha, dloss, losses,
                                 dlogits, stream);
}

ln_status ln_xent_bf16(const ln_bf16* logits, const int32_t* targets, int64_t rows, int64_t V,
                       float alpha, float dloss, float* losses, ln_bf16* dlogits,
                       ln_stream_t stream) {
    using B = __nv_bfloat16;
    return lnk::xent_impl<B>(Dtype::BF16, reinterpret_cast<const B*>(logits), targets, rows, V,
                             alpha, dloss, losses, reinterpret_cast<B*>(dlogits), stream);
}

ln_status ln_fwd_bias_dropout_f32(const float* h, const float* bias, const float* res,
                                  const float* gamma, const float* beta, float eps, float p,
                                  uint64_t seed, uint64_t offset, int64_t rows, int64_t cols,
                                  float* out, float* res_out, float* mean, float* rstd,
                                  ln_stream_t stream) {
    if (!bias || (rows > 0 && !res) || !std::isfinite(p) || p < 0.f || p >= 1.f) return LN_EINVAL;
    return lnk::fwd_impl<float>(Dtype::F32, false, h, res, gamma, beta, eps, rows, cols, out,
                                res_out, mean, rstd, stream, bias, p, seed, offset);
}

ln_status ln_fwd_bias_dropout_bf16(const ln_bf16* h, const ln_bf16* bias, const ln_bf16* res,
                                   const ln_bf16* gamma, const ln_bf16* beta, float eps, float p,
                                   uint64_t seed, uint64_t offset, int64_t rows, int64_t cols,
                                   ln_bf16* out, ln_bf16* res_out, float* mean, float* rstd,
                                   ln_stream_t stream) {
    using B = __nv_bfloat16;
    if (!bias || (rows > 0 && !res) || !std::isfinite(p) || p < 0.f || p >= 1.f) return LN_EINVAL;
    return lnk::fwd_impl<B>(Dtype::BF16, false, reinterpret_cast<const B*>(h),
                            reinterpret_cast<const B*>(res), reinterpret_cast<const B*>(gamma),
                            reinterpret_cast<const B*>(beta), eps, rows, cols,
                            reinterpret_cast<B*>(out), reinterpret_cast<B*>(res_out), mean, rstd,
                            stream, reinterpret_cast<const B*>(bias), p, seed, offset);
}

ln_status ln_dropout_bwd_f32(const float* ds, float p, uint64_t seed, uint64_t offset,
                             int64_t rows, int64_t cols, float* dh, float* dbias,
                             ln_stream_t stream) {
    return lnk::dropout_bwd_impl<float>(Dtype::F32, ds, p, seed, offset, rows, cols, dh, dbias,
                                        nullptr, 0, true, stream);
}

ln_status ln_dropout_bwd_bf16(const ln_bf16* ds, float p, uint64_t seed, uint64_t offset,
                              int64_t rows, int64_t cols, ln_bf16* dh, ln_bf16* dbias,
                              ln_stream_t stream) {
    using B = __nv_bfloat16;
    return lnk::dropout_bwd_impl<B>(Dtype::BF16, reinterpret_cast<const B*>(ds), p, seed, offset,
                                    rows, cols, reinterpret_cast<B*>(dh),
                                    reinterpret_cast<B*>(dbias), nullptr, 0, true, stream);
}

ln_status ln_dropout_bwd_f32_ws(const float* ds, float p, uint64_t seed, uint64_t offset,
                                int64_t rows, int64_t cols, float* dh, float* dbias,
                                void* workspace, size_t workspace_bytes, ln_stream_t stream) {
    return lnk::dropout_bwd_impl<float>(Dtype::F32, ds, p, seed, offset, rows, cols, dh, dbias,
                                        workspace, workspace_bytes, false, stream);
}

ln_status ln_dropout_bwd_bf16_ws(const ln_bf16* ds, float p, uint64_t seed, uint64_t offset,
                                 int64_t rows, int64_t cols, ln_bf16* dh, ln_bf16* dbias,
                                 void* workspace, size_t workspace_bytes, ln_stream_t stream) {
    using B = __nv_bfloat16;
    return lnk::dropout_bwd_impl<B>(Dtype::BF16, reinterpret_cast<const B*>(ds), p, seed, offset,
                                    rows, cols, reinterpret_cast<B*>(dh),
                                    reinterpret_cast<B*>(dbias), workspace, workspace_bytes, false,
                                    stream);
}

size_t ln_dropout_keep_bytes(int64_t rows, int64_t cols) {
    if (lnk::check_sizes(rows, cols) != LN_OK) return 0;
    return (size_t)rows * (size_t)((cols + 7) / 8);
}

ln_status ln_fwd_bias_dropout_keep_f32(const float* h, const float* bias, const float* res,
                                       const float* gamma, const float* beta, float eps, float p,
                                       uint64_t seed, uint64_t offset, int64_t rows, int64_t cols,
                                       float* out, float* res_out, float* mean, float* rstd,
                                       uint8_t* keep, ln_stream_t stream) {
    if (!bias || (rows > 0 && (!res || !keep)) || !std::isfinite(p) || p < 0.f || p >= 1.f)
        return LN_EINVAL;
    return lnk::fwd_impl<float>(Dtype::F32, false, h, res, gamma, beta, eps, rows, cols, out,
                                res_out, mean, rstd, stream, bias, p, seed, offset, keep);
}

ln_status ln_fwd_bias_dropout_keep_bf16(const ln_bf16* h, const ln_bf16* bias,
                                        const ln_bf16* res, const ln_bf16* gamma,
                                        const ln_bf16* beta, float eps, float p, uint64_t seed,
                                        uint64_t offset, int64_t rows, int64_t cols,
                                        ln_bf16* out, ln_bf16* res_out, float* mean, float* rstd,
                                        uint8_t* keep, ln_stream_t stream) {
    using B = __nv_bfloat16;
    if (!bias || (rows > 0 && (!res || !keep)) || !std::isfinite(p) || p < 0.f || p >= 1.f)
        return LN_EINVAL;
    return lnk::fwd_impl<B>(Dtype::BF16, false, reinterpret_cast<const B*>(h),
                            reinterpret_cast<const B*>(res), reinterpret_cast<const B*>(gamma),
                            reinterpret_cast<const B*>(beta), eps, rows, cols,
                            reinterpret_cast<B*>(out), reinterpret_cast<B*>(res_out), mean, rstd,
                            stream, reinterpret_cast<const B*>(bias), p, seed, offset, keep);
}

ln_status ln_dropout_bwd_keep_f32(const float* ds, float p, const uint8_t* keep, int64_t rows,
                                  int64_t cols, float* dh, float* dbias, ln_stream_t stream) {
    if (rows > 0 && !keep) return LN_EINVAL;
    return lnk::dropout_bwd_impl<float>(Dtype::F32, ds, p, 0, 0, rows, cols, dh, dbias, nullptr,
                                        0, true, stream, keep);
}

ln_status ln_dropout_bwd_keep_bf16(const ln_bf16* ds, float p, const uint8_t* keep,
                                   int64_t rows, int64_t cols, ln_bf16* dh, ln_bf16* dbias,
                                   ln_stream_t stream) {
    using B = __nv_bfloat16;
    if (rows > 0 && !keep) return LN_EINVAL;
    return lnk::dropout_bwd_impl<B>(Dtype::BF16, reinterpret_cast<const B*>(ds), p, 0, 0, rows,
                                    cols, reinterpret_cast<B*>(dh), reinterpret_cast<B*>(dbias),
                                    nullptr, 0, true, stream, keep);
}

ln_status ln_dropout_bwd_keep_f32_ws(const float* ds, float p, const uint8_t* keep,
                                     int64_t rows, int64_t cols, float* dh, float* dbias,
                                     void* workspace, size_t workspace_bytes, ln_stream_t stream) {
    if (rows > 0 && !keep) return LN_EINVAL;
    return lnk::dropout_bwd_impl<float>(Dtype::F32, ds, p, 0, 0, rows, cols, dh, dbias, workspace,
                                        workspace_bytes, false, stream, keep);
}

ln_status ln_dropout_bwd_keep_bf16_ws(const ln_bf16* ds, float p, const uint8_t* keep,
                                      int64_t rows, int64_t cols, ln_bf16* dh, ln_bf16* dbias,
                                      void* workspace, size_t workspace_bytes,
                                      ln_stream_t stream) {
    using B = __nv_bfloat16;
    if (rows > 0 && !keep) return LN_EINVAL;
    return lnk::dropout_bwd_impl<B>(Dtype::BF16, reinterpret_cast<const B*>(ds), p, 0, 0, rows,
                                    cols, reinterpret_cast<B*>(dh), reinterpret_cast<B*>(dbias),
                                    workspace, workspace_bytes, false, stream, keep);
}

ln_status ln_device_check(ln_stream_t stream_) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return lnk::cuda_fail(e);
    unsigned* sw = lnk::status_word();
    if (!sw) return lnk::cuda_fail(cudaGetLastError());
    unsigned word = 0;
    e = cudaMemcpy(&word, sw, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return lnk::cuda_fail(e);
    if (word == 0) return LN_OK;
    const unsigned zero = 0;
    e = cudaMemcpy(sw, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return lnk::cuda_fail(e);
    // A backward that gave up may have left partial sums in its workspace, where the next
    // call would take them for its own: clear this stream's workspace and the fixed scratch
    // of the allocation-free entry point, on this stream (so that the clearing is ordered
    // before any later work on it, whatever kind of stream it is), and wait for it.
    {
        const int dev = lnk::current_device();
        std::lock_guard<std::mutex> lk(lnk::g_mu);
        auto it = lnk::g_workspaces.find(std::make_pair(dev, stream));
        if (it != lnk::g_workspaces.end() && it->second.ptr) {
            e = cudaMemsetAsync(it->second.ptr, 0, it->second.bytes, stream);
            if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return lnk::cuda_fail(e);
        }
    }
    e = lnk::noalloc_scratch_clear(stream);
    if (e != cudaSuccess) return lnk::cuda_fail(e);
    return (word & lnk::kStatusTimeout) ? LN_ETIMEOUT : LN_OK;
}

ln_status ln_release(void) {
    std::lock_guard<std::mutex> lk(lnk::g_mu);
    int cur = -1;
    cudaGetDevice(&cur);
    ln_status st = LN_OK;
    for (auto& kv : lnk::g_workspaces) {
        if (!kv.second.ptr) continue;
        cudaSetDevice(kv.first.first);
        cudaError_t e = cudaDeviceSynchronize();
        if (e == cudaSuccess) e = cudaFree(kv.second.ptr);
        if (e != cudaSuccess) st = lnk::cuda_fail(e);
    }
    lnk::g_workspaces.clear();
    if (cur >= 0) cudaSetDevice(cur);
    return st;
}

const char* ln_status_str(ln_status status) {
    switch (status) {
        case LN_OK: return "LN_OK";
        case LN_EINVAL: return "LN_EINVAL: invalid argument";
        case LN_EALIGN: return "LN_EALIGN: workspace not 256-byte aligned";
        case LN_EUNSUPPORTED: return "LN_EUNSUPPORTED: size or device not supported";
        case LN_ECUDA: return "LN_ECUDA: CUDA runtime error";
        case LN_ETIMEOUT: return "LN_ETIMEOUT: a bounded device wait ran out";
        case LN_ENOSPACE: return "LN_ENOSPACE: workspace too small";
    }
    return "unknown ln_status";
}

int ln_last_cuda_error(void) { return lnk::t_last_cuda_error; }

int ln_version(void) { return 10000; }

int ln_debug_force_path(int path) {
    if (path < lnk::kPathAuto || path > lnk::kPathScalar) path = lnk::kPathAuto;
    return lnk::g_force_path.exchange(path);
}

void ln_debug_wait_test(unsigned limit_us) { lnk::g_wait_test_us.store(limit_us); }

int ln_last_launch_count(void) { return lnk::t_last_launches; }

}  // extern "C"
