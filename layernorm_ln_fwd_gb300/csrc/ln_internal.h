// ln_internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dropout_rng.h"
#include "ln.h"

namespace lnk {

enum class Dtype { F32, BF16 };

enum Path { kPathAuto = 0, kPathWarp = 1, kPathBlock = 2, kPathScalar = 3 };

struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int smem_optin = 0;     // max dynamic shared memory per block (opt-in), bytes
    int smem_per_sm = 0;    // shared memory per SM, bytes
    int l2_bytes = 0;
    int cc_major = 0, cc_minor = 0;
};

// Cached properties of device `dev` (-1: the current device).
const DeviceInfo& device_info(int dev);

// Per-device status word (a __device__ variable); its device address on the current device.
unsigned* status_word();

// The bias + dropout + residual prologue of the LayerNorm forward: s = res + keep * (x +
// bias) * scale, keep from Philox-4x32-10 at (seed, offset) with threshold floor(p 2^32)
// (DropoutRng::make), scale = 1 / (1 - p).  bias == nullptr: no prologue.
struct Prologue {
    const void* bias = nullptr;
    float scale = 1.f;
    DropoutRng rng{};
    // Optional: the keep decisions also stored as bits, rows padded to whole bytes: bit
    // (c % 8) of keep_out[row * keep_stride + c / 8] for column c, keep_stride = ceil(cols / 8).
    uint8_t* keep_out = nullptr;
    int keep_stride = 0;
};

struct FwdArgs {
    const void* x;
    const void* res;    // may be null
    const void* gamma;
    const void* beta;
    float eps;
    int rows;
    int cols;
    void* out;
    void* res_out;      // may be null
    float* mean;
    float* rstd;
    unsigned* status;
    uint64_t wait_limit_ns;
    Prologue pro;
};

struct BwdArgs {
    const void* dy;
    const void* xr;
    const void* gamma;
    const float* mean;    // null for the RMSNorm backward
    const float* rstd;    // rstd, or the RMSNorm's 1 / rms
    void* dx;
    void* dgamma;
    void* dbeta;          // null for the RMSNorm backward
    int rows;
    int cols;
    float* partials;      // [2][grid][cols] (hi, lo) fp32 pairs: dgamma, then dbeta
    unsigned* counters;   // the workspace header: zero words that no kernel writes
    unsigned* status;
    uint64_t wait_limit_ns;
    unsigned wait_extra;  // test hook: the finish also waits for a word nothing writes
};

// A launch plan for the backward: which kernel, how many blocks (= rows of partials).
struct BwdPlan {
    bool rms = false;     // the RMSNorm backward (one row sum, one column sum: dgamma)
    int path = kPathAuto;
    int per_thread = 0;   // vectors per lane (warp path) or per thread (block path)
    int wpr = 1;          // warp path: warps per row
    int tile_rows = 0;    // warp path: rows per tile
    int threads = 0;
    int grid = 0;
    bool kahan = false;   // compensated per-thread column sums (block path)
    int stages = 0;       // rows in flight per block (block path); accumulator place (scalar)
    size_t smem = 0;
};

// Whether the 128-bit vector kernels may be used: every pointer 16-byte aligned and a row a
// multiple of 16 bytes.
bool vector_ok(Dtype dt, int cols, const void* const* ptrs, int nptrs);

// Launch `kern` with programmatic stream serialization allowed (and cooperatively when
// `cooperative`): cudaLaunchKernelEx, so that it can also be captured into a CUDA graph.
cudaError_t launch_kernel(const void* kern, dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, void** args, bool cooperative);

cudaError_t launch_fwd(Dtype dt, const FwdArgs& a, bool aligned, int path_override,
                       cudaStream_t stream, int* launches);
// The RMSNorm forward: `beta` and `mean` are unused (may be null); `rstd` receives 1 / rms.
cudaError_t launch_rms_fwd(Dtype dt, const FwdArgs& a, bool aligned, int path_override,
                           cudaStream_t stream, int* launches);
// The LayerNorm forward with the bias + dropout + residual prologue (a.pro.bias set).
cudaError_t launch_bdr_fwd(Dtype dt, const FwdArgs& a, bool aligned, int path_override,
                           cudaStream_t stream, int* launches);

// Plans (kernel, grid, shared memory) the backward of a LayerNorm, or of an RMSNorm when
// `rms` (then the plan's launch goes to launch_rms_bwd).
cudaError_t plan_bwd(Dtype dt, bool rms, int rows, int cols, bool aligned, int path_override,
                     BwdPlan* plan);
cudaError_t plan_rms_bwd(Dtype dt, int rows, int cols, bool aligned, int path_override,
                         BwdPlan* plan);

// Largest grid any backward plan can use for `rows` rows on a device with `sms` SMs.
int bwd_max_grid(int rows, int sms);

constexpr size_t kWorkspaceHeader = 256;  // a header of zero words, kept for alignment

// Whether the scalar kernel's running (hi, lo) column sums fit its shared memory.
inline bool bwd_scalar_acc_in_smem(int cols, size_t smem_optin) {
    return 16ull * (size_t)cols <= smem_optin / 2;
}

// The workspace: the header, the partial sums [2 statistics][grid][cols] as (hi, lo) fp32
// pairs, and -- when `acc_region` (the scalar kernel on rows too wide for its shared memory)
// -- as much again for that kernel's running sums.  Every byte is zero between calls.
inline size_t bwd_workspace_bytes(int grid, int cols, bool acc_region) {
    return kWorkspaceHeader + 2ull * (size_t)grid * (size_t)cols * 2 * sizeof(float) *
                                  (acc_region ? 2 : 1);
}

// Whether a plan's kernel keeps running sums in the workspace.
inline bool bwd_plan_acc_region(const BwdPlan& p) {
    return p.path == kPathScalar && p.stages == 0;
}

cudaError_t launch_bwd(Dtype dt, const BwdArgs& a, const BwdPlan& plan, cudaStream_t stream,
                       int* launches);
cudaError_t launch_rms_bwd(Dtype dt, const BwdArgs& a, const BwdPlan& plan, cudaStream_t stream,
                           int* launches);

// The fused softmax: forward (a = x, optional additive mask [mask_rows, cols], out = y) or
// backward (a = dy, b = y, out = dx).
struct SoftmaxArgs {
    const void* a;
    const void* b;
    const void* mask;
    int mask_rows;
    float scale;
    int rows;
    int cols;
    void* out;
    unsigned* status;
    uint64_t wait_limit_ns;
};

cudaError_t launch_softmax(Dtype dt, bool bwd, const SoftmaxArgs& a, bool aligned,
                           int path_override, cudaStream_t stream, int* launches);

// The fused cross-entropy with label smoothing: losses (optional) and dlogits (optional;
// may alias logits).
struct XentArgs {
    const void* logits;
    const int* targets;
    int rows;
    int V;
    float alpha;
    float dloss;
    float* losses;
    void* dlogits;
    unsigned* status;  // the per-device status word (bounded waits)
    uint64_t wait_limit_ns;
};

cudaError_t launch_xent(Dtype dt, const XentArgs& a, bool aligned, cudaStream_t stream,
                        int* launches);

// Backward of the bias + dropout + residual prologue: dh = ds * keep * scale (keep from the
// generator, or from the bits the forward stored) and the deterministic column sums dbias (partials: [segs][cols] (hi, lo) fp32 pairs that announce
// themselves, left zero), in one cooperative launch.
struct DropoutBwdArgs {
    const void* ds;
    void* dh;
    void* dbias;
    float* partials;
    int rows, cols, segs;
    float scale;
    uint32_t thr;
    unsigned long long seed, offset;
    unsigned* status;          // the per-device status word (bounded waits)
    uint64_t wait_limit_ns;
    const uint8_t* keep = nullptr;  // stored keep bits (Prologue::keep_out's layout), or null
};

// Whether the kernels take 16-byte vectors (rows of whole vectors, aligned pointers).
bool dropout_bwd_vector(Dtype dt, int cols, bool aligned);
// Row segments (partial rows) for cv columns per thread (16-byte vectors or 1); at most
// min(rows, 8 * sms).
int dropout_bwd_segments(int rows, int cols, int sms, int cv);
cudaError_t launch_dropout_bwd(Dtype dt, const DropoutBwdArgs& a, bool vec, cudaStream_t stream,
                               int* launches);

// Zeroes the allocation-free entry point's fixed scratch on the current device, if a call
// there has used it: on `stream`, which is then synchronised (after a backward gave up).
cudaError_t noalloc_scratch_clear(cudaStream_t stream);

// The backward behind every ln_bwd_* entry point: argument checks, the launch plan, the
// workspace (the library's own per-stream one when `own_ws`, else `ws` of `ws_bytes` bytes,
// zero between calls), the launch, and the LN_CHECK handling.  Instantiated for float and
// __nv_bfloat16.
// `rms`: the RMSNorm backward (mean and dbeta unused and may be null).
template <typename T>
ln_status bwd_impl(Dtype dt, bool rms, const T* dy, const T* xr, const T* gamma,
                   const float* mean, const float* rstd, T* dx, T* dgamma, T* dbeta,
                   int64_t rows, int64_t cols, void* ws, size_t ws_bytes, bool own_ws,
                   ln_stream_t stream);

// Occupancy (resident blocks per SM) of a kernel, cached per (device, kernel, threads, smem).
int blocks_per_sm(const void* kernel, int threads, size_t smem);

// Records `e` as the value ln_last_cuda_error() reports on this host thread.
void record_cuda_error(cudaError_t e);

}  // namespace lnk
