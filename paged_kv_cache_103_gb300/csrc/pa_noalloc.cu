// pa_decode_noalloc: pa_decode for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a decode workspace: code that runs where
// cudaMalloc is off limits (inside a custom allocator's own callbacks, in a
// process whose device memory is owned and pre-partitioned by a host
// framework, or in plugins that must not change the device's memory footprint
// per call).  This entry point takes only inputs and outputs.  Its scratch is
// one file-scope __device__ array of kScratchBytes, which every GPU that loads
// the library holds until the process exits.
//
// The array's name, used in host code, is only a host-side stand-in; its
// device address is looked up once per device with cudaGetSymbolAddress
// (with that device current) and cached together with the device's current
// context.  A device reset tears the context down and unloads the module, so
// a call under a different context looks the address up again instead of
// using a stale one.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB, PA_NOALLOC_SCRATCH_BYTES
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// The driver's cuCtxGetCurrent, reached through the runtime (no link-time
// dependence on the driver library).
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

// Device address of the current device's scratch array, set up on the first
// use under each context of the device.
pa_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    CtxGetCurrentFn get = ctx_get_current();
    CUcontext ctx = nullptr;
    if (!get || get(&ctx) != CUDA_SUCCESS) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
        // The lookup also makes the device's primary context current if no
        // context was yet; the context is then what the cached address keys on.
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
        if (get(&ctx) != CUDA_SUCCESS || !ctx) return PA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" {

PA_API pa_status pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int32_t max_blocks,
                                   const int32_t* context_lens, int32_t max_context_len,
                                   int32_t B, int32_t H, int32_t Hkv, int32_t d,
                                   int32_t block_size, int32_t num_blocks, float scale,
                                   pa_dtype dtype, void* out, void* stream) {
    if (B == 0) return PA_OK;
    const size_t need = pa_decode_workspace_size(B, H, d);
    if (need == 0) return (B < 0 || H <= 0) ? PA_ERR_INVALID : PA_ERR_UNSUPPORTED;
    if (need > kScratchBytes) return PA_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const pa_status st = scratch_address(&scratch);
    if (st != PA_OK) return st;
    // The arrival counters at the front of the workspace must start at zero;
    // clear them on every call (a memset, not an allocation).
    const size_t counters = (((size_t)B * H * sizeof(int32_t)) + 255) & ~size_t(255);
    if (cudaMemsetAsync(scratch, 0, counters, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    return pa_decode(q, k_cache, v_cache, block_tables, max_blocks, context_lens,
                     max_context_len, B, H, Hkv, d, block_size, num_blocks, scale, dtype, out,
                     scratch, kScratchBytes, stream);
}

}  // extern "C"
