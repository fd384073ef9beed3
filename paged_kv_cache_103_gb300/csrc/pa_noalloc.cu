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
// (with that device current) and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB, PA_NOALLOC_SCRATCH_BYTES
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the current device's scratch array, set up on first use.
pa_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
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
