// Runtime pieces of the C ABI: status strings, the per-device error word that
// kernels raise bits in (instead of trapping), SM-count caching, the decode
// workspace initialisation, and two measurement aids (the bounded-wait self
// test and the mma.sync throughput ceiling).
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"
#include "pa_common.cuh"

namespace {

// One word per device (a file-scope __device__ variable exists once per device
// that loads this library).  Kernels OR PA_DEVERR_* bits into it.
__device__ unsigned int g_error_word;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_error_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

// One CTA waits, with the pipelines' own bounded wait, on an mbarrier that
// nothing ever arrives on; the wait gives up after limit_ns and reports it.
__global__ void wait_selftest_kernel(uint64_t limit_ns, unsigned int* err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        pa::mbar_init(&bar, 1);
        pa::fence_barrier_init();
    }
    __syncthreads();
    const bool done = pa::mbar_wait(&bar, 0, limit_ns);
    if (!__all_sync(0xffffffffu, done) && threadIdx.x == 0)
        pa::raise_error(err, PA_DEVERR_TIMEOUT);
}

// Throughput ceiling of the mma.sync m16n8k16 path the attention kernels
// use: every warp issues kMmaChains independent MMAs per iteration from
// registers (no memory traffic in the loop) and writes one float at the end.
constexpr int kMmaChains = 8;
constexpr int kMmaWarps = 8;         // per CTA
constexpr int kMmaCtasPerSm = 2;

template <bool kBF16>
__global__ void __launch_bounds__(kMmaWarps * 32)
mma_ceiling_kernel(int32_t iters, uint32_t seed, float* sink) {
    // small finite f16 / bf16 pairs (the exponent field kept below its top)
    uint32_t a[4] = {seed & 0x3bff3bffu, (seed * 3u) & 0x3bff3bffu, (seed * 5u) & 0x3bff3bffu,
                     (seed * 7u) & 0x3bff3bffu};
    const uint32_t b0 = (seed * 11u) & 0x3bff3bffu, b1 = (seed * 13u) & 0x3bff3bffu;
    float d[kMmaChains][4];
#pragma unroll
    for (int j = 0; j < kMmaChains; ++j) d[j][0] = d[j][1] = d[j][2] = d[j][3] = 0.f;
    for (int32_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < kMmaChains; ++j) pa::mma_16816<kBF16>(d[j], a, b0, b1);
    }
    float t = 0.f;
#pragma unroll
    for (int j = 0; j < kMmaChains; ++j) t += d[j][0] + d[j][1] + d[j][2] + d[j][3];
    sink[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = t;
}

}  // namespace

namespace pa {

unsigned int* device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_error_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        g_error_ptr[dev] = static_cast<unsigned int*>(p);
    }
    return g_error_ptr[dev];
}

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 0;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

}  // namespace pa

extern "C" {

PA_API const char* pa_status_str(pa_status s) {
    switch (s) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID: return "invalid argument or operation";
        case PA_ERR_OOM: return "out of KV blocks";
        case PA_ERR_NOT_FOUND: return "unknown sequence";
        case PA_ERR_BOUNDS: return "kernel met an index outside its buffers";
        case PA_ERR_CUDA: return "CUDA runtime error";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PA_ERR_TIMEOUT: return "kernel wait timed out";
    }
    return "unknown status";
}

PA_API int32_t pa_version(void) { return 1; }

PA_API pa_status pa_check_device_errors(void* stream, uint32_t* flags) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
    unsigned int* word = pa::device_error_word();
    if (!word) return PA_ERR_CUDA;
    unsigned int host = 0;
    if (cudaMemcpyAsync(&host, word, sizeof host, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return PA_ERR_CUDA;
    if (cudaMemsetAsync(word, 0, sizeof host, st) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return PA_ERR_CUDA;
    if (flags) *flags = host;
    if (host & PA_DEVERR_TIMEOUT) return PA_ERR_TIMEOUT;
    if (host) return PA_ERR_BOUNDS;
    return PA_OK;
}

PA_API pa_status pa_selftest_wait_timeout(uint32_t limit_us, void* stream) {
    if (limit_us == 0 || limit_us > 1000000) return PA_ERR_INVALID;
    unsigned int* err = pa::device_error_word();
    if (!err) return PA_ERR_CUDA;
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        (uint64_t)limit_us * 1000u, err);
    return pa::cuda_status(cudaGetLastError());
}

PA_API pa_status pa_measure_mma_ceiling(int32_t bf16, int32_t iters, float* sink,
                                        size_t sink_bytes, int64_t* flops, void* stream) {
    if (iters <= 0 || iters > (1 << 20) || !sink || !flops) return PA_ERR_INVALID;
    const int sms = pa::device_sm_count();
    if (sms <= 0) return PA_ERR_CUDA;
    const int grid = sms * kMmaCtasPerSm;
    if (sink_bytes < (size_t)grid * kMmaWarps * 32 * sizeof(float)) return PA_ERR_INVALID;
    // 2 flops per multiply-add, 16 x 8 x 16 multiply-adds per MMA
    *flops = (int64_t)2 * 16 * 8 * 16 * kMmaChains * iters * (int64_t)grid * kMmaWarps;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (bf16)
        mma_ceiling_kernel<true><<<grid, kMmaWarps * 32, 0, st>>>(iters, 0x9e3779b9u, sink);
    else
        mma_ceiling_kernel<false><<<grid, kMmaWarps * 32, 0, st>>>(iters, 0x9e3779b9u, sink);
    return pa::cuda_status(cudaGetLastError());
}

PA_API pa_status pa_decode_workspace_init(void* workspace, size_t bytes, void* stream) {
    if (!workspace && bytes) return PA_ERR_INVALID;
    if (!bytes) return PA_OK;
    return pa::cuda_status(
        cudaMemsetAsync(workspace, 0, bytes, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
