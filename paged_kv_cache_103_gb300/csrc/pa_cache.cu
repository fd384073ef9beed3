// KV append (pa_reshape_and_cache) and copy-on-write block copies
// (pa_copy_blocks).  Both are bit copies of 16-byte vectors; every index is
// checked against its buffer before the access, and a bad one raises a bit in
// the device error word instead of being used.
//
// Sources: "vLLM推理加速深度解析：从PagedAttention原理到生产部署实战", section 2.2
// (each new token's K/V goes into the physical block its current logical block
// points to); "vLLM 深度拆解：当大模型推理学会「分页注意力」", section 3.3
// (append_slot; shared blocks copied only when a sharer writes).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pa.h"
#include "pa_common.cuh"

namespace {

constexpr int kThreads = 256;

// One thread moves one 16-byte vector of K and the same vector of V.
__global__ void __launch_bounds__(kThreads)
reshape_and_cache_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                         const int64_t* __restrict__ slot_mapping, int32_t T,
                         int32_t vecs_per_token, uint4* __restrict__ k_cache,
                         uint4* __restrict__ v_cache, int64_t num_slots,
                         unsigned int* __restrict__ err) {
    const int64_t total = (int64_t)T * vecs_per_token;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = idx / vecs_per_token;
        const int64_t v = idx - t * vecs_per_token;
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;  // padding token
        if (slot >= num_slots) {
            if (v == 0) pa::raise_error(err, PA_DEVERR_SLOT);
            continue;
        }
        const int64_t dst = slot * vecs_per_token + v;
        k_cache[dst] = __ldg(k_new + idx);
        v_cache[dst] = __ldg(v_new + idx);
    }
}

// Two fp32 values -> two OCP E4M3 codes, round to nearest even, saturating at
// +-448; `lo` goes to the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Four fp32 values -> four INT8 codes (nearest integer, ties to even,
// clamped to [-127, 127]); the first value goes to the low byte.
__device__ __forceinline__ uint32_t s8x4(float a, float b, float c, float d) {
    const float v[4] = {a, b, c, d};
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int q = max(-127, min(127, __float2int_rn(v[i])));
        r |= ((uint32_t)q & 0xFFu) << (8 * i);
    }
    return r;
}

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// 8-bit KV append: one warp per (token, KV head) row of 128 values, each lane
// four consecutive values.  FP8: scale = fl32(amax / 448) and code =
// e4m3_rne_sat(fl32(x / scale)); INT8 (kInt8): scale = fl32(amax / 127) and
// code = the nearest integer of fl32(x / scale), ties to even, clamped to
// +-127.  IEEE fp32 divisions; an all-zero row gets scale 0 and zero codes.
// Codes go to cache[slot / bs][slot % bs][h][:], the scale to
// scale[slot / bs][h][slot % bs].
template <typename T, bool kInt8>
__global__ void __launch_bounds__(kThreads)
reshape_and_cache_q8_kernel(const T* __restrict__ k_new, const T* __restrict__ v_new,
                             const int64_t* __restrict__ slot_mapping, int32_t T_tokens,
                             int32_t Hkv, int32_t block_size, uint32_t* __restrict__ k_cache,
                             uint32_t* __restrict__ v_cache, float* __restrict__ k_scale,
                             float* __restrict__ v_scale, int64_t num_slots,
                             unsigned int* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)T_tokens * Hkv;
    for (int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows;
         row += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int64_t t = row / Hkv;
        const int32_t h = (int32_t)(row - t * Hkv);
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (lane == 0) pa::raise_error(err, PA_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / block_size, off = slot - blk * block_size;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const T* src = (which ? v_new : k_new) + row * 128 + lane * 4;
            float x[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) x[e] = to_f32<T>(src[e]);
            float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float s = __fdiv_rn(amax, kInt8 ? 127.0f : 448.0f);
            uint32_t packed = 0;
            if (s != 0.f) {
                if constexpr (kInt8) {
                    packed = s8x4(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s), __fdiv_rn(x[2], s),
                                  __fdiv_rn(x[3], s));
                } else {
                    const uint16_t lo = e4m3x2(__fdiv_rn(x[0], s), __fdiv_rn(x[1], s));
                    const uint16_t hi = e4m3x2(__fdiv_rn(x[2], s), __fdiv_rn(x[3], s));
                    packed = (uint32_t)lo | ((uint32_t)hi << 16);
                }
            }
            uint32_t* dst = (which ? v_cache : k_cache) + (slot * Hkv + h) * 32 + lane;
            *dst = packed;
            if (lane == 0)
                ((which ? v_scale : k_scale))[(blk * Hkv + h) * block_size + off] = s;
        }
    }
}

constexpr int kMaxLayersPerLaunch = 32;

struct LayerPtrs {
    uint4* k[kMaxLayersPerLaunch];
    uint4* v[kMaxLayersPerLaunch];
};

// blockIdx.x = pair, blockIdx.y = layer within this launch's group.
__global__ void __launch_bounds__(kThreads)
copy_blocks_kernel(const __grid_constant__ LayerPtrs layers, const int32_t* __restrict__ pairs,
                   int64_t vecs_per_block, int32_t num_blocks, unsigned int* __restrict__ err) {
    const int32_t p = blockIdx.x;
    const int32_t src = __ldg(pairs + 2 * p);
    const int32_t dst = __ldg(pairs + 2 * p + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0) pa::raise_error(err, PA_DEVERR_PAIR);
        return;
    }
    const uint4* ks = layers.k[blockIdx.y] + (int64_t)src * vecs_per_block;
    const uint4* vs = layers.v[blockIdx.y] + (int64_t)src * vecs_per_block;
    uint4* kd = layers.k[blockIdx.y] + (int64_t)dst * vecs_per_block;
    uint4* vd = layers.v[blockIdx.y] + (int64_t)dst * vecs_per_block;
    for (int64_t i = threadIdx.x; i < vecs_per_block; i += kThreads) {
        kd[i] = ks[i];
        vd[i] = vs[i];
    }
}

// Block copies between two pools (device <-> pinned host for swapping): for
// every pool pair and every (src, dst) pair, block dst of the destination pool
// becomes a copy of block src of the source pool.  blockIdx.x = pair,
// blockIdx.y = pool pair; each thread moves four 16-byte vectors per step
// (loads first, then stores), streaming hints on both sides.
constexpr int kMaxSwapPools = 64;

struct SwapPools {
    const uint4* src[kMaxSwapPools];
    uint4* dst[kMaxSwapPools];
};

__global__ void __launch_bounds__(kThreads)
swap_blocks_kernel(const __grid_constant__ SwapPools pools, const int32_t* __restrict__ pairs,
                   int64_t vecs_per_block, int32_t src_blocks, int32_t dst_blocks,
                   unsigned int* __restrict__ err) {
    const int32_t s = pairs[2 * blockIdx.x];
    const int32_t d = pairs[2 * blockIdx.x + 1];
    if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0) pa::raise_error(err, PA_DEVERR_PAIR);
        return;
    }
    const uint4* from = pools.src[blockIdx.y] + (int64_t)s * vecs_per_block;
    uint4* to = pools.dst[blockIdx.y] + (int64_t)d * vecs_per_block;
    int64_t i = threadIdx.x;
    for (; i + 3 * kThreads < vecs_per_block; i += 4 * kThreads) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldcs(from + i + u * kThreads);
#pragma unroll
        for (int u = 0; u < 4; ++u) __stcs(to + i + u * kThreads, v[u]);
    }
    for (; i < vecs_per_block; i += kThreads) __stcs(to + i, __ldcs(from + i));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

PA_API pa_status pa_reshape_and_cache(const void* k_new, const void* v_new,
                                      const int64_t* slot_mapping, int32_t T, void* k_cache,
                                      void* v_cache, int32_t num_blocks, int32_t block_size,
                                      int32_t Hkv, int32_t d, pa_dtype dtype, void* stream) {
    if (T < 0 || num_blocks < 0 || block_size <= 0 || Hkv <= 0 || d <= 0) return PA_ERR_INVALID;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if ((Hkv * d * 2) % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (T == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID;
    unsigned int* err = pa::device_error_word();
    const int sms = pa::device_sm_count();
    if (!err || !sms) return PA_ERR_CUDA;
    const int32_t vecs = Hkv * d * 2 / 16;
    const int64_t total = (int64_t)T * vecs;
    int64_t blocks = (total + kThreads - 1) / kThreads;
    if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
    reshape_and_cache_kernel<<<(unsigned)blocks, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping, T, vecs,
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
        (int64_t)num_blocks * block_size, err);
    return pa::cuda_status(cudaGetLastError());
}

}  // extern "C"

namespace {

template <bool kInt8>
pa_status reshape_and_cache_q8(const void* k_new, const void* v_new, const int64_t* slot_mapping,
                               int32_t T, void* k_cache, void* v_cache, float* k_scale,
                               float* v_scale, int32_t num_blocks, int32_t block_size, int32_t Hkv,
                               int32_t d, pa_dtype dtype, void* stream) {
    if (T < 0 || num_blocks < 0 || block_size <= 0 || Hkv <= 0) return PA_ERR_INVALID;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (d != 128) return PA_ERR_UNSUPPORTED;
    if (T == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
        return PA_ERR_INVALID;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
        return PA_ERR_INVALID;
    unsigned int* err = pa::device_error_word();
    const int sms = pa::device_sm_count();
    if (!err || !sms) return PA_ERR_CUDA;
    const int64_t warps = (int64_t)T * Hkv;
    int64_t blocks = (warps * 32 + kThreads - 1) / kThreads;
    if (blocks > (int64_t)sms * 16) blocks = (int64_t)sms * 16;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t slots = (int64_t)num_blocks * block_size;
    if (dtype == PA_BF16)
        reshape_and_cache_q8_kernel<__nv_bfloat16, kInt8><<<(unsigned)blocks, kThreads, 0, st>>>(
            static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new),
            slot_mapping, T, Hkv, block_size, static_cast<uint32_t*>(k_cache),
            static_cast<uint32_t*>(v_cache), k_scale, v_scale, slots, err);
    else
        reshape_and_cache_q8_kernel<__half, kInt8><<<(unsigned)blocks, kThreads, 0, st>>>(
            static_cast<const __half*>(k_new), static_cast<const __half*>(v_new), slot_mapping, T,
            Hkv, block_size, static_cast<uint32_t*>(k_cache), static_cast<uint32_t*>(v_cache),
            k_scale, v_scale, slots, err);
    return pa::cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" {

PA_API pa_status pa_reshape_and_cache_fp8(const void* k_new, const void* v_new,
                                          const int64_t* slot_mapping, int32_t T, void* k_cache,
                                          void* v_cache, float* k_scale, float* v_scale,
                                          int32_t num_blocks, int32_t block_size, int32_t Hkv,
                                          int32_t d, pa_dtype dtype, void* stream) {
    return reshape_and_cache_q8<false>(k_new, v_new, slot_mapping, T, k_cache, v_cache, k_scale,
                                       v_scale, num_blocks, block_size, Hkv, d, dtype, stream);
}

PA_API pa_status pa_reshape_and_cache_int8(const void* k_new, const void* v_new,
                                           const int64_t* slot_mapping, int32_t T, void* k_cache,
                                           void* v_cache, float* k_scale, float* v_scale,
                                           int32_t num_blocks, int32_t block_size, int32_t Hkv,
                                           int32_t d, pa_dtype dtype, void* stream) {
    return reshape_and_cache_q8<true>(k_new, v_new, slot_mapping, T, k_cache, v_cache, k_scale,
                                      v_scale, num_blocks, block_size, Hkv, d, dtype, stream);
}

PA_API pa_status pa_swap_blocks(const void* const* src_pools, void* const* dst_pools,
                                int32_t num_pools, const int32_t* pairs, int32_t num_pairs,
                                int64_t block_bytes, int32_t src_blocks, int32_t dst_blocks,
                                void* stream) {
    if (num_pools < 0 || num_pairs < 0 || block_bytes <= 0 || block_bytes % 16 != 0 ||
        src_blocks < 0 || dst_blocks < 0)
        return PA_ERR_INVALID;
    if (num_pools == 0 || num_pairs == 0) return PA_OK;
    if (!src_pools || !dst_pools || !pairs) return PA_ERR_INVALID;
    if (num_pairs > 0x7fffffff / 2) return PA_ERR_UNSUPPORTED;
    unsigned int* err = pa::device_error_word();
    if (!err) return PA_ERR_CUDA;
    for (int32_t l0 = 0; l0 < num_pools; l0 += kMaxSwapPools) {
        const int32_t nl = num_pools - l0 < kMaxSwapPools ? num_pools - l0 : kMaxSwapPools;
        SwapPools sp{};
        for (int32_t l = 0; l < nl; ++l) {
            const void* s = src_pools[l0 + l];
            void* d = dst_pools[l0 + l];
            if (!s || !d || !aligned16(s) || !aligned16(d)) return PA_ERR_INVALID;
            sp.src[l] = static_cast<const uint4*>(s);
            sp.dst[l] = static_cast<uint4*>(d);
        }
        swap_blocks_kernel<<<dim3((unsigned)num_pairs, (unsigned)nl), kThreads, 0,
                             static_cast<cudaStream_t>(stream)>>>(sp, pairs, block_bytes / 16,
                                                                   src_blocks, dst_blocks, err);
        if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

PA_API pa_status pa_copy_blocks(void* const* k_caches, void* const* v_caches,
                                int32_t num_layers, const int32_t* pairs, int32_t num_pairs,
                                int64_t block_bytes, int32_t num_blocks, void* stream) {
    if (num_layers < 0 || num_pairs < 0 || block_bytes <= 0 || block_bytes % 16 != 0 ||
        num_blocks < 0)
        return PA_ERR_INVALID;
    if (num_layers == 0 || num_pairs == 0) return PA_OK;
    if (!k_caches || !v_caches || !pairs) return PA_ERR_INVALID;
    if (num_pairs > 65535 * 64) return PA_ERR_UNSUPPORTED;
    unsigned int* err = pa::device_error_word();
    if (!err) return PA_ERR_CUDA;
    for (int32_t l0 = 0; l0 < num_layers; l0 += kMaxLayersPerLaunch) {
        const int32_t nl = num_layers - l0 < kMaxLayersPerLaunch ? num_layers - l0
                                                                 : kMaxLayersPerLaunch;
        LayerPtrs lp{};
        for (int32_t l = 0; l < nl; ++l) {
            if (!k_caches[l0 + l] || !v_caches[l0 + l] || !aligned16(k_caches[l0 + l]) ||
                !aligned16(v_caches[l0 + l]))
                return PA_ERR_INVALID;
            lp.k[l] = static_cast<uint4*>(k_caches[l0 + l]);
            lp.v[l] = static_cast<uint4*>(v_caches[l0 + l]);
        }
        copy_blocks_kernel<<<dim3((unsigned)num_pairs, (unsigned)nl), kThreads, 0,
                             static_cast<cudaStream_t>(stream)>>>(lp, pairs, block_bytes / 16,
                                                                   num_blocks, err);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    return PA_OK;
}

}  // extern "C"
