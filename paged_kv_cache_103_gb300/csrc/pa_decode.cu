// Paged decode attention for sm_103a (pa_decode).
//
// What it computes -- "LLM推理优化：vLLM PagedAttention深度解析与工程实践", section 二
// (attn = softmax(Q K^T / sqrt(d)) V), sections 3.1 and 4.1 (K/V in fixed-size
// physical blocks [num_blocks, block_size, heads, head_dim] reached through a
// per-sequence block table); "vLLM 深度拆解：当大模型推理学会「分页注意力」",
// section 1.1 (the new token's query attends to every cached K/V) and section
// 2.1 (logical -> physical block map); "LLM推理优化技术地图：从KV Cache到量化与
// 投机解码", section 2.3 (GQA: a group of query heads shares one KV head).
//
// The pages' A100 kernels -- one pass per block (v1) and partial accumulate
// then merge (v2), "LLM推理优化：vLLM PagedAttention深度解析与工程实践" section 4.1 --
// are prior art; this kernel keeps their two behaviours in one launch:
//
//  * Work is the list of (sequence i, KV head g, 32-token chunk c) triples in
//    that order.  Every CTA (one per SM, persistent) takes an equal contiguous
//    share of the list, so long and short contexts balance to one chunk.  A
//    (sequence, KV head) pair that falls inside one CTA is finished in one
//    pass; a pair split between CTAs leaves a partial (row max m, row sum l,
//    unnormalised output o) per CTA, and the last CTA to finish it -- found with
//    an atomic ticket, never by waiting -- merges them:
//        M = max m_p,  out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p.
//  * One producer warp walks the same list and streams K and V chunks into an
//    8-stage shared-memory ring with 2-D TMA tile loads (one 128-byte-wide box
//    per block, head and 64-column half; 128-byte swizzle), signalled through
//    mbarriers.  Table entries are read 32 at a time.  Blocks past a context's
//    end, and out-of-pool ids, are loaded from outside the tensor map and arrive
//    as zeros, so no address outside the cache is ever formed.
//  * Four consumer warps take the chunks round-robin.  Each warp computes the
//    logits of all G query heads of the group against 32 keys with m16n8k16
//    tensor-core MMAs (the G heads are the M rows, padded to 16), applies an
//    online softmax in base 2 and accumulates P V with MMAs, so each K/V byte is
//    read from HBM once for the whole group.  At a pair's end the four warps'
//    states are merged through shared memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "pa.h"
#include "pa_common.cuh"

namespace {

constexpr int kChunk = 32;           // tokens per pipeline stage
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kStages = 8;
constexpr int kMaxG = 16;            // query heads per KV head (MMA rows)
constexpr int kMaxBatch = 4096;
constexpr int kMaxCtas = 512;
constexpr uint64_t kWaitLimitNs = 1ull << 30;  // about one second
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
    const uint16_t* q;
    uint16_t* out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t* counters;  // [B * Hkv] arrival tickets of split pairs
    float* partials;    // [2 * kMaxCtas][slot_floats]
    unsigned int* err;
    int32_t max_blocks, B, H, Hkv, G, bs, num_blocks;
    float scale_log2;
};

template <int D>
struct Layout {
    static constexpr uint32_t kHalves = D / 64;
    static constexpr uint32_t kTileBytes = kChunk * D * 2;   // one of K or V
    static constexpr uint32_t kStageBytes = 2 * kTileBytes;
    static constexpr uint32_t kSlotFloats = 2 * kMaxG + kMaxG * D;
    static constexpr uint32_t kStagesOff = 0;
    static constexpr uint32_t kMergeOOff = kStagesOff + kStages * kStageBytes;
    static constexpr uint32_t kMergeMOff = kMergeOOff + kConsumerWarps * kMaxG * D * 4;
    static constexpr uint32_t kMergeLOff = kMergeMOff + kConsumerWarps * kMaxG * 4;
    static constexpr uint32_t kFacOff = kMergeLOff + kConsumerWarps * kMaxG * 4;
    static constexpr uint32_t kRowOff = kFacOff + kConsumerWarps * kMaxG * 4;
    static constexpr uint32_t kBarOff = kRowOff + 2 * kMaxG * 4;
    static constexpr uint32_t kFlagOff = kBarOff + 2 * kStages * 8;
    static constexpr uint32_t kScanOff = kFlagOff + 16;
    static constexpr uint32_t kPrefixOff = kScanOff + 8 * 8;
    static constexpr size_t bytes(int B) { return 1024 + kPrefixOff + (size_t)(B + 1) * 8; }
};

struct Segment {
    int32_t i, g, c0, len, nc;
    int64_t a;  // flattened index of the pair's first chunk
};

__device__ __forceinline__ int32_t clamp_len(int32_t n, int32_t cap) {
    return n < 0 ? 0 : (n > cap ? cap : n);
}

// Finds the pair containing flattened chunk `pos` (pos < prefix[B]).
__device__ __forceinline__ Segment find_segment(const int64_t* prefix, int32_t B, int32_t Hkv,
                                                int64_t pos, int64_t hi) {
    int32_t lo_i = 0, hi_i = B;  // largest i with prefix[i] <= pos
    while (hi_i - lo_i > 1) {
        const int32_t mid = (lo_i + hi_i) >> 1;
        if (prefix[mid] <= pos) lo_i = mid; else hi_i = mid;
    }
    Segment s;
    s.i = lo_i;
    s.nc = (int32_t)((prefix[lo_i + 1] - prefix[lo_i]) / Hkv);
    const int64_t local = pos - prefix[lo_i];
    s.g = (int32_t)(local / s.nc);
    s.c0 = (int32_t)(local - (int64_t)s.g * s.nc);
    s.a = prefix[lo_i] + (int64_t)s.g * s.nc;
    const int64_t rest = s.nc - s.c0;
    s.len = (int32_t)(hi - pos < rest ? hi - pos : rest);
    return s;
}

// First flattened chunk of CTA c when W chunks are split over C CTAs.
__device__ __forceinline__ int64_t cta_begin(int64_t c, int64_t W, int64_t C) {
    return c * W / C;
}

// Shared-memory byte offset of 16-byte column `chunk` of row `row` in a
// 128-byte-swizzled half tile (1024-byte aligned).
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk) {
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__device__ __forceinline__ uint32_t ld_u32(const uint16_t* p) {
    return __ldg(reinterpret_cast<const unsigned int*>(p));
}

template <bool kBF16>
__device__ __forceinline__ uint32_t pack_out(float a, float b) {
    return pa::pack2<kBF16>(a, b);
}

template <int D, bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
    using L = Layout<D>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* stages = smem + L::kStagesOff;
    float* merge_o = reinterpret_cast<float*>(smem + L::kMergeOOff);  // [W][16][D]
    float* merge_m = reinterpret_cast<float*>(smem + L::kMergeMOff);  // [W][16]
    float* merge_l = reinterpret_cast<float*>(smem + L::kMergeLOff);  // [W][16]
    float* fac = reinterpret_cast<float*>(smem + L::kFacOff);         // [W][16]
    float* rowinfo = reinterpret_cast<float*>(smem + L::kRowOff);     // M[16], 1/L or L [16]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
    uint64_t* empty = full + kStages;
    int* flags = reinterpret_cast<int*>(smem + L::kFlagOff);
    int64_t* scan = reinterpret_cast<int64_t*>(smem + L::kScanOff);
    int64_t* prefix = reinterpret_cast<int64_t*>(smem + L::kPrefixOff);  // [B + 1]

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int32_t B = p.B, Hkv = p.Hkv, G = p.G, bs = p.bs;
    const int32_t max_len = p.max_blocks * bs;

    // ---- prefix of chunk counts: prefix[i] = Hkv * sum_{i' < i} ceil(n_i' / 32)
    {
        const int per = (B + kThreads - 1) / kThreads;
        const int beg = min(tid * per, B), end = min(beg + per, B);
        int64_t local = 0;
        for (int i = beg; i < end; ++i) {
            const int32_t raw = __ldg(p.context_lens + i);
            if (blockIdx.x == 0) {
                if (raw < 0) pa::raise_error(p.err, PA_DEVERR_CONTEXT);
                if (raw > max_len) pa::raise_error(p.err, PA_DEVERR_TABLE_WIDTH);
            }
            local += (clamp_len(raw, max_len) + kChunk - 1) / kChunk;
        }
        int64_t x = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) scan[warp] = x;
        if (tid == 0) {
            for (int s = 0; s < kStages; ++s) {
                pa::mbar_init(&full[s], 1);
                pa::mbar_init(&empty[s], 1);
            }
            pa::fence_barrier_init();
        }
        __syncthreads();
        int64_t run = x - local;
        for (int w = 0; w < warp; ++w) run += scan[w];
        for (int i = beg; i < end; ++i) {
            prefix[i] = run * Hkv;
            run += (clamp_len(__ldg(p.context_lens + i), max_len) + kChunk - 1) / kChunk;
        }
        if (tid == 0) {
            int64_t total = 0;
            for (int w = 0; w < kThreads / 32; ++w) total += scan[w];
            prefix[B] = total * Hkv;
        }
        __syncthreads();
    }

    // ---- zero rows of empty contexts
    for (int32_t i = blockIdx.x; i < B; i += gridDim.x) {
        if (prefix[i + 1] != prefix[i]) continue;
        uint4* row = reinterpret_cast<uint4*>(p.out + (int64_t)i * p.H * D);
        for (int v = tid; v < p.H * D / 8; v += kThreads) row[v] = make_uint4(0, 0, 0, 0);
    }

    const int64_t W = prefix[B];
    const int64_t C = W < (int64_t)gridDim.x ? W : (int64_t)gridDim.x;
    if ((int64_t)blockIdx.x >= C) return;
    const int64_t lo = cta_begin(blockIdx.x, W, C);
    const int64_t hi = cta_begin(blockIdx.x + 1, W, C);

    if (warp == kConsumerWarps) {
        // =========================== producer warp ===========================
        if (lane == 0) {
            pa::prefetch_tensormap(&kmap);
            pa::prefetch_tensormap(&vmap);
        }
        const uint64_t policy = pa::l2_policy_evict_first();
        const int bpc = kChunk / bs;  // blocks per chunk
        const int32_t oob_row = p.num_blocks * bs;
        int64_t k = 0;  // chunks issued so far
        bool dead = false;
        for (int64_t pos = lo; pos < hi && !dead;) {
            const Segment s = find_segment(prefix, B, Hkv, pos, hi);
            const int32_t n = clamp_len(__ldg(p.context_lens + s.i), max_len);
            const int32_t nb = (n + bs - 1) / bs;
            const int32_t* trow = p.block_tables + (int64_t)s.i * p.max_blocks;
            int32_t wbase = -1, went = -1;
            for (int32_t t = 0; t < s.len; ++t, ++k) {
                const int32_t j0 = (s.c0 + t) * bpc;
                if (wbase < 0 || j0 + bpc > wbase + 32) {
                    wbase = j0;
                    const int32_t jj = wbase + lane;
                    went = jj < nb ? __ldg(trow + jj) : -1;
                }
                const int stage = (int)(k % kStages);
                if (k >= kStages) {
                    const uint32_t par = (uint32_t)((k / kStages - 1) & 1);
                    if (!__all_sync(0xffffffffu, pa::mbar_wait(&empty[stage], par, kWaitLimitNs))) {
                        dead = true;
                        if (lane == 0) pa::raise_error(p.err, PA_DEVERR_TIMEOUT);
                        break;
                    }
                }
                unsigned char* kt = stages + stage * L::kStageBytes;
                unsigned char* vt = kt + L::kTileBytes;
                if (lane == 0) pa::mbar_arrive_expect_tx(&full[stage], L::kStageBytes);
                for (int b = 0; b < bpc; ++b) {
                    const int32_t jj = j0 + b;
                    const int32_t blk = __shfl_sync(0xffffffffu, went, (jj - wbase) & 31);
                    bool ok = jj < nb;
                    if (ok && (blk < 0 || blk >= p.num_blocks)) {
                        ok = false;
                        if (lane == 0) pa::raise_error(p.err, PA_DEVERR_BLOCK_ID);
                    }
                    const int32_t y = ok ? blk * bs : oob_row;
                    if (lane == 0) {
#pragma unroll
                        for (uint32_t h = 0; h < L::kHalves; ++h) {
                            const uint32_t off = h * (kChunk * 128) + (uint32_t)b * bs * 128;
                            const int32_t x = s.g * D + (int32_t)h * 64;
                            pa::tma_load_2d(kt + off, &kmap, &full[stage], x, y, policy);
                            pa::tma_load_2d(vt + off, &vmap, &full[stage], x, y, policy);
                        }
                    }
                }
            }
            pos += s.len;
        }
        // Every issued load has landed before the CTA may exit.
        const int64_t issued = k;
        for (int s = 0; s < kStages && s < issued; ++s) {
            const int64_t last_use = (issued - 1 - s) / kStages;
            pa::mbar_wait(&full[s], (uint32_t)(last_use & 1), kWaitLimitNs);
        }
        return;
    }

    // ============================= consumer warps =============================
    const int r0 = lane >> 2;        // MMA row (query head in group) of c0/c1
    const int r1 = r0 + 8;           // row of c2/c3
    const int cq = 2 * (lane & 3);   // column pair inside an 8-wide tile
    const uint32_t stages_addr = pa::smem_addr(stages);
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix / row this lane addresses
    int64_t k = 0;
    bool dead = false;

    for (int64_t pos = lo; pos < hi;) {
        const Segment s = find_segment(prefix, B, Hkv, pos, hi);
        const int32_t n = clamp_len(__ldg(p.context_lens + s.i), max_len);
        const int32_t head0 = s.g * G;

        uint32_t qa[D / 16][4];
        {
            const uint16_t* q0 = p.q + ((int64_t)s.i * p.H + head0 + r0) * D;
            const uint16_t* q1 = p.q + ((int64_t)s.i * p.H + head0 + r1) * D;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int col = ks * 16 + cq;
                qa[ks][0] = r0 < G ? ld_u32(q0 + col) : 0u;
                qa[ks][1] = r1 < G ? ld_u32(q1 + col) : 0u;
                qa[ks][2] = r0 < G ? ld_u32(q0 + col + 8) : 0u;
                qa[ks][3] = r1 < G ? ld_u32(q1 + col + 8) : 0u;
            }
        }
        float m_run[2] = {-INFINITY, -INFINITY};
        float l_run[2] = {0.f, 0.f};
        float o[D / 8][4];
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;

        for (int32_t t = warp; t < s.len; t += kConsumerWarps) {
            const int64_t kk = k + t;
            const int stage = (int)(kk % kStages);
            const bool ready =
                dead || pa::mbar_wait(&full[stage], (uint32_t)((kk / kStages) & 1), kWaitLimitNs);
            if (!__all_sync(0xffffffffu, ready)) {
                dead = true;
                if (lane == 0) pa::raise_error(p.err, PA_DEVERR_TIMEOUT);
            }
            if (!dead) {
                const int32_t tok0 = (s.c0 + t) * kChunk;
                const int32_t valid = n - tok0 < kChunk ? n - tok0 : kChunk;
                const uint32_t kt = stages_addr + stage * L::kStageBytes;
                const uint32_t vt = kt + L::kTileBytes;
                if (valid < kChunk) {
                    // Rows past the context may hold anything (even NaN): zero
                    // them in V so that 0-weight rows add exactly nothing.
                    uint4* vrow = reinterpret_cast<uint4*>(stages + stage * L::kStageBytes +
                                                           L::kTileBytes);
                    const int per_half = (kChunk - valid) * 8;
                    for (int e = lane; e < per_half * (int)L::kHalves; e += 32) {
                        const int h = e / per_half, rem = e - h * per_half;
                        vrow[(h * kChunk * 128 + (valid + rem / 8) * 128) / 16 + rem % 8] =
                            make_uint4(0, 0, 0, 0);
                    }
                    pa::fence_proxy_async_smem();
                    __syncwarp();
                }

                // S = Q K^T for 32 keys: 4 n-tiles of 8 keys.
                float sc[4][4];
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t half_base = kt + (uint32_t)(ks >> 2) * (kChunk * 128);
                    const uint32_t chunk = (uint32_t)((ks & 3) * 2 + (mi & 1));
#pragma unroll
                    for (int pp = 0; pp < 2; ++pp) {
                        const uint32_t row = (uint32_t)(pp * 16 + (mi >> 1) * 8 + rr);
                        uint32_t b0, b1, b2, b3;
                        pa::ldsm_x4(half_base + swz(row, chunk), b0, b1, b2, b3);
                        pa::mma_16816<kBF16>(sc[2 * pp], qa[ks], b0, b1);
                        pa::mma_16816<kBF16>(sc[2 * pp + 1], qa[ks], b2, b3);
                    }
                }

                // Online softmax in base 2 (rows r0 and r1).
                float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int tok = nt * 8 + cq + (e & 1);
                        const float x = tok < valid ? sc[nt][e] * p.scale_log2 : -INFINITY;
                        sc[nt][e] = x;
                        mx[e >> 1] = fmaxf(mx[e >> 1], x);
                    }
                }
                float alpha[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
                    mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
                    const float m_new = fmaxf(m_run[h], mx[h]);
                    alpha[h] = pa::fast_exp2(m_run[h] - m_new);
                    m_run[h] = m_new;
                    l_run[h] *= alpha[h];
                }
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float pe = pa::fast_exp2(sc[nt][e] - m_run[e >> 1]);
                        sc[nt][e] = pe;
                        l_run[e >> 1] += pe;
                    }
                }
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt) {
                    o[nt][0] *= alpha[0];
                    o[nt][1] *= alpha[0];
                    o[nt][2] *= alpha[1];
                    o[nt][3] *= alpha[1];
                }

                // O += P V: k = 32 keys in two 16-key steps, n = D in 8-wide tiles.
#pragma unroll
                for (int ks2 = 0; ks2 < 2; ++ks2) {
                    uint32_t pa_frag[4];
                    pa_frag[0] = pa::pack2<kBF16>(sc[2 * ks2][0], sc[2 * ks2][1]);
                    pa_frag[1] = pa::pack2<kBF16>(sc[2 * ks2][2], sc[2 * ks2][3]);
                    pa_frag[2] = pa::pack2<kBF16>(sc[2 * ks2 + 1][0], sc[2 * ks2 + 1][1]);
                    pa_frag[3] = pa::pack2<kBF16>(sc[2 * ks2 + 1][2], sc[2 * ks2 + 1][3]);
                    const uint32_t row = (uint32_t)(ks2 * 16 + (mi & 1) * 8 + rr);
#pragma unroll
                    for (int dt = 0; dt < D / 16; ++dt) {
                        const int dim = dt * 16 + (mi >> 1) * 8;
                        const uint32_t addr = vt + (uint32_t)(dim >> 6) * (kChunk * 128) +
                                              swz(row, (uint32_t)((dim & 63) >> 3));
                        uint32_t b0, b1, b2, b3;
                        pa::ldsm_x4_trans(addr, b0, b1, b2, b3);
                        pa::mma_16816<kBF16>(o[2 * dt], pa_frag, b0, b1);
                        pa::mma_16816<kBF16>(o[2 * dt + 1], pa_frag, b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(&empty[stage]);
        }
        k += s.len;

        // ---- merge the four warps' states for this pair
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
            l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
        }
        if ((lane & 3) == 0) {
            if (r0 < G) {
                merge_m[warp * kMaxG + r0] = m_run[0];
                merge_l[warp * kMaxG + r0] = l_run[0];
            }
            if (r1 < G) {
                merge_m[warp * kMaxG + r1] = m_run[1];
                merge_l[warp * kMaxG + r1] = l_run[1];
            }
        }
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
            const int dim = nt * 8 + cq;
            if (r0 < G)
                *reinterpret_cast<float2*>(&merge_o[(warp * kMaxG + r0) * D + dim]) =
                    make_float2(o[nt][0], o[nt][1]);
            if (r1 < G)
                *reinterpret_cast<float2*>(&merge_o[(warp * kMaxG + r1) * D + dim]) =
                    make_float2(o[nt][2], o[nt][3]);
        }
        pa::named_barrier_sync(1, kConsumerThreads);

        const bool whole = (s.c0 == 0 && s.len == s.nc);
        if (tid < G) {
            float M = -INFINITY;
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, merge_m[w * kMaxG + tid]);
            float Lsum = 0.f;
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float f = pa::fast_exp2(merge_m[w * kMaxG + tid] - M);
                fac[w * kMaxG + tid] = f;
                Lsum += f * merge_l[w * kMaxG + tid];
            }
            rowinfo[tid] = M;
            rowinfo[kMaxG + tid] = whole ? 1.f / Lsum : Lsum;
        }
        pa::named_barrier_sync(1, kConsumerThreads);

        if (whole) {
            for (int e = tid; e < G * D / 2; e += kConsumerThreads) {
                const int r = e / (D / 2), dp = (e - r * (D / 2)) * 2;
                float v0 = 0.f, v1 = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float f = fac[w * kMaxG + r];
                    const float2 ov = *reinterpret_cast<const float2*>(
                        &merge_o[(w * kMaxG + r) * D + dp]);
                    v0 += f * ov.x;
                    v1 += f * ov.y;
                }
                const float inv = rowinfo[kMaxG + r];
                *reinterpret_cast<uint32_t*>(p.out + ((int64_t)s.i * p.H + head0 + r) * D + dp) =
                    pack_out<kBF16>(v0 * inv, v1 * inv);
            }
        } else {
            // Partial result of this CTA for a pair split between CTAs.
            const int64_t c_first = (((s.a + 1) * C) - 1) / W;
            const int64_t c_last = (((s.a + s.nc) * C) - 1) / W;
            const int64_t slot = lo >= s.a ? 2 * (int64_t)blockIdx.x : 2 * (int64_t)blockIdx.x + 1;
            float* ps = p.partials + slot * L::kSlotFloats;
            if (tid < G) {
                ps[tid] = rowinfo[tid];
                ps[kMaxG + tid] = rowinfo[kMaxG + tid];
            }
            for (int e = tid; e < G * D; e += kConsumerThreads) {
                const int r = e / D, dim = e - r * D;
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w)
                    v += fac[w * kMaxG + r] * merge_o[(w * kMaxG + r) * D + dim];
                ps[2 * kMaxG + r * D + dim] = v;
            }
            __threadfence();
            pa::named_barrier_sync(1, kConsumerThreads);
            if (tid == 0) {
                int32_t* ctr = p.counters + (int64_t)s.i * Hkv + s.g;
                const int prev = atomicAdd(ctr, 1);
                const int last = prev == (int)(c_last - c_first);
                if (last) atomicExch(ctr, 0);
                flags[1] = last;
            }
            pa::named_barrier_sync(1, kConsumerThreads);
            if (flags[1]) {
                __threadfence();
                if (tid < G) {
                    float M = -INFINITY;
                    for (int64_t c = c_first; c <= c_last; ++c) {
                        const int64_t sl = cta_begin(c, W, C) >= s.a ? 2 * c : 2 * c + 1;
                        M = fmaxf(M, __ldcg(p.partials + sl * L::kSlotFloats + tid));
                    }
                    float Lsum = 0.f;
                    for (int64_t c = c_first; c <= c_last; ++c) {
                        const int64_t sl = cta_begin(c, W, C) >= s.a ? 2 * c : 2 * c + 1;
                        const float* q = p.partials + sl * L::kSlotFloats;
                        Lsum += pa::fast_exp2(__ldcg(q + tid) - M) * __ldcg(q + kMaxG + tid);
                    }
                    rowinfo[tid] = M;
                    rowinfo[kMaxG + tid] = 1.f / Lsum;
                }
                pa::named_barrier_sync(1, kConsumerThreads);
                for (int e = tid; e < G * D / 2; e += kConsumerThreads) {
                    const int r = e / (D / 2), dp = (e - r * (D / 2)) * 2;
                    const float M = rowinfo[r];
                    float v0 = 0.f, v1 = 0.f;
                    for (int64_t c = c_first; c <= c_last; ++c) {
                        const int64_t sl = cta_begin(c, W, C) >= s.a ? 2 * c : 2 * c + 1;
                        const float* q = p.partials + sl * L::kSlotFloats;
                        const float f = pa::fast_exp2(__ldcg(q + r) - M);
                        const float2 ov = __ldcg(
                            reinterpret_cast<const float2*>(q + 2 * kMaxG + r * D + dp));
                        v0 += f * ov.x;
                        v1 += f * ov.y;
                    }
                    const float inv = rowinfo[kMaxG + r];
                    *reinterpret_cast<uint32_t*>(p.out + ((int64_t)s.i * p.H + head0 + r) * D +
                                                 dp) = pack_out<kBF16>(v0 * inv, v1 * inv);
                }
            }
        }
        pa::named_barrier_sync(1, kConsumerThreads);
        pos += s.len;
    }
}

// ---- host side -----------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// A 2-D view [num_blocks * block_size rows][Hkv * d columns] of one cache, read
// in boxes of 64 columns x block_size rows with 128-byte swizzle.
bool encode_cache_map(CUtensorMap* map, const void* base, int32_t rows, int32_t cols,
                      int32_t box_rows, pa_dtype dtype) {
    auto encode = get_encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = encode(
        map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
        2, const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

size_t slot_floats(int32_t d) { return 2 * kMaxG + (size_t)kMaxG * d; }

size_t counters_bytes(int32_t B, int32_t H) {
    return (((size_t)B * H * sizeof(int32_t)) + 255) & ~size_t(255);
}

template <int D, bool kBF16>
pa_status launch(const CUtensorMap& km, const CUtensorMap& vm, const DecodeParams& prm, int grid,
                 cudaStream_t stream) {
    auto kern = paged_decode_kernel<D, kBF16>;
    const size_t smem = Layout<D>::bytes(prm.B);
    static std::mutex mu;
    static size_t configured = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (smem > configured) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)Layout<D>::bytes(kMaxBatch)) != cudaSuccess)
                return PA_ERR_CUDA;
            configured = Layout<D>::bytes(kMaxBatch);
        }
    }
    kern<<<grid, kThreads, smem, stream>>>(km, vm, prm);
    return pa::cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" {

PA_API size_t pa_decode_workspace_size(int32_t B, int32_t H, int32_t d) {
    if (B < 0 || H <= 0 || (d != 64 && d != 128)) return 0;
    return counters_bytes(B, H) + 2 * (size_t)kMaxCtas * slot_floats(d) * sizeof(float);
}

PA_API int32_t pa_decode_grid_size(void) {
    const int sms = pa::device_sm_count();
    return sms > kMaxCtas ? kMaxCtas : sms;
}

PA_API pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int32_t max_blocks,
                           const int32_t* context_lens, int32_t max_context_len, int32_t B,
                           int32_t H, int32_t Hkv, int32_t d, int32_t block_size,
                           int32_t num_blocks, float scale, pa_dtype dtype, void* out,
                           void* workspace, size_t ws_bytes, void* stream) {
    if (B < 0 || H <= 0 || Hkv <= 0 || max_blocks <= 0 || num_blocks <= 0 ||
        max_context_len < 0 || !std::isfinite(scale))
        return PA_ERR_INVALID;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (H % Hkv != 0 || H / Hkv > kMaxG) return PA_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return PA_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
    if (B > kMaxBatch) return PA_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
    if (B == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace)
        return PA_ERR_INVALID;
    if (ws_bytes < pa_decode_workspace_size(B, H, d)) return PA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15u)
        return PA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(q) & 3u) || (reinterpret_cast<uintptr_t>(out) & 15u))
        return PA_ERR_INVALID;
    // Flattened chunk indices must stay far from 64-bit overflow in c * W.
    const int64_t chunks = (int64_t)B * Hkv * (((int64_t)max_context_len + kChunk - 1) / kChunk);
    if (chunks > ((int64_t)1 << 40)) return PA_ERR_UNSUPPORTED;

    unsigned int* err = pa::device_error_word();
    const int grid = pa_decode_grid_size();
    if (!err || grid <= 0) return PA_ERR_CUDA;

    CUtensorMap km, vm;
    const int32_t rows = num_blocks * block_size, cols = Hkv * d;
    if (!encode_cache_map(&km, k_cache, rows, cols, block_size, dtype) ||
        !encode_cache_map(&vm, v_cache, rows, cols, block_size, dtype))
        return PA_ERR_CUDA;

    DecodeParams prm;
    prm.q = static_cast<const uint16_t*>(q);
    prm.out = static_cast<uint16_t*>(out);
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.counters = static_cast<int32_t*>(workspace);
    prm.partials = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) +
                                            counters_bytes(B, H));
    prm.err = err;
    prm.max_blocks = max_blocks;
    prm.B = B;
    prm.H = H;
    prm.Hkv = Hkv;
    prm.G = H / Hkv;
    prm.bs = block_size;
    prm.num_blocks = num_blocks;
    prm.scale_log2 = scale * kLog2e;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (d == 128)
        return dtype == PA_BF16 ? launch<128, true>(km, vm, prm, grid, st)
                                : launch<128, false>(km, vm, prm, grid, st);
    return dtype == PA_BF16 ? launch<64, true>(km, vm, prm, grid, st)
                            : launch<64, false>(km, vm, prm, grid, st);
}

}  // extern "C"
