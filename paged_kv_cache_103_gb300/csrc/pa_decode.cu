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
//    that order.  The persistent CTAs (two per SM) each take an equal
//    contiguous share of the list, so long and short contexts balance to one
//    chunk.  A (sequence, KV head) pair inside one CTA's share is finished in
//    one pass; a pair split between CTAs leaves a partial (row max m, row sum
//    l, unnormalised output o) per CTA, and the last CTA to finish it -- found
//    with an atomic ticket, never by waiting -- merges them:
//        M = max m_p,  out = sum_p 2^(m_p - M) o_p / sum_p 2^(m_p - M) l_p.
//  * Two producer warps (even and odd chunks) walk the same list and stream K
//    and V chunks into a shared-memory ring with 3-D TMA tile loads: one box per
//    block and tensor (block_size rows x head_dim, 128-byte swizzle), all of a
//    chunk's boxes issued by one lane, completion counted on the stage's
//    mbarrier.  The table is read 32 entries at a time, one window and one
//    pair ahead of use.  Blocks past a context's end, and out-of-pool ids, are
//    loaded from outside the tensor map and arrive as zeros, so no address
//    outside the cache is ever formed.
//  * Four consumer warps take the chunks; stage s always goes to warp s % 4.  A warp computes
//    S^T = K Q^T for 32 keys with m16n8k16 tensor-core MMAs (keys are the M
//    rows, the group's G query heads the N columns), runs the online softmax
//    in base 2 per head, transposes P in registers (movmatrix) and accumulates
//    O^T = V^T P^T with MMAs -- each K/V byte is read from HBM once for the
//    whole GQA group.  At a pair's end the warps' states merge in shared memory.
//
// The same kernel reads an FP8 cache (pa_decode_fp8; "LLM推理优化技术地图：从KV
// Cache到量化与投机解码", section 4.3, KV cache quantisation): E4M3 codes
// [num_blocks][block_size][Hkv][128] plus one fp32 scale per (token, KV head),
// laid out [num_blocks][Hkv][block_size].  A stage then holds 32 code rows of
// 128 bytes per tensor and the chunk's 2 x 32 scales (their own TMA boxes).
// Both products run as f16 MMAs: codes widen to f16 exactly; a bf16 query is
// scaled by a power of two into f16 range (the factor leaves the scores through
// the score multiplier); the V scale is folded into P, and P is kept in f16
// range by a running power-of-two factor on the accumulator.  Because the
// head-dim and key orders of an MMA are free, the code bytes are read in
// permuted orders that make each lane's loads contiguous and conflict-free,
// and the output rows are put back in order when the state is deposited.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "pa.h"
#include "pa_common.cuh"

namespace {

constexpr int kChunk = 32;           // tokens per pipeline stage (16 or 32)
constexpr int kKeyTiles = kChunk / 16;  // 16-key MMA tiles per chunk
constexpr int kConsumerWarps = 4;
constexpr int kConsumerThreads = kConsumerWarps * 32;
// Producer warps: two for a 16-bit cache (even and odd chunks); one per
// consumer warp for an 8-bit cache, each refilling only that consumer's
// stages, with the registers rebalanced between the two warpgroups.
__host__ __device__ constexpr int producer_warps(bool fp8) { return fp8 ? 4 : 2; }
__host__ __device__ constexpr int cta_threads(bool fp8) {
    return (kConsumerWarps + producer_warps(fp8)) * 32;
}
// 8-bit register split: launched at 128 registers a thread (256 threads, two
// CTAs per SM); the producer warpgroup gives back down to 72 and the consumer
// warpgroup takes 184: 128 x 72 + 128 x 184 = 256 x 128.
constexpr int kQ8LaunchRegs = 128;
constexpr int kQ8ProducerRegs = 72;
constexpr int kQ8ConsumerRegs = 184;
static_assert(128 * kQ8ProducerRegs + 128 * kQ8ConsumerRegs == 256 * kQ8LaunchRegs,
              "8-bit register split");
constexpr int kCtasPerSm = 2;
constexpr int kMaxStages = 16;
constexpr int kMaxG = 16;            // query heads per KV head (two 8-wide MMA tiles)
constexpr int kMaxBatch = 4096;
constexpr int kMaxCtas = 512;
constexpr int kMinChunksPerCta = 4;
constexpr uint32_t kSmemBudget = 113 * 1024;   // dynamic shared memory per CTA (two per SM)
constexpr uint64_t kWaitLimitNs = 1ull << 30;  // about one second
constexpr float kLog2e = 1.4426950408889634f;
// FP8 stages: per tensor one 128-byte scale slot per block of the chunk (one
// TMA box of block_size fp32 each).
constexpr uint32_t kScaleSlotBytes = 128;

struct DecodeParams {
    const uint16_t* q;
    uint16_t* out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t* counters;  // [B * Hkv] arrival tickets of split pairs
    float* partials;    // [2 * kMaxCtas][slot_floats]
    unsigned int* err;
    // Hkv and G as the kernel sees them: a KV head with more than kMaxG query
    // heads is split into `subs` pairs of kMaxG heads each, pair g reading KV
    // head g / subs (query heads g * G .. g * G + G - 1 either way).
    int32_t max_blocks, B, H, Hkv, G, bs, num_blocks, stages, subs;
    int32_t len_hint;   // the caller's max_context_len: a guess of every context's length
    float scale_log2;
};

// Dynamic shared-memory carve-up; the same function runs on host and device.
struct Layout {
    uint32_t stage_bytes, scale_stage, scales, merge_o, merge_m, merge_l, rowinfo, bars, flags, scan, prefix, total;
};

// Merge slots (two when the warps merge asynchronously, pairs alternating;
// one when they merge together): each holds every consumer warp's
// unnormalised output [W][G][D], row maxima [W][16] and row sums [W][16].
__host__ __device__ inline Layout make_layout(int D, int G, int B, int stages, int slots,
                                              bool fp8, int bs) {
    Layout L;
    L.stage_bytes = 2u * kChunk * D * (fp8 ? 1 : 2);
    // fp8: [stages][K, V][blocks per chunk][32] fp32
    L.scale_stage = fp8 ? 2u * (kChunk / (bs < kChunk ? bs : kChunk)) * kScaleSlotBytes : 0u;
    L.scales = stages * L.stage_bytes;
    L.merge_o = L.scales + stages * L.scale_stage;                   // [slots][W][G][D] fp32
    L.merge_m = L.merge_o + slots * kConsumerWarps * G * D * 4;      // [slots][W][16]
    L.merge_l = L.merge_m + slots * kConsumerWarps * kMaxG * 4;      // [slots][W][16]
    L.rowinfo = L.merge_l + slots * kConsumerWarps * kMaxG * 4;      // [slots][2 + W][16]
    L.bars = L.rowinfo + slots * (2 + kConsumerWarps) * kMaxG * 4;   // full[], empty[]
    L.flags = L.bars + 2 * kMaxStages * 8;                           // count[2] free[2] flag[2]
    L.scan = L.flags + 32;
    L.prefix = L.scan + 32 * 4;                                      // [B + 1] int32
    L.total = 1024 + L.prefix + (uint32_t)(B + 1) * 4;               // + alignment slack
    return L;
}

struct Segment {
    int32_t i, g, c0, len, nc;
    int32_t a;  // flattened index of the pair's first chunk
};

__device__ __forceinline__ int32_t clamp_len(int32_t n, int32_t cap) {
    return n < 0 ? 0 : (n > cap ? cap : n);
}

// The pair containing flattened chunk `pos` (pos < prefix[B]), cut at `hi`.
__device__ __forceinline__ Segment find_segment(const int32_t* prefix, int32_t B, int32_t Hkv,
                                                int32_t pos, int32_t hi) {
    int32_t lo_i = 0, hi_i = B;  // largest i with prefix[i] <= pos
    while (hi_i - lo_i > 1) {
        const int32_t mid = (lo_i + hi_i) >> 1;
        if (prefix[mid] <= pos) lo_i = mid; else hi_i = mid;
    }
    Segment s;
    s.i = lo_i;
    s.nc = (prefix[lo_i + 1] - prefix[lo_i]) / Hkv;
    const int32_t local = pos - prefix[lo_i];
    s.g = local / s.nc;
    s.c0 = local - s.g * s.nc;
    s.a = prefix[lo_i] + s.g * s.nc;
    const int32_t rest = s.nc - s.c0;
    s.len = hi - pos < rest ? hi - pos : rest;
    return s;
}

// First flattened chunk of CTA c when W chunks are split over C CTAs.
__device__ __forceinline__ int32_t cta_begin(int64_t c, int64_t W, int64_t C) {
    return (int32_t)(c * W / C);
}

// Workspace slot of the partial that CTA c leaves for the pair starting at a:
// its first slot if the pair is where its share begins, else its second.
__device__ __forceinline__ int64_t partial_slot(int64_t c, int64_t W, int64_t C, int32_t a) {
    return cta_begin(c, W, C) >= a ? 2 * c : 2 * c + 1;
}

// Waits, for at most about limit_ns, until the shared-memory word holds
// `value`; returns false if the limit ran out.
__device__ __forceinline__ bool wait_flag(const int* flag, int value, uint64_t limit_ns) {
    const volatile int* f = flag;
    if (*f == value) return true;
    const uint64_t t0 = pa::global_timer_ns();
    for (;;) {
#pragma unroll 1
        for (int k = 0; k < 64; ++k)
            if (*f == value) return true;
        if (pa::global_timer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ uint32_t u4_word(const uint4& v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

__device__ __forceinline__ uint32_t ld_u32(const uint16_t* p) {
    return __ldg(reinterpret_cast<const unsigned int*>(p));
}

// A stage holds one chunk of K then one of V, each laid out [block][64-column
// half][block_size rows][128 bytes] with the TMA 128-byte swizzle (16-byte
// column c of row r stored at column c ^ (r & 7)).  Byte offset of (token t,
// half h, 16-byte column c) inside a tensor's chunk:
__device__ __forceinline__ uint32_t tile_offset(uint32_t t, uint32_t h, uint32_t c,
                                                uint32_t halves, uint32_t rows_shift) {
    const uint32_t b = t >> rows_shift, r = t & ((1u << rows_shift) - 1u);
    return ((((b * halves + h) << rows_shift) + r) << 7) + ((c ^ (t & 7u)) << 4);
}

// kFp8: the cache holds E4M3 codes with per-(token, KV head) scales (ksmap,
// vsmap); otherwise the cache has the dtype of q and the scale maps are unused.
// Four 8-bit codes as two f16x2 registers: E4M3, or INT8 (kInt8).
template <bool kInt8>
__device__ __forceinline__ void q8x4_to_f16(uint32_t x, uint32_t& lo, uint32_t& hi) {
    if constexpr (kInt8)
        pa::s8x4_to_f16(x, lo, hi);
    else
        pa::e4m3x4_to_f16(x, lo, hi);
}

template <int D, bool kBF16, int NT, bool kAsync, bool kFp8, bool kInt8>
__global__ void __launch_bounds__(cta_threads(kFp8), kCtasPerSm)
paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap,
                    const __grid_constant__ CUtensorMap ksmap,
                    const __grid_constant__ CUtensorMap vsmap, const DecodeParams p) {
    static_assert(!kFp8 || D == 128, "FP8 rows are one 128-byte swizzle row");
    constexpr int kProducerWarps = producer_warps(kFp8);
    constexpr int kThreads = cta_threads(kFp8);
    constexpr uint32_t kHalves = kFp8 ? 1 : D / 64;  // 128-byte pieces of a token row
    const int32_t B = p.B, Hkv = p.Hkv, G = p.G, bs = p.bs, S = p.stages;
    const Layout L = make_layout(D, G, B, S, kAsync ? 2 : 1, kFp8, bs);
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* merge_o = reinterpret_cast<float*>(smem + L.merge_o);
    float* merge_m = reinterpret_cast<float*>(smem + L.merge_m);
    float* merge_l = reinterpret_cast<float*>(smem + L.merge_l);
    float* rowinfo = reinterpret_cast<float*>(smem + L.rowinfo);  // per slot: M[16], 1/L[16]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + kMaxStages;
    int* slot_count = reinterpret_cast<int*>(smem + L.flags);      // arrivals per merge slot
    int* slot_free = slot_count + 2;  // a slot takes pair j once it holds the value j
    int* slot_flag = slot_count + 4;  // "this CTA is the pair's last" for the slot's merge
    int32_t* scan = reinterpret_cast<int32_t*>(smem + L.scan);
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + L.prefix);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int32_t max_len = p.max_blocks * bs;
    // Rows of one TMA box: a whole block, or a chunk-sized slice of a larger one.
    const uint32_t rows_shift = (uint32_t)(31 - __clz(bs < kChunk ? bs : kChunk));

    // ---- a producer's first table window, guessed before the lengths arrive:
    // were every context len_hint tokens long, this CTA's share would start at
    // chunk lo_g of sequence g_i.  The window is loaded now, in the shadow of
    // the length scan, and used only if the scan confirms the guess (batches
    // of equal lengths); otherwise it is read again after the scan.
    int32_t g_i = -1, g_wbase = -1, g_went = -1, g_wnext = -1;
    if (warp >= kConsumerWarps && p.len_hint > 0) {
        const int32_t nc = (min(p.len_hint, max_len) + kChunk - 1) / kChunk;
        const int64_t Wg = (int64_t)B * Hkv * nc;
        int64_t Cg = Wg / kMinChunksPerCta;
        if (Cg > (int64_t)gridDim.x) Cg = gridDim.x;
        if (Cg < 1) Cg = 1;
        if (nc > 0 && (int64_t)blockIdx.x < Cg) {
            const int32_t lo_g = cta_begin(blockIdx.x, Wg, Cg);
            g_i = lo_g / (Hkv * nc);
            const int32_t c0 = (lo_g - g_i * Hkv * nc) % nc;
            g_wbase = (c0 * kChunk) >> (31 - __clz(bs));
            const int32_t* trow = p.block_tables + (int64_t)g_i * p.max_blocks;
            const int32_t j = g_wbase + lane;
            g_went = j < p.max_blocks ? __ldg(trow + j) : -1;
            g_wnext = j + 32 < p.max_blocks ? __ldg(trow + j + 32) : -1;
            // ... and the K / V blocks of this producer's first chunk (chunk
            // c0 + prod of the guessed pair) are prefetched into L2, so that
            // the real loads after the scan find them there; a wrong guess only
            // costs the prefetch.  Block ids are checked as for a load.
            // Only when CTAs average four chunks or more: with a chunk or two
            // each, the real load follows the prefetch at once (measured slower).
            const int32_t prod = warp - kConsumerWarps;
            const int32_t cg = c0 + prod;
            if (cg < nc && Wg >= 4 * Cg) {
                const int bpc_g = kChunk >> rows_shift;
                const int32_t j0 = (cg * kChunk) >> (31 - __clz(bs));
                const int32_t kvh_g = ((lo_g - g_i * Hkv * nc) / nc) / p.subs;
                for (int b = 0; b < bpc_g; ++b) {
                    const int32_t e = __shfl_sync(0xffffffffu, g_went, (j0 - g_wbase + b) & 31);
                    if (lane == 0 && e >= 0 && e < p.num_blocks) {
                        pa::tma_prefetch_3d(&kmap, 0, e * bs, kvh_g * (int32_t)kHalves);
                        pa::tma_prefetch_3d(&vmap, 0, e * bs, kvh_g * (int32_t)kHalves);
                    }
                }
            }
        }
    }

    // ---- prefix of chunk counts: prefix[i] = Hkv * sum_{i' < i} ceil(n_i' / 32)
    {
        const int per = (B + kThreads - 1) / kThreads;
        const int beg = min(tid * per, B), end = min(beg + per, B);
        int32_t local = 0;
        for (int i = beg; i < end; ++i) {
            const int32_t raw = __ldg(p.context_lens + i);
            if (blockIdx.x == 0) {
                if (raw < 0) pa::raise_error(p.err, PA_DEVERR_CONTEXT);
                if (raw > max_len) pa::raise_error(p.err, PA_DEVERR_TABLE_WIDTH);
            }
            local += (clamp_len(raw, max_len) + kChunk - 1) / kChunk;
        }
        int32_t x = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) scan[warp] = x;
        if (tid == 0) {
            for (int s = 0; s < S; ++s) {
                pa::mbar_init(&full[s], 1);
                pa::mbar_init(&empty[s], 1);
            }
            pa::fence_barrier_init();
            slot_count[0] = slot_count[1] = 0;
            slot_free[0] = 0;
            slot_free[1] = 1;
        }
        __syncthreads();
        int32_t run = x - local;
        for (int w = 0; w < warp; ++w) run += scan[w];
        for (int i = beg; i < end; ++i) {
            prefix[i] = run * Hkv;
            run += (clamp_len(__ldg(p.context_lens + i), max_len) + kChunk - 1) / kChunk;
        }
        if (tid == 0) {
            int32_t total = 0;
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
    // CTAs in use: every one gets at least kMinChunksPerCta chunks, so short
    // batches are not cut into more partials than their size pays for.
    int64_t C = W / kMinChunksPerCta;
    if (C > (int64_t)gridDim.x) C = gridDim.x;
    if (C < 1) C = 1;
    if ((int64_t)blockIdx.x >= C) return;
    const int32_t lo = cta_begin(blockIdx.x, W, C);
    const int32_t hi = cta_begin(blockIdx.x + 1, W, C);

    if (warp >= kConsumerWarps) {
        // =========================== producer warps ===========================
        // 8-bit caches: the producer warpgroup gives registers back before
        // anything else (the consumers' increase waits for them).
        if constexpr (kFp8) pa::setmaxnreg_dec<kQ8ProducerRegs>();
        const int prod = warp - kConsumerWarps;  // issues the chunks k with k % kProducerWarps == prod
        if (lane == 0 && prod == 0) {
            pa::prefetch_tensormap(&kmap);
            pa::prefetch_tensormap(&vmap);
            if constexpr (kFp8) {
                pa::prefetch_tensormap(&ksmap);
                pa::prefetch_tensormap(&vsmap);
            }
        }
        const uint64_t policy = pa::l2_policy_evict_first();
        const int bs_shift = 31 - __clz(bs);          // block_size is 8, 16 or 32
        const int bpc = kChunk >> rows_shift;         // blocks (TMA boxes per tensor) per chunk
        const int32_t oob_row = p.num_blocks * bs;
        const uint32_t tx_bytes = L.stage_bytes + (kFp8 ? 2 * kChunk * 4 : 0);
        // A pair's table entries are read 32 at a time into a register window
        // (lane l holds entry wbase + l).  The window after it, and the next
        // pair's length and first window, are loaded one step ahead, so no
        // chunk waits on a table read.  Entries past the context (up to the
        // table width) are read but never used.
        struct Walk {
            Segment s;
            int32_t n_raw, wbase, went, wnext;
            int32_t kvh;  // the cache's KV head of the pair
            const int32_t* trow;
        };
        auto open = [&](int32_t at) {
            Walk w;
            w.s = find_segment(prefix, B, Hkv, at, hi);
            w.kvh = w.s.g / p.subs;
            w.n_raw = __ldg(p.context_lens + w.s.i);
            w.trow = p.block_tables + (int64_t)w.s.i * p.max_blocks;
            w.wbase = (w.s.c0 * kChunk) >> bs_shift;
            if (w.s.i == g_i && w.wbase == g_wbase) {   // the window loaded at entry
                w.went = g_went;
                w.wnext = g_wnext;
                g_i = -1;
                return w;
            }
            const int32_t j = w.wbase + lane;
            w.went = j < p.max_blocks ? __ldg(w.trow + j) : -1;
            w.wnext = j + 32 < p.max_blocks ? __ldg(w.trow + j + 32) : -1;
            return w;
        };
        int32_t k = 0;      // chunks of this CTA walked so far
        int stage = 0;      // k % S
        uint32_t use = 0;   // (k / S) & 1: parity of the stage's current use
        bool dead = false;
        Walk cur{}, nxt{};
        if (lo < hi) cur = open(lo);
        for (int32_t pos = lo; pos < hi && !dead;) {
            const int32_t npos = pos + cur.s.len;
            if (npos < hi) nxt = open(npos);
            const int32_t nb = (clamp_len(cur.n_raw, max_len) + bs - 1) >> bs_shift;
            for (int32_t t = 0; t < cur.s.len; ++t, ++k) {
                if ((k & (kProducerWarps - 1)) == prod) {
                    // Blocks j0 .. j0 + bpc - 1 of the chunk lie in one window
                    // (windows start at multiples of bpc); a producer moves at
                    // most 2 bpc <= 8 blocks per chunk, so one step suffices.
                    const int32_t j0 = ((cur.s.c0 + t) * kChunk) >> bs_shift;
                    if (j0 + bpc > cur.wbase + 32) {
                        cur.wbase += 32;
                        cur.went = cur.wnext;
                        const int32_t j = cur.wbase + 32 + lane;
                        cur.wnext = j < p.max_blocks ? __ldg(cur.trow + j) : -1;
                    }
                    if (k >= S && !__all_sync(0xffffffffu,
                                              pa::mbar_wait(&empty[stage], use ^ 1u, kWaitLimitNs))) {
                        dead = true;
                        if (lane == 0) pa::raise_error(p.err, PA_DEVERR_TIMEOUT);
                        break;
                    }
                    int32_t blk[4];
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        blk[b] = __shfl_sync(0xffffffffu, cur.went, (j0 - cur.wbase + b) & 31);
                    // One lane issues the chunk's boxes: per block, K then V
                    // (and, for FP8, their scales).  Blocks past the context
                    // and out-of-pool ids load from outside the map: zeros.
                    if (lane == 0) {
                        pa::mbar_arrive_expect_tx(&full[stage], tx_bytes);
                        unsigned char* kdst = smem + stage * L.stage_bytes;
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            if (b >= bpc) break;
                            bool ok = j0 + b < nb;
                            if (ok && (blk[b] < 0 || blk[b] >= p.num_blocks)) {
                                ok = false;
                                pa::raise_error(p.err, PA_DEVERR_BLOCK_ID);
                            }
                            const uint32_t off = ((uint32_t)b * kHalves << rows_shift) * 128;
                            const int32_t row = ok ? blk[b] * bs : oob_row;
                            const int32_t z = cur.kvh * (int32_t)kHalves;
                            pa::tma_load_3d(kdst + off, &kmap, &full[stage], 0, row, z, policy);
                            pa::tma_load_3d(kdst + L.stage_bytes / 2 + off, &vmap, &full[stage], 0,
                                            row, z, policy);
                            if constexpr (kFp8) {
                                unsigned char* sdst = smem + L.scales + stage * L.scale_stage +
                                                      (uint32_t)b * kScaleSlotBytes;
                                const int32_t sb = ok ? blk[b] : p.num_blocks;
                                pa::tma_load_3d(sdst, &ksmap, &full[stage], 0, cur.kvh, sb, policy);
                                pa::tma_load_3d(sdst + L.scale_stage / 2, &vsmap, &full[stage], 0,
                                                cur.kvh, sb, policy);
                            }
                        }
                    }
                    __syncwarp();
                }
                if (++stage == S) {
                    stage = 0;
                    use ^= 1u;
                }
            }
            cur = nxt;
            pos = npos;
        }
        // Every load this warp issued has landed before the CTA may exit.
        for (int s = prod; s < S && s < k; s += kProducerWarps) {
            const int32_t last_use = (k - 1 - s) / S;
            pa::mbar_wait(&full[s], (uint32_t)(last_use & 1), kWaitLimitNs);
        }
        return;
    }

    // ============================= consumer warps =============================
    if constexpr (kFp8) pa::setmaxnreg_inc<kQ8ConsumerRegs>();
    const int cr = lane >> 2;        // fragment row inside an 8-row group
    const int cc = 2 * (lane & 3);   // fragment column pair
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix / row this lane addresses
    const uint32_t smem_base = pa::smem_addr(smem);
    int32_t k = 0;
    bool dead = false;

    // Q^T fragments (MMA B operand) of a pair: lane holds query head 8 nt + cr.
    uint32_t qb[NT][D / 16][2];
    // Multiplier from an MMA score to the base-2 logit (FP8: times the K scale).
    float qsc = p.scale_log2;
    auto load_q = [&](const Segment& sg) {
        if constexpr (!kFp8) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hq = 8 * nt + cr;
                const uint16_t* qrow = p.q + ((int64_t)sg.i * p.H + sg.g * G + hq) * D + cc;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    qb[nt][ks][0] = hq < G ? ld_u32(qrow + ks * 16) : 0u;
                    qb[nt][ks][1] = hq < G ? ld_u32(qrow + ks * 16 + 8) : 0u;
                }
            }
        } else {
            // Head-dim order of the FP8 path: in k-step ks, the lane with
            // c4 = lane % 4 holds dims 32 c4 + 4 ks + {0, 1} (b0) and {2, 3}
            // (b1), so its 32 dims are contiguous.  A bf16 query is scaled by
            // 2^e (max |q| of the group into [2^14, 2^15)) and rounded to f16,
            // exact for elements down to 2^-29 of the largest.
            const int c4 = lane & 3;
            float amax = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int hq = 8 * nt + cr;
                const uint16_t* qrow = p.q + ((int64_t)sg.i * p.H + sg.g * G + hq) * D + 32 * c4;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    qb[nt][ks][0] = hq < G ? ld_u32(qrow + 4 * ks) : 0u;
                    qb[nt][ks][1] = hq < G ? ld_u32(qrow + 4 * ks + 2) : 0u;
                    if constexpr (kBF16)
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            amax = fmaxf(amax,
                                         fmaxf(fabsf(__uint_as_float(qb[nt][ks][j] << 16)),
                                               fabsf(__uint_as_float(qb[nt][ks][j] & 0xFFFF0000u))));
                }
            }
            if constexpr (kBF16) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
                const int e = min(141 - pa::biased_exponent(amax), 126);
                const float up = pa::exp2_int(e);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            qb[nt][ks][j] =
                                pa::pack2<false>(__uint_as_float(qb[nt][ks][j] << 16) * up,
                                                 __uint_as_float(qb[nt][ks][j] & 0xFFFF0000u) * up);
                qsc = p.scale_log2 * pa::exp2_int(-e);
            }
        }
    };
    constexpr int kSlotFloats = 2 * kMaxG + kMaxG * D;
    // The merge of one pair by a group of `nthr` threads (`t` = index in the
    // group, `sync` = the group's barrier): the final output if the pair lies
    // in this CTA's share, else this CTA's partial, and, if this CTA is the
    // pair's last, the merge of all CTAs' partials.  `so`, `sm`, `sl` hold the
    // consumer warps' unnormalised outputs, row maxima and row sums; `rinfo`
    // receives per row M = max_w m_w, L = sum_w 2^(m_w - M) l_w and the factors
    // f_w = 2^(m_w - M) (times 1/L for a final output).
    auto merge_pair = [&](const Segment& sg, int32_t h0, float* so, float* sm, float* sl,
                          float* rinfo, int* flag, int t, int nthr, auto sync) {
        const bool whole = sg.c0 == 0 && sg.len == sg.nc;
        if (t < G) {
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm[w * kMaxG + t]);
            float f[kConsumerWarps], Lsum = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                f[w] = pa::fast_exp2(sm[w * kMaxG + t] - M);
                Lsum += f[w] * sl[w * kMaxG + t];
            }
            const float scale = whole ? 1.f / Lsum : 1.f;
            rinfo[t] = M;
            rinfo[kMaxG + t] = Lsum;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) rinfo[(2 + w) * kMaxG + t] = f[w] * scale;
        }
        sync();
        // 4 consecutive head-dim values of one row, combined over the warps.
        auto combined4 = [&](int e) -> float4 {
            const int r = e / (D / 4), d4 = (e - r * (D / 4)) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float f = rinfo[(2 + w) * kMaxG + r];
                const float4 ov = *reinterpret_cast<const float4*>(&so[(w * G + r) * D + d4]);
                v.x += f * ov.x;
                v.y += f * ov.y;
                v.z += f * ov.z;
                v.w += f * ov.w;
            }
            return v;
        };
        auto store4 = [&](int r, int d4, float4 v) {
            uint2 packed;
            packed.x = pa::pack2<kBF16>(v.x, v.y);
            packed.y = pa::pack2<kBF16>(v.z, v.w);
            *reinterpret_cast<uint2*>(p.out + ((int64_t)sg.i * p.H + h0 + r) * D + d4) = packed;
        };
        if (whole) {
            for (int e = t; e < G * D / 4; e += nthr)
                store4(e / (D / 4), (e % (D / 4)) * 4, combined4(e));
            return;
        }
        // Partial result of this CTA for a pair split between CTAs.
        const int64_t c_first = ((int64_t)(sg.a + 1) * C - 1) / W;
        const int64_t c_last = ((int64_t)(sg.a + sg.nc) * C - 1) / W;
        float* ps = p.partials + partial_slot(blockIdx.x, W, C, sg.a) * kSlotFloats;
        for (int e = t; e < G * D / 4; e += nthr) {
            const int r = e / (D / 4), d4 = (e - r * (D / 4)) * 4;
            *reinterpret_cast<float4*>(&ps[2 * kMaxG + r * D + d4]) = combined4(e);
        }
        if (t < G) {
            ps[t] = rinfo[t];
            ps[kMaxG + t] = rinfo[kMaxG + t];
        }
        // Publish: the group barrier orders every thread's stores before thread
        // 0's release (cumulativity); the acquire-release ticket names the
        // pair's last CTA and, for that CTA, acquires every other CTA's partial.
        sync();
        if (t == 0) {
            int32_t* ctr = p.counters + (int64_t)sg.i * Hkv + sg.g;
            const int prev = pa::atomic_add_acq_rel_gpu(ctr, 1);
            const int last = prev == (int)(c_last - c_first);
            if (last) atomicExch(ctr, 0);   // ready for the next launch
            *flag = last;
        }
        sync();
        if (!*flag) return;
        // Last CTA of the pair: each thread folds, for its 4 output values, the
        // ncov partials (m_c, l_c, O_c) eight at a time (all eight loads in
        // flight at once): M = max m_c, out = sum 2^(m_c - M) O_c / sum
        // 2^(m_c - M) l_c.
        const int ncov = (int)(c_last - c_first + 1);
        // CTA c > c_first starts inside the pair (its first slot); c_first
        // uses its first slot only if its share starts there.
        const int64_t slot0 = 2 * c_first + (cta_begin(c_first, W, C) == sg.a ? 0 : 1);
        for (int e = t; e < G * D / 4; e += nthr) {
            const int r = e / (D / 4), d4 = (e - r * (D / 4)) * 4;
            float M = -INFINITY, Ls = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int c0 = 0; c0 < ncov; c0 += 8) {
                float pm[8], pl[8];
                float4 po[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int c = c0 + j;
                    if (c < ncov) {
                        const float* q = p.partials + (c ? 2 * (c_first + c) : slot0) * kSlotFloats;
                        pm[j] = __ldcg(q + r);
                        pl[j] = __ldcg(q + kMaxG + r);
                        po[j] = __ldcg(reinterpret_cast<const float4*>(q + 2 * kMaxG + r * D + d4));
                    } else {
                        pm[j] = -INFINITY;
                        pl[j] = 0.f;
                        po[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                float Mb = M;
#pragma unroll
                for (int j = 0; j < 8; ++j) Mb = fmaxf(Mb, pm[j]);
                if (Mb == -INFINITY) continue;
                const float a = pa::fast_exp2(M - Mb);   // 0 while M = -inf
                Ls *= a;
                acc.x *= a;
                acc.y *= a;
                acc.z *= a;
                acc.w *= a;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float f = pa::fast_exp2(pm[j] - Mb);
                    Ls += f * pl[j];
                    acc.x += f * po[j].x;
                    acc.y += f * po[j].y;
                    acc.z += f * po[j].z;
                    acc.w += f * po[j].w;
                }
                M = Mb;
            }
            const float inv = 1.f / Ls;
            store4(r, d4, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
        }
    };

    Segment s{};
    int32_t n = 0;
    int32_t segn = 0;  // pairs this CTA has walked (selects the merge slot)
    if (lo < hi) {
        s = find_segment(prefix, B, Hkv, lo, hi);
        n = clamp_len(__ldg(p.context_lens + s.i), max_len);
        load_q(s);
    }
    for (int32_t pos = lo; pos < hi;) {
        const int32_t head0 = s.g * G;
        // Running state for the heads 8 nt + cc + {0, 1} this lane tracks.
        float m_run[NT][2], l_run[NT][2];
        float o[D / 16][NT][4];  // O^T: rows = head_dim, columns = heads
        // FP8: o holds the output times 2^vexp (P scaled by the V scales and by
        // 2^vexp stays below 2^15, inside f16 range).
        int vexp = 126;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m_run[nt][0] = m_run[nt][1] = -INFINITY;
            l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt)
                o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
        }

        // Chunk k lives in stage k % S and stage s is always consumed by warp
        // s % kConsumerWarps, so consecutive uses of a stage meet the same warp
        // (a warp owning no stage, when S < kConsumerWarps, takes no chunk).
        const int s0 = k % S;
        const int d0 = (warp - s0 % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
        const int32_t first = warp >= S ? s.len : (s0 + d0 < S ? d0 : (S - s0) + warp);
        for (int32_t t = first; t < s.len;) {
            const int32_t kk = k + t;
            const int stage = kk % S;
            const bool ready =
                dead || pa::mbar_wait(&full[stage], (uint32_t)((kk / S) & 1), kWaitLimitNs);
            if (!__all_sync(0xffffffffu, ready)) {
                dead = true;
                if (lane == 0) pa::raise_error(p.err, PA_DEVERR_TIMEOUT);
            }
            if (!dead) {
                const int32_t valid = min(n - (s.c0 + t) * kChunk, kChunk);
                const uint32_t kt = smem_base + stage * L.stage_bytes;
                const uint32_t vt = kt + L.stage_bytes / 2;
                if (valid < kChunk) {
                    // Rows past the context may hold anything (even NaN): zero
                    // them in V so that 0-weight rows add exactly nothing.
                    unsigned char* vbytes = smem + stage * L.stage_bytes + L.stage_bytes / 2;
                    const int per_half = (kChunk - valid) * 8;
                    for (int e = lane; e < per_half * (int)kHalves; e += 32) {
                        const int h = e / per_half, rem = e - h * per_half;
                        const uint32_t tok = (uint32_t)(valid + (rem >> 3));
                        *reinterpret_cast<uint4*>(
                            vbytes + tile_offset(tok, h, rem & 7, kHalves, rows_shift)) =
                            make_uint4(0, 0, 0, 0);
                    }
                    pa::fence_proxy_async_smem();
                    __syncwarp();
                }

                // Per-token factors of this lane's key rows 16 mt + cr + 8 h:
                // kmul takes an MMA score to a base-2 logit, vmul scales P.
                float kmul[kKeyTiles][2], vmul[kKeyTiles][2];
                float rs = 1.f;  // extra factor on o this chunk
                if constexpr (kFp8) {
                    const uint32_t sk = smem_base + L.scales + (uint32_t)stage * L.scale_stage;
                    float vmax = 0.f;
#pragma unroll
                    for (int mt = 0; mt < kKeyTiles; ++mt)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t tok = (uint32_t)(mt * 16 + cr + 8 * h);
                            const uint32_t off =
                                ((tok >> rows_shift) * (kScaleSlotBytes / 4) +
                                 (tok & ((1u << rows_shift) - 1u))) * 4;
                            kmul[mt][h] = pa::lds_f32(sk + off) * qsc;
                            const float sv = (int)tok < valid
                                                 ? pa::lds_f32(sk + L.scale_stage / 2 + off)
                                                 : 0.f;
                            vmul[mt][h] = sv;
                            vmax = fmaxf(vmax, sv);
                        }
                    // the warp's largest scale magnitude in one reduction: the
                    // bit patterns of non-negative floats order like the values
                    vmax = __uint_as_float(
                        __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(vmax))));
                    if (vmax > 0.f) {
                        const int e = min(vexp, 141 - pa::biased_exponent(vmax));
                        if (e < vexp) {
                            rs = e - vexp >= -126 ? pa::exp2_int(e - vexp) : 0.f;
                            vexp = e;
                        }
                    }
                    const float f = pa::exp2_int(vexp);
#pragma unroll
                    for (int mt = 0; mt < kKeyTiles; ++mt) {
                        vmul[mt][0] *= f;
                        vmul[mt][1] *= f;
                    }
                } else {
#pragma unroll
                    for (int mt = 0; mt < kKeyTiles; ++mt) {
                        kmul[mt][0] = kmul[mt][1] = p.scale_log2;
                        vmul[mt][0] = vmul[mt][1] = 1.f;
                    }
                }

                // S^T = K Q^T: kChunk / 16 key m-tiles x NT 8-head n-tiles.
                float st[kKeyTiles][NT][4];
#pragma unroll
                for (int mt = 0; mt < kKeyTiles; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        st[mt][nt][0] = st[mt][nt][1] = st[mt][nt][2] = st[mt][nt][3] = 0.f;
                if constexpr (kFp8) {
                    // Rows 16 mt + cr (+ 8): 16-byte columns 2 c4 and 2 c4 + 1
                    // (stored at column ^ cr) hold the 32 dims of the lane's
                    // k-order; 8 lanes of a phase hit 8 distinct columns.
                    const uint32_t c4 = (uint32_t)(lane & 3);
#pragma unroll
                    for (int mt = 0; mt < kKeyTiles; ++mt) {
                        uint4 w[2][2];
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const uint32_t tok = (uint32_t)(mt * 16 + cr + 8 * h);
                                w[h][j] = pa::lds128(kt + (tok << 7) +
                                                     (((2 * c4 + j) ^ (uint32_t)cr) << 4));
                            }
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            uint32_t a[4];
                            q8x4_to_f16<kInt8>(u4_word(w[0][ks >> 2], ks & 3), a[0], a[2]);
                            q8x4_to_f16<kInt8>(u4_word(w[1][ks >> 2], ks & 3), a[1], a[3]);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                pa::mma_16816<false>(st[mt][nt], a, qb[nt][ks][0], qb[nt][ks][1]);
                        }
                    }
                }
#pragma unroll
                for (int ks = 0; ks < (kFp8 ? 0 : D / 16); ++ks) {
                    const uint32_t col = (uint32_t)((ks & 3) * 2 + (mi >> 1));
#pragma unroll
                    for (int mt = 0; mt < kKeyTiles; ++mt) {
                        const uint32_t tok = (uint32_t)(mt * 16 + (mi & 1) * 8 + rr);
                        uint32_t a[4];
                        pa::ldsm_x4(kt + tile_offset(tok, (uint32_t)(ks >> 2), col, kHalves,
                                                     rows_shift),
                                    a[0], a[1], a[2], a[3]);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            pa::mma_16816<kBF16>(st[mt][nt], a, qb[nt][ks][0], qb[nt][ks][1]);
                    }
                }

                // Online softmax in base 2, per head (column).
                float mx[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mx[nt][0] = mx[nt][1] = -INFINITY;
#pragma unroll
                    for (int mt = 0; mt < kKeyTiles; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int tok = mt * 16 + cr + 8 * (e >> 1);
                            const float x =
                                tok < valid ? st[mt][nt][e] * kmul[mt][e >> 1] : -INFINITY;
                            st[mt][nt][e] = x;
                            mx[nt][e & 1] = fmaxf(mx[nt][e & 1], x);
                        }
                }
                bool grew = false;
                float alpha[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        float v = mx[nt][j];
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                        const float m_new = fmaxf(m_run[nt][j], v);
                        grew |= m_new > m_run[nt][j];
                        alpha[nt][j] = pa::fast_exp2(m_run[nt][j] - m_new);
                        m_run[nt][j] = m_new;
                        l_run[nt][j] *= alpha[nt][j];
                    }
                if (__any_sync(0xffffffffu, grew) || rs != 1.f) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        alpha[nt][0] *= rs;
                        alpha[nt][1] *= rs;
                    }
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            o[mt][nt][0] *= alpha[nt][0];
                            o[mt][nt][1] *= alpha[nt][1];
                            o[mt][nt][2] *= alpha[nt][0];
                            o[mt][nt][3] *= alpha[nt][1];
                        }
                }
                // P^T as MMA B fragments: exp2, pack to 16 bits, transpose 8x8 tiles.
                // A bf16 P keeps 8 bits; its rounding residual (pbl, a second
                // B operand) restores about 16, so a short context whose V terms
                // cancel stays within the tolerance (f16 and FP8 use f16 P).
                constexpr bool kPbf16 = kBF16 && !kFp8;
                uint32_t pb[kKeyTiles][NT][2];
                uint32_t pbl[kKeyTiles][NT][2];
#pragma unroll
                for (int mt = 0; mt < kKeyTiles; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        float e4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            e4[e] = pa::fast_exp2(st[mt][nt][e] - m_run[nt][e & 1]);
                            l_run[nt][e & 1] += e4[e];
                        }
                        if constexpr (kFp8) {
                            // V scale folded into P; rows past the context get
                            // exactly 0 (vmul = 0 there).
                            e4[0] *= vmul[mt][0];
                            e4[1] *= vmul[mt][0];
                            e4[2] *= vmul[mt][1];
                            e4[3] *= vmul[mt][1];
                        }
                        const uint32_t h01 = pa::pack2<kPbf16>(e4[0], e4[1]);
                        const uint32_t h23 = pa::pack2<kPbf16>(e4[2], e4[3]);
                        pb[mt][nt][0] = pa::movmatrix_trans(h01);
                        pb[mt][nt][1] = pa::movmatrix_trans(h23);
                        if constexpr (kPbf16) {
                            pbl[mt][nt][0] =
                                pa::movmatrix_trans(pa::bf16x2_residual(h01, e4[0], e4[1]));
                            pbl[mt][nt][1] =
                                pa::movmatrix_trans(pa::bf16x2_residual(h23, e4[2], e4[3]));
                        }
                    }

                // O^T += V^T P^T: head_dim in 16-row m-tiles, keys in 16-key steps.
                if constexpr (kFp8) {
                    // Row rho of m-tile mt is head dim 8 rho + mt, so the lane's
                    // rows cr and cr + 8 of all eight m-tiles are 8 contiguous
                    // bytes (dims 8 cr .. and 64 + 8 cr ..) of each key row it
                    // needs: keys 16 ks2 + 2 c4 + {0, 1, 8, 9}.
                    const uint32_t c4 = (uint32_t)(lane & 3);
                    const uint32_t part = (uint32_t)(cr & 1) * 8;
#pragma unroll
                    for (int ks2 = 0; ks2 < kKeyTiles; ++ks2) {
                        uint2 lo[4], hi[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const uint32_t tok = 16 * ks2 + 2 * c4 + (u & 1) + 8 * (u >> 1);
                            const uint32_t row = vt + (tok << 7) + part;
                            lo[u] = pa::lds64(row + ((((uint32_t)cr >> 1) ^ (tok & 7)) << 4));
                            hi[u] = pa::lds64(row + (((4 + ((uint32_t)cr >> 1)) ^ (tok & 7)) << 4));
                        }
#pragma unroll
                        for (int q4 = 0; q4 < 2; ++q4) {
                            // A fragment u of m-tiles 4 q4 .. 4 q4 + 3: keys of
                            // fragment u from rows (lo | hi)[2 (u >> 1)] and
                            // [2 (u >> 1) + 1], interleaved byte by byte.
                            uint32_t af[4][4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const uint2* src = (u & 1) ? hi : lo;
                                const uint32_t x = q4 ? src[2 * (u >> 1)].y : src[2 * (u >> 1)].x;
                                const uint32_t y =
                                    q4 ? src[2 * (u >> 1) + 1].y : src[2 * (u >> 1) + 1].x;
                                q8x4_to_f16<kInt8>(__byte_perm(x, y, 0x5140), af[u][0], af[u][1]);
                                q8x4_to_f16<kInt8>(__byte_perm(x, y, 0x7362), af[u][2], af[u][3]);
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const uint32_t a[4] = {af[0][i], af[1][i], af[2][i], af[3][i]};
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
                                    pa::mma_16816<false>(o[4 * q4 + i][nt], a, pb[ks2][nt][0],
                                                         pb[ks2][nt][1]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int ks2 = 0; ks2 < (kFp8 ? 0 : kKeyTiles); ++ks2) {
                    const uint32_t tok = (uint32_t)(ks2 * 16 + (mi >> 1) * 8 + rr);
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        const int dd = mt * 16 + (mi & 1) * 8;
                        uint32_t a[4];
                        pa::ldsm_x4_trans(vt + tile_offset(tok, (uint32_t)(dd >> 6),
                                                           (uint32_t)((dd & 63) >> 3), kHalves,
                                                           rows_shift),
                                          a[0], a[1], a[2], a[3]);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            pa::mma_16816<kBF16>(o[mt][nt], a, pb[ks2][nt][0], pb[ks2][nt][1]);
                            if constexpr (kPbf16)
                                pa::mma_16816<kBF16>(o[mt][nt], a, pbl[ks2][nt][0],
                                                     pbl[ks2][nt][1]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(&empty[stage]);
            // next chunk whose stage belongs to this warp
            const int next_stage = stage + kConsumerWarps;
            t += next_stage < S ? kConsumerWarps : (S - stage) + warp;
        }
        k += s.len;

        // ---- hand this warp's state for the pair to the pair's merge slot.
        // The four warps do not wait for each other: each deposits its state
        // in slot (pair index & 1) and the last to arrive merges the pair
        // while the others go on to the next one.
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float v = l_run[nt][j];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                l_run[nt][j] = v;
            }
        const int slot = kAsync ? (segn & 1) : 0;
        const int slot_floats_o = kConsumerWarps * G * D;
        float* so = merge_o + slot * slot_floats_o;
        float* sm = merge_m + slot * (kConsumerWarps * kMaxG);
        float* sl = merge_l + slot * (kConsumerWarps * kMaxG);
        float* rinfo = rowinfo + slot * (2 + kConsumerWarps) * kMaxG;
        if constexpr (kAsync) {
            // The slot is free once the merge of pair segn - 2 has read it.
            if (!__all_sync(0xffffffffu, wait_flag(&slot_free[slot], segn, kWaitLimitNs)) &&
                lane == 0)
                pa::raise_error(p.err, PA_DEVERR_TIMEOUT);
            __threadfence_block();
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int h = 8 * nt + cc + j;
                if (cr == 0 && h < G) {
                    sm[warp * kMaxG + h] = m_run[nt][j];
                    sl[warp * kMaxG + h] = l_run[nt][j];
                }
            }
        if constexpr (kFp8) {
            // o[mt][nt][e] is head dim 8 (cr + 8 (e >> 1)) + mt, scaled by 2^vexp.
            const float inv = pa::exp2_int(-vexp);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int h = 8 * nt + cc + (e & 1);
                    if (h < G) {
                        float4* dst = reinterpret_cast<float4*>(
                            &so[(warp * G + h) * D + 8 * cr + 64 * (e >> 1)]);
                        dst[0] = make_float4(o[0][nt][e] * inv, o[1][nt][e] * inv,
                                             o[2][nt][e] * inv, o[3][nt][e] * inv);
                        dst[1] = make_float4(o[4][nt][e] * inv, o[5][nt][e] * inv,
                                             o[6][nt][e] * inv, o[7][nt][e] * inv);
                    }
                }
        } else {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = 8 * nt + cc + (e & 1);
                        if (h < G)
                            so[(warp * G + h) * D + mt * 16 + cr + 8 * (e >> 1)] = o[mt][nt][e];
                    }
        }

        // The next pair's length and query fragments load while this one merges.
        const int32_t npos = pos + s.len;
        Segment sn = s;
        int32_t n_next = n;
        if (npos < hi) {
            sn = find_segment(prefix, B, Hkv, npos, hi);
            n_next = clamp_len(__ldg(p.context_lens + sn.i), max_len);
            load_q(sn);
        }

        if constexpr (kAsync) {
            // The four warps do not wait for each other: the last one to
            // deposit its state merges the pair while the others go on.
            __syncwarp();
            int last = 0;
            if (lane == 0) {
                __threadfence_block();
                last = atomicAdd(&slot_count[slot], 1) == kConsumerWarps - 1;
                if (last) __threadfence_block();
            }
            if (__shfl_sync(0xffffffffu, last, 0)) {
                __syncwarp();
                merge_pair(s, head0, so, sm, sl, rinfo, &slot_flag[slot], lane, 32,
                           [] { __syncwarp(); });
                __syncwarp();
                if (lane == 0) {
                    slot_count[slot] = 0;
                    __threadfence_block();
                    *reinterpret_cast<volatile int*>(&slot_free[slot]) = segn + 2;
                }
            }
        } else {
            // All four warps meet and merge the pair together.
            pa::named_barrier_sync(1, kConsumerThreads);
            merge_pair(s, head0, so, sm, sl, rinfo, &slot_flag[slot], tid, kConsumerThreads,
                       [] { pa::named_barrier_sync(1, kConsumerThreads); });
            pa::named_barrier_sync(1, kConsumerThreads);
        }
        ++segn;
        s = sn;
        n = n_next;
        pos = npos;
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

// A 3-D view of one cache for the TMA: x = 64 elements (128 bytes), y = token
// row of the pool (num_blocks * block_size rows, stride Hkv * d elements),
// z = 64-column half over all KV heads (stride 128 bytes).  A box of
// {64, block_size, d / 64} at (0, block * block_size, head * d / 64) is one
// block of one KV head, landing as [half][row][64] in shared memory.
bool encode_cache_map(CUtensorMap* map, const void* base, int32_t rows, int32_t Hkv, int32_t d,
                      int32_t block_size, pa_dtype dtype) {
    auto encode = get_encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)Hkv * d / 64};
    const cuuint64_t strides[2] = {(cuuint64_t)Hkv * d * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)(block_size < kChunk ? block_size : kChunk),
                               (cuuint32_t)(d / 64)};
    const cuuint32_t elem[3] = {1, 1, 1};
    const CUresult r = encode(
        map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
        3, const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// FP8 codes: x = the 128 code bytes of a (token, KV head) row, y = token row
// of the pool (stride Hkv * 128 bytes), z = KV head (stride 128 bytes).  A box
// of {128, block_size, 1} at (0, block * block_size, head) is one block of one
// KV head, [row][128 bytes] in shared memory with the 128-byte swizzle.
bool encode_code_map(CUtensorMap* map, const void* base, int32_t rows, int32_t Hkv,
                     int32_t block_size) {
    auto encode = get_encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)Hkv};
    const cuuint64_t strides[2] = {(cuuint64_t)Hkv * 128, 128};
    const cuuint32_t box[3] = {128, (cuuint32_t)(block_size < kChunk ? block_size : kChunk), 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    // 128-byte promotion: a row of one KV head is 128 bytes; 256 would pull in
    // the next head's row, which another CTA reads much later.
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP8 scales [num_blocks][Hkv][block_size] fp32: a box of {block_size, 1, 1}
// at (0, head, block) is the block's scales for one KV head; a block index of
// num_blocks lies outside and arrives as zeros.
bool encode_scale_map(CUtensorMap* map, const float* base, int32_t num_blocks, int32_t Hkv,
                      int32_t block_size) {
    auto encode = get_encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)block_size, (cuuint64_t)Hkv, (cuuint64_t)num_blocks};
    const cuuint64_t strides[2] = {(cuuint64_t)block_size * 4, (cuuint64_t)Hkv * block_size * 4};
    const cuuint32_t box[3] = {(cuuint32_t)block_size, 1, 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides,
                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t slot_floats(int32_t d) { return 2 * kMaxG + (size_t)kMaxG * d; }

size_t counters_bytes(int32_t B, int32_t H) {
    return (((size_t)B * H * sizeof(int32_t)) + 255) & ~size_t(255);
}

// Pipeline depth that fits the shared-memory budget.  The stage waits use
// mbarrier phase parity, which is only sound if use u + 1 of a stage is never
// awaited before use u completed.  Chunks k and k + S share stage k % S; the
// stage is issued by producer k % 2 (S is even) and consumed by warp
// (k % S) % kConsumerWarps, so consecutive uses of a stage always belong to
// the same producer and the same consumer warp, and each waiter is at most one
// phase ahead.
// Narrow groups (G <= 2) merge asynchronously: per pair end the math is small
// and the ring depth decides; wider groups merge with all four warps.
bool async_merge(int G) { return G <= 2; }

int choose_stages(int D, int G, int B, bool fp8, int bs) {
    const int align = fp8 ? producer_warps(true) : 2;   // stages per producer turn
    const Layout L0 = make_layout(D, G, B, 0, async_merge(G) ? 2 : 1, fp8, bs);
    if (L0.total >= kSmemBudget) return 0;
    const uint32_t per_stage = L0.stage_bytes + L0.scale_stage;
    int s = (int)((kSmemBudget - L0.total) / per_stage);
    if (s > kMaxStages) s = kMaxStages;
    s -= s % align;  // each producer owns every align-th stage
    // Wider groups make the consumers the limit: give every consumer warp the
    // same number of stages.  Narrow ones are bound by bytes in flight: keep
    // the deepest ring.
    if (G > 2 && s >= kConsumerWarps) s -= s % kConsumerWarps;
    return s;
}

template <int D, bool kBF16, int NT, bool kAsync, bool kFp8, bool kInt8>
pa_status launch(const CUtensorMap& km, const CUtensorMap& vm, const CUtensorMap& ksm,
                 const CUtensorMap& vsm, const DecodeParams& prm, size_t smem,
                 cudaStream_t stream) {
    auto kern = paged_decode_kernel<D, kBF16, NT, kAsync, kFp8, kInt8>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    static int regs = 0;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kSmemBudget);
        cudaFuncAttributes fa{};
        if (attr_err == cudaSuccess) attr_err = cudaFuncGetAttributes(&fa, kern);
        regs = fa.numRegs;
    });
    if (attr_err != cudaSuccess) return PA_ERR_CUDA;
    // The 8-bit register split adds up only against this launch allocation: a
    // kernel built with another count would wait forever in setmaxnreg.
    if (kFp8 && regs != kQ8LaunchRegs) return PA_ERR_UNSUPPORTED;
    kern<<<pa_decode_grid_size(), cta_threads(kFp8), smem, stream>>>(km, vm, ksm, vsm, prm);
    return pa::cuda_status(cudaGetLastError());
}

template <int D, bool kBF16, bool kFp8, bool kInt8 = false>
pa_status launch_g(const CUtensorMap& km, const CUtensorMap& vm, const CUtensorMap& ksm,
                   const CUtensorMap& vsm, const DecodeParams& prm, size_t smem,
                   cudaStream_t stream) {
    if (async_merge(prm.G))
        return launch<D, kBF16, 1, true, kFp8, kInt8>(km, vm, ksm, vsm, prm, smem, stream);
    return prm.G <= 8
               ? launch<D, kBF16, 1, false, kFp8, kInt8>(km, vm, ksm, vsm, prm, smem, stream)
               : launch<D, kBF16, 2, false, kFp8, kInt8>(km, vm, ksm, vsm, prm, smem, stream);
}

// Checks shared by pa_decode and pa_decode_fp8; fills everything of prm but the
// pointers and returns the shared-memory size in *smem.
pa_status prepare(int32_t max_blocks, int32_t max_context_len, int32_t B, int32_t H, int32_t Hkv,
                  int32_t d, int32_t block_size, int32_t num_blocks, float scale, pa_dtype dtype,
                  size_t ws_bytes, bool fp8, DecodeParams* prm, size_t* smem) {
    if (B < 0 || H <= 0 || Hkv <= 0 || max_blocks <= 0 || num_blocks <= 0 ||
        max_context_len < 0 || !std::isfinite(scale))
        return PA_ERR_INVALID;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (H % Hkv != 0) return PA_ERR_UNSUPPORTED;
    // Groups wider than kMaxG query heads (multi-query attention) are split
    // into sub-groups of kMaxG heads, each a pair of its own.
    int G = H / Hkv, subs = 1;
    if (G > kMaxG) {
        if (G % kMaxG != 0) return PA_ERR_UNSUPPORTED;
        subs = G / kMaxG;
        G = kMaxG;
    }
    if (d != 128 && (fp8 || d != 64)) return PA_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
    if (B > kMaxBatch) return PA_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
    // Flattened chunk indices are int32: every sequence's chunks times Hkv.
    const int64_t max_chunks = ((int64_t)max_blocks * block_size + kChunk - 1) / kChunk;
    if ((int64_t)B * Hkv * subs * max_chunks >= ((int64_t)1 << 30)) return PA_ERR_UNSUPPORTED;
    const int stages = choose_stages(d, G, B, fp8, block_size);
    if (stages < 2) return PA_ERR_UNSUPPORTED;
    if (B > 0 && ws_bytes < pa_decode_workspace_size(B, H, d)) return PA_ERR_INVALID;
    prm->max_blocks = max_blocks;
    prm->B = B;
    prm->H = H;
    prm->Hkv = Hkv * subs;
    prm->G = G;
    prm->subs = subs;
    prm->bs = block_size;
    prm->num_blocks = num_blocks;
    prm->stages = stages;
    prm->len_hint = max_context_len;
    prm->scale_log2 = scale * kLog2e;
    *smem = make_layout(d, G, B, stages, async_merge(G) ? 2 : 1, fp8, block_size).total;
    return PA_OK;
}

}  // namespace

extern "C" {

PA_API size_t pa_decode_workspace_size(int32_t B, int32_t H, int32_t d) {
    if (B < 0 || H <= 0 || (d != 64 && d != 128)) return 0;
    return counters_bytes(B, H) + 2 * (size_t)kMaxCtas * slot_floats(d) * sizeof(float);
}

PA_API int32_t pa_decode_grid_size(void) {
    const int ctas = pa::device_sm_count() * kCtasPerSm;
    return ctas > kMaxCtas ? kMaxCtas : ctas;
}

PA_API pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int32_t max_blocks,
                           const int32_t* context_lens, int32_t max_context_len, int32_t B,
                           int32_t H, int32_t Hkv, int32_t d, int32_t block_size,
                           int32_t num_blocks, float scale, pa_dtype dtype, void* out,
                           void* workspace, size_t ws_bytes, void* stream) {
    DecodeParams prm;
    size_t smem = 0;
    const pa_status st0 = prepare(max_blocks, max_context_len, B, H, Hkv, d, block_size,
                                  num_blocks, scale, dtype, ws_bytes, false, &prm, &smem);
    if (st0 != PA_OK || B == 0) return st0;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace)
        return PA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15u)
        return PA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(q) & 3u) || (reinterpret_cast<uintptr_t>(out) & 15u))
        return PA_ERR_INVALID;

    unsigned int* err = pa::device_error_word();
    if (!err || pa_decode_grid_size() <= 0) return PA_ERR_CUDA;

    CUtensorMap km, vm;
    const int32_t rows = num_blocks * block_size;
    if (!encode_cache_map(&km, k_cache, rows, Hkv, d, block_size, dtype) ||
        !encode_cache_map(&vm, v_cache, rows, Hkv, d, block_size, dtype))
        return PA_ERR_CUDA;

    prm.q = static_cast<const uint16_t*>(q);
    prm.out = static_cast<uint16_t*>(out);
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.counters = static_cast<int32_t*>(workspace);
    prm.partials = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) +
                                            counters_bytes(B, H));
    prm.err = err;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (d == 128)
        return dtype == PA_BF16 ? launch_g<128, true, false>(km, vm, km, vm, prm, smem, st)
                                : launch_g<128, false, false>(km, vm, km, vm, prm, smem, st);
    return dtype == PA_BF16 ? launch_g<64, true, false>(km, vm, km, vm, prm, smem, st)
                            : launch_g<64, false, false>(km, vm, km, vm, prm, smem, st);
}

}  // extern "C"

namespace {

// pa_decode_fp8 and pa_decode_int8: the decode over an 8-bit cache of E4M3
// (kInt8 false) or INT8 codes with per-(token, KV head) scales.
template <bool kInt8>
pa_status decode_q8(const void* q, const void* k_cache, const void* v_cache,
                    const float* k_scale, const float* v_scale, const int32_t* block_tables,
                    int32_t max_blocks, const int32_t* context_lens, int32_t max_context_len,
                    int32_t B, int32_t H, int32_t Hkv, int32_t d, int32_t block_size,
                    int32_t num_blocks, float scale, pa_dtype dtype, void* out, void* workspace,
                    size_t ws_bytes, void* stream) {
    DecodeParams prm;
    size_t smem = 0;
    const pa_status st0 = prepare(max_blocks, max_context_len, B, H, Hkv, d, block_size,
                                  num_blocks, scale, dtype, ws_bytes, true, &prm, &smem);
    if (st0 != PA_OK || B == 0) return st0;
    if (!q || !k_cache || !v_cache || !k_scale || !v_scale || !block_tables || !context_lens ||
        !out || !workspace)
        return PA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
         reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale)) &
        15u)
        return PA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(q) & 3u) || (reinterpret_cast<uintptr_t>(out) & 15u))
        return PA_ERR_INVALID;

    unsigned int* err = pa::device_error_word();
    if (!err || pa_decode_grid_size() <= 0) return PA_ERR_CUDA;

    CUtensorMap km, vm, ksm, vsm;
    const int32_t rows = num_blocks * block_size;
    if (!encode_code_map(&km, k_cache, rows, Hkv, block_size) ||
        !encode_code_map(&vm, v_cache, rows, Hkv, block_size) ||
        !encode_scale_map(&ksm, k_scale, num_blocks, Hkv, block_size) ||
        !encode_scale_map(&vsm, v_scale, num_blocks, Hkv, block_size))
        return PA_ERR_CUDA;

    prm.q = static_cast<const uint16_t*>(q);
    prm.out = static_cast<uint16_t*>(out);
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.counters = static_cast<int32_t*>(workspace);
    prm.partials = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) +
                                            counters_bytes(B, H));
    prm.err = err;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return dtype == PA_BF16 ? launch_g<128, true, true, kInt8>(km, vm, ksm, vsm, prm, smem, st)
                            : launch_g<128, false, true, kInt8>(km, vm, ksm, vsm, prm, smem, st);
}

}  // namespace

extern "C" {

PA_API pa_status pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                               const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, int32_t max_blocks,
                               const int32_t* context_lens, int32_t max_context_len, int32_t B,
                               int32_t H, int32_t Hkv, int32_t d, int32_t block_size,
                               int32_t num_blocks, float scale, pa_dtype dtype, void* out,
                               void* workspace, size_t ws_bytes, void* stream) {
    return decode_q8<false>(q, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks,
                            context_lens, max_context_len, B, H, Hkv, d, block_size, num_blocks,
                            scale, dtype, out, workspace, ws_bytes, stream);
}

PA_API pa_status pa_decode_int8(const void* q, const void* k_cache, const void* v_cache,
                                const float* k_scale, const float* v_scale,
                                const int32_t* block_tables, int32_t max_blocks,
                                const int32_t* context_lens, int32_t max_context_len, int32_t B,
                                int32_t H, int32_t Hkv, int32_t d, int32_t block_size,
                                int32_t num_blocks, float scale, pa_dtype dtype, void* out,
                                void* workspace, size_t ws_bytes, void* stream) {
    return decode_q8<true>(q, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks,
                           context_lens, max_context_len, B, H, Hkv, d, block_size, num_blocks,
                           scale, dtype, out, workspace, ws_bytes, stream);
}

}  // extern "C"
