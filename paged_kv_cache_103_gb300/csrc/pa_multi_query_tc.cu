// Several query tokens per sequence over the paged cache on the 5th-generation
// tensor cores (pa_multi_query_tc): the chunked-prefill shape of "vLLM 深度拆解：
// 当大模型推理学会「分页注意力」", section 5 (a long prompt's prefill cut into
// chunks that run between decode steps), where a KV head's group of query heads
// times the chunk's tokens fills 128-row tiles.  It computes what
// pa_multi_query computes: sequence i's queries are its last qlen_i cached
// tokens (rows q_start[i] .. q_start[i+1]-1 of q); query t attends to cached
// tokens 0 .. n_i - qlen_i + t, softmax(q k^T * scale) v.
//
//  * A query tile is 128 rows, a row being one (query token, query head of a
//    KV head g's group) pair in token-major order, so the group's G heads share
//    every K/V tile.  A work item is two consecutive query tiles of one
//    (sequence, KV head): both read the same 128-key K/V tiles, so each K/V
//    byte brought in serves 256 rows.  One CTA per SM walks its items (a
//    balanced static order: each sequence's heaviest tiles first, dealt to the
//    CTAs back and forth).
//  * Warp 0 issues TMA for the item's Q tiles (two 4-D boxes per tile, one per
//    64-column half, landing as 128 rows x 128 bytes with the 128-byte
//    swizzle) and for K; warp 2 for V.  Each walks the block table (the next
//    tile's entries read before the current tile's stage is awaited) and loads
//    a key tile as 8-row boxes of both halves, so every 8 keys x 64 columns
//    form one 1024-byte swizzle atom (K-major for K, MN-major for V).
//  * Warp 1 issues tcgen05.mma (one thread) into tensor memory, per query tile
//    w: S_w = Q_w K^T (M = N = 128, eight K = 16 steps over the head dim) and
//    O_w += P_w V (N = head dim, eight K = 16 steps over the keys, P read from
//    TMEM).  The order PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) keeps the tensor
//    core on one tile's products while the other tile's softmax runs; since
//    one thread's tcgen05.mma run in issue order, S_w(j+1) -- written over the
//    columns that hold P_w(j) -- follows PV_w(j).
//  * Warpgroups 1 and 2 (warps 4-7, 8-11) run the online softmax of tiles 0
//    and 1 (thread r of a warpgroup owns TMEM lane r, i.e. row r), in base 2
//    with each row's causal limit: S is read with tcgen05.ld, P = 2^(s - m) is
//    rounded to 16 bits and written back with tcgen05.st over the first 64
//    columns of S (two keys per column).  Tiles wholly below every row's
//    causal limit take an unmasked path.  The running maximum m moves only
//    when a tile's maximum exceeds it by more than 2^8, so O is rescaled in
//    TMEM (tcgen05.ld, scale, tcgen05.st) rarely and P stays below 2^8.  At the
//    item's end O is read from TMEM, divided by the row sum and stored.  A bf16
//    P keeps 8 significant bits; on tiles whose first row has fewer than 256
//    keys (where a few keys whose V terms cancel can carry the whole row) a
//    second product with P's rounding residual restores about 16.
//  * V rows past a context are zeroed in shared memory before use (unwritten
//    slots may hold NaN); blocks past the table's used entries and out-of-pool
//    ids load as zeros from outside the tensor map.  Every wait is bounded.
//  * Launches in which every sequence's rows fit one tile (speculative
//    verification: a few draft tokens times the group) run the split mode
//    further down instead: one query tile per (sequence, KV head), the key
//    tiles of all of them cut into equal shares over the CTAs, double-buffered
//    S, both softmax warpgroups on every tile, partials folded across CTAs.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "pa.h"
#include "pa_common.cuh"

namespace {

constexpr int kM = 128;             // query rows per tile = TMEM lanes
constexpr int kN = 128;             // keys per key tile
constexpr int kD = 128;             // head dim
constexpr int kTiles = 2;           // query tiles per item, one per softmax warpgroup
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kThreads = 384;       // warps 0 Q/K TMA, 1 MMA, 2 V TMA, 3 idle, 4-11 softmax
constexpr uint32_t kTmemCols = 512; // tile w: S/P at 256 w, O at 256 w + 128
constexpr int kMaxBatch = 4096;
constexpr int kResidualKeys = 256;
constexpr float kRescaleLog2 = 8.f; // move the running max only when it grows by more
constexpr uint64_t kWaitLimitNs = 1ull << 30;
constexpr float kLog2e = 1.4426950408889634f;

constexpr uint32_t kTileBytes = kM * kD * 2;   // 32 KB: a Q tile, one K or V stage
constexpr uint32_t kHalfBytes = kTileBytes / 2;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTiles * kTileBytes;
constexpr uint32_t kOffV = kOffK + kKStages * kTileBytes;
constexpr uint32_t kOffBar = kOffV + kVStages * kTileBytes;
constexpr int kNumBars = 26;
constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;      // TMEM base, dead flag
constexpr uint32_t kOffPrefix = kOffMisc + 16;             // [B + 1] int32 items

__host__ __device__ constexpr uint32_t smem_total(int B) {
    return 1024 + kOffPrefix + (uint32_t)(B + 1) * 4;
}

// mbarrier slots; the per-tile ones come in pairs (tile w at + w)
enum : int {
    kQFull = 0, kQEmpty = 1, kKFull = 2, kKEmpty = 4, kVFull = 6, kVEmpty = 8,
    kSFull = 10, kPFull = 12, kPvDone = 14, kOFree = 16, kDrain = 18,
    kQFull1 = 20, kQEmpty1 = 21,   // the split mode's second Q stage
    kAll8 = 19,                    // the split mode's eight softmax warps meet
    kXch = 22                      // the split mode's row-quarter pair exchanges (+ quarter)
};

struct Params {
    const int32_t* q_start;
    uint16_t* out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    unsigned int* err;
    int32_t max_blocks, B, H, Hkv, G, log_g, bs, num_blocks;
    float scale_log2;
};

__device__ __forceinline__ int32_t clamp_len(int32_t n, int32_t cap) {
    return n < 0 ? 0 : (n > cap ? cap : n);
}

struct Item {
    int32_t i, g;
    int32_t n, qlen, q0;     // context, queries, first query row of the sequence
    int32_t t0[kTiles];      // first token of query tile w (within the queries)
    int32_t tok[kTiles];     // its tokens (0: no tile w in this item)
    int32_t nkt[kTiles];     // its 128-key tiles
    int32_t nkt_all;         // key tiles loaded for the item (tile 1 has the later tokens)
    bool residual[kTiles];   // second P V product with P's rounding residual
};

__device__ __forceinline__ int32_t pairs_of(int32_t qlen, int32_t tm) {
    return ((qlen + tm - 1) / tm + 1) / 2;
}

// The w-th item of the flattened list: sequence i by the item prefix, then
// (tile pair descending, KV head).
template <bool kBF16>
__device__ __forceinline__ Item item_at(const Params& p, const int32_t* prefix, int32_t w) {
    int32_t lo = 0, hi = p.B;   // largest i with prefix[i] <= w
    while (hi - lo > 1) {
        const int32_t mid = (lo + hi) >> 1;
        if (prefix[mid] <= w) lo = mid; else hi = mid;
    }
    Item it;
    it.i = lo;
    const int32_t local = w - prefix[lo];
    const int32_t pairs = (prefix[lo + 1] - prefix[lo]) / p.Hkv;
    const int32_t pair = pairs - 1 - local / p.Hkv;
    it.g = local - (local / p.Hkv) * p.Hkv;
    it.n = clamp_len(__ldg(p.context_lens + lo), p.max_blocks * p.bs);
    it.q0 = __ldg(p.q_start + lo);
    it.qlen = __ldg(p.q_start + lo + 1) - it.q0;
    const int32_t tm = kM >> p.log_g;
#pragma unroll
    for (int w2 = 0; w2 < kTiles; ++w2) {
        it.t0[w2] = (2 * pair + w2) * tm;
        it.tok[w2] = max(0, min(tm, it.qlen - it.t0[w2]));
        const int32_t kmax = it.n - it.qlen + it.t0[w2] + it.tok[w2];   // last row's keys
        it.nkt[w2] = it.tok[w2] > 0 ? (kmax + kN - 1) / kN : 0;
        it.residual[w2] =
            kBF16 && it.tok[w2] > 0 && (it.n - it.qlen + it.t0[w2] + 1 < kResidualKeys);
    }
    it.nkt_all = max(it.nkt[0], it.nkt[1]);
    return it;
}

// This CTA's r-th item: rounds of gridDim.x items, dealt forwards in even
// rounds and backwards in odd ones.
__device__ __forceinline__ int32_t cta_item(int32_t r) {
    const int32_t C = gridDim.x, c = blockIdx.x;
    return r * C + ((r & 1) ? C - 1 - c : c);
}

// Bounded wait of one thread; a wait that runs out marks the CTA dead, and
// every later wait then fails at once, so all roles wind down.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* dead) {
    if (*dead) return false;
    if (pa::mbar_wait(bar, parity, kWaitLimitNs)) return true;
    *dead = 1;
    return false;
}

// The same for a whole warp, with one outcome for all lanes (the warp's
// tcgen05.ld / st are warp-collective).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* dead) {
    const bool ok = __all_sync(0xffffffffu, wait_bar(bar, parity, dead));
    if (!ok) *dead = 1;
    return ok;
}

// One TMA producer warp's walk over the key tiles of the CTA's items: per
// key tile, 16 boxes of 8 keys x both halves into `stages` ring slots of
// 32 KB (key group q of the tile at 2048 q: [half][8 rows][128 B]).  The Q
// tiles of each item are loaded first when `with_q`.
template <bool kBF16>
__device__ __forceinline__ void produce(const Params& p, const int32_t* prefix, int32_t W,
                                        const CUtensorMap* map, const CUtensorMap* qmap,
                                        bool with_q, unsigned char* smem, uint32_t ring_off,
                                        uint64_t* full, uint64_t* empty, int stages,
                                        uint64_t* bar, volatile int* dead, int lane) {
    const uint64_t kv_policy = pa::l2_policy_evict_last();  // re-read by the group's tiles
    const uint64_t q_policy = pa::l2_policy_evict_first();
    const int32_t oob_row = p.num_blocks * p.bs;
    const int32_t nb_shift = 31 - __clz(p.bs);   // block size 8, 16 or 32
    const int32_t bpt = kN >> nb_shift;           // blocks per key tile (<= 16)
    uint32_t kt = 0;   // key tiles issued
    int32_t r = 0, q_issued = 0;
    for (;; ++r) {
        const int32_t w = cta_item(r);
        if (w >= W) break;
        const Item it = item_at<kBF16>(p, prefix, w);
        if (with_q) {
            if (r > 0 && !warp_wait(&bar[kQEmpty], (uint32_t)((r - 1) & 1), dead)) break;
            if (lane == 0) {
                pa::mbar_arrive_expect_tx(&bar[kQFull],
                                          (it.tok[1] > 0 ? 2u : 1u) * kTileBytes);
                for (int t = 0; t < kTiles; ++t)
                    if (it.tok[t] > 0)
                        for (int h = 0; h < 2; ++h)
                            pa::tma_load_4d(smem + kOffQ + t * kTileBytes + h * kHalfBytes, qmap,
                                            &bar[kQFull], 0, it.g * p.G, it.q0 + it.t0[t], h,
                                            q_policy);
            }
            q_issued = r + 1;
        }
        const int32_t* trow = p.block_tables + (int64_t)it.i * p.max_blocks;
        const int32_t nblk = (it.n + p.bs - 1) >> nb_shift;   // table entries in use
        // lane l holds table entry j * bpt + l of key tile j; a used entry that
        // is not a pool block is flagged and read as zeros
        auto entry = [&](int32_t j) {
            const int32_t jb = j * bpt + lane;
            if (lane >= bpt || jb >= nblk) return -1;
            const int32_t e = __ldg(trow + jb);
            if (e < 0 || e >= p.num_blocks) {
                pa::raise_error(p.err, PA_DEVERR_BLOCK_ID);
                return -1;
            }
            return e;
        };
        int32_t blk = entry(0);
        bool ok_all = true;
        for (int32_t j = 0; j < it.nkt_all; ++j) {
            const int32_t blk_next = j + 1 < it.nkt_all ? entry(j + 1) : -1;
            int32_t rows[16];
#pragma unroll
            for (int q8 = 0; q8 < 16; ++q8) {
                const int32_t e = __shfl_sync(0xffffffffu, blk, (q8 * 8) >> nb_shift);
                rows[q8] = e >= 0 ? e * p.bs + ((q8 * 8) & (p.bs - 1)) : oob_row;
            }
            const uint32_t st = kt % stages;
            if (kt >= (uint32_t)stages &&
                !warp_wait(&empty[st], (kt / stages - 1) & 1, dead)) {
                ok_all = false;
                break;
            }
            if (lane == 0) {
                pa::mbar_arrive_expect_tx(&full[st], kTileBytes);
                unsigned char* dst = smem + ring_off + st * kTileBytes;
#pragma unroll
                for (int q8 = 0; q8 < 16; ++q8)
                    pa::tma_load_3d(dst + q8 * 2048, map, &full[st], 0, rows[q8], it.g * 2,
                                    kv_policy);
            }
            ++kt;
            __syncwarp();
            blk = blk_next;
        }
        if (!ok_all) break;
    }
    if (*dead && lane == 0) pa::raise_error(p.err, PA_DEVERR_TIMEOUT);
    // Drain: every load issued has landed before the CTA may exit.
    if (q_issued > 0)
        pa::mbar_wait(&bar[kQFull], (uint32_t)((q_issued - 1) & 1), kWaitLimitNs);
    for (uint32_t u = kt > (uint32_t)stages ? kt - stages : 0; u < kt; ++u)
        pa::mbar_wait(&full[u % stages], (u / stages) & 1, kWaitLimitNs);
}

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
multi_query_tc_kernel(const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const Params p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
    volatile int* dead = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + kOffPrefix);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t B = p.B;
    const int32_t max_len = p.max_blocks * p.bs;

    // ---- item prefix: prefix[i] = Hkv * sum_{i' < i} (tile pairs of i'), by
    // warp 0 (lane l sums a contiguous slice of the sequences, then a scan)
    if (warp == 0) {
        const int32_t tm = kM >> p.log_g;
        const int32_t per = (B + 31) / 32;
        const int32_t beg = min(lane * per, B), end = min(beg + per, B);
        auto items_of = [&](int32_t i, bool flag) {
            const int32_t raw = __ldg(p.context_lens + i);
            const int32_t n = clamp_len(raw, max_len);
            const int32_t ql = __ldg(p.q_start + i + 1) - __ldg(p.q_start + i);
            if (flag && blockIdx.x == 0) {
                if (raw > max_len) pa::raise_error(p.err, PA_DEVERR_TABLE_WIDTH);
                if (raw < 0 || ql < 0 || ql > n) pa::raise_error(p.err, PA_DEVERR_CONTEXT);
            }
            return (ql > 0 && ql <= n) ? p.Hkv * pairs_of(ql, tm) : 0;
        };
        int32_t local = 0;
        for (int32_t i = beg; i < end; ++i) local += items_of(i, true);
        int32_t x = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        int32_t run = x - local;
        for (int32_t i = beg; i < end; ++i) {
            prefix[i] = run;
            run += items_of(i, false);
        }
        if (lane == 31) prefix[B] = x;
    }
    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) pa::mbar_init(&bar[b], 1);
        pa::mbar_init(&bar[kPFull], 4);
        pa::mbar_init(&bar[kPFull + 1], 4);
        pa::mbar_init(&bar[kOFree], 4);
        pa::mbar_init(&bar[kOFree + 1], 4);
        pa::fence_barrier_init();
        *dead = 0;
    }
    __syncthreads();
    const int32_t W = prefix[B];
    if ((int32_t)blockIdx.x >= W) return;   // no item for this CTA: no TMEM taken
    if (warp == 1) {
        pa::tmem_alloc(tmem_slot, kTmemCols);
        pa::tmem_relinquish();
    }
    pa::tc_fence_before();
    __syncthreads();
    pa::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ====================== TMA producer: Q tiles and K ======================
        if (lane == 0) {
            pa::prefetch_tensormap(&qmap);
            pa::prefetch_tensormap(&kmap);
        }
        produce<kBF16>(p, prefix, W, &kmap, &qmap, true, smem, kOffK, &bar[kKFull],
                       &bar[kKEmpty], kKStages, bar, dead, lane);
    } else if (warp == 2) {
        // =========================== TMA producer: V ============================
        if (lane == 0) pa::prefetch_tensormap(&vmap);
        produce<kBF16>(p, prefix, W, &vmap, &qmap, false, smem, kOffV, &bar[kVFull],
                       &bar[kVEmpty], kVStages, bar, dead, lane);
    } else if (warp == 1) {
        // ============================ MMA issuer ============================
        if (lane == 0) {
            constexpr uint32_t idS = pa::idesc_f16(kBF16, false, kM, kN);
            constexpr uint32_t idPV = pa::idesc_f16(kBF16, true, kM, kD);
            const uint32_t sQ = pa::smem_addr(smem + kOffQ);
            const uint32_t sK = pa::smem_addr(smem + kOffK);
            const uint32_t sV = pa::smem_addr(smem + kOffV);
            uint32_t kc = 0, vc = 0;          // K / V tiles consumed
            uint32_t pc[kTiles] = {0, 0};     // P hand-overs consumed per tile
            uint32_t oc[kTiles] = {0, 0};     // items whose O tile w was used
            bool alive = true;
            auto s_mma = [&](int w, uint32_t kb) {   // S_w = Q_w K^T
                const uint32_t qb = sQ + w * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    // A = Q rows x dims 16 kk ..: K-major, half kk / 4
                    const uint64_t a =
                        pa::smem_desc_sw128(qb + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
                    // B = K keys x dims 16 kk ..: K-major, 8-key groups 2048 B
                    // apart, half kk / 4 at + 1024
                    const uint64_t b =
                        pa::smem_desc_sw128(kb + (kk >> 2) * 1024 + (kk & 3) * 32, 16, 2048);
                    pa::umma_f16(tmem + w * 256, a, b, idS, kk > 0 ? 1u : 0u);
                }
                pa::umma_commit(&bar[kSFull + w]);
            };
            auto pv_mma = [&](int w, uint32_t vb, bool accumulate) {   // O_w += P_w V
#pragma unroll
                for (int kk = 0; kk < kN / 16; ++kk) {
                    // B = V keys 16 kk .. x head dim: MN-major, two 8-key groups
                    // of 2048 B, halves 1024 B apart
                    const uint64_t b = pa::smem_desc_sw128(vb + kk * 4096, 1024, 2048);
                    // A = P rows x keys 16 kk ..: 8 TMEM columns of key pairs
                    pa::umma_f16_tmem_a(tmem + w * 256 + 128, tmem + w * 256 + kk * 8, b, idPV,
                                        (accumulate || kk > 0) ? 1u : 0u);
                }
            };
            for (int32_t r = 0; alive; ++r) {
                const int32_t w = cta_item(r);
                if (w >= W) break;
                const Item it = item_at<kBF16>(p, prefix, w);
                if (!wait_bar(&bar[kQFull], (uint32_t)(r & 1), dead)) break;
                // S_w(0) of both tiles
                if (!wait_bar(&bar[kKFull + kc % kKStages], (kc / kKStages) & 1, dead)) break;
                pa::tc_fence_after();
                for (int t = 0; t < kTiles; ++t)
                    if (it.nkt[t] > 0) s_mma(t, sK + (kc % kKStages) * kTileBytes);
                pa::umma_commit(&bar[kKEmpty + kc % kKStages]);
                ++kc;
                for (int32_t j = 0; j < it.nkt_all && alive; ++j) {
                    bool v_ready = false, k_ready = false;
                    const uint32_t vb = sV + (vc % kVStages) * kTileBytes;
                    const uint32_t kb = sK + (kc % kKStages) * kTileBytes;
                    for (int t = 0; t < kTiles && alive; ++t) {
                        if (j < it.nkt[t]) {
                            // O_t of the previous item must have been read out
                            if (j == 0 && oc[t] > 0 &&
                                !wait_bar(&bar[kOFree + t], (oc[t] - 1) & 1, dead)) {
                                alive = false;
                                break;
                            }
                            if (!wait_bar(&bar[kPFull + t], pc[t] & 1, dead)) {
                                alive = false;
                                break;
                            }
                            ++pc[t];
                            if (!v_ready) {
                                if (!wait_bar(&bar[kVFull + vc % kVStages], (vc / kVStages) & 1,
                                              dead)) {
                                    alive = false;
                                    break;
                                }
                                v_ready = true;
                            }
                            pa::tc_fence_after();
                            pv_mma(t, vb, j > 0);
                            if (it.residual[t]) {
                                pa::umma_commit(&bar[kPvDone + t]);   // P's high part read
                                if (!wait_bar(&bar[kPFull + t], pc[t] & 1, dead)) {
                                    alive = false;
                                    break;
                                }
                                ++pc[t];
                                pa::tc_fence_after();
                                pv_mma(t, vb, true);
                            }
                            pa::umma_commit(&bar[kPvDone + t]);
                        }
                        if (j + 1 < it.nkt[t]) {
                            if (!k_ready) {
                                if (!wait_bar(&bar[kKFull + kc % kKStages], (kc / kKStages) & 1,
                                              dead)) {
                                    alive = false;
                                    break;
                                }
                                k_ready = true;
                                pa::tc_fence_after();
                            }
                            s_mma(t, kb);
                        }
                    }
                    if (!alive) break;
                    pa::umma_commit(&bar[kVEmpty + vc % kVStages]);
                    ++vc;
                    if (k_ready) {
                        pa::umma_commit(&bar[kKEmpty + kc % kKStages]);
                        ++kc;
                    }
                }
                if (!alive) break;
                for (int t = 0; t < kTiles; ++t)
                    if (it.nkt[t] > 0) ++oc[t];
                pa::umma_commit(&bar[kQEmpty]);   // every S of the item done: Q is free
            }
            // Drain: every MMA issued has completed before TMEM is released.
            pa::umma_commit(&bar[kDrain]);
            pa::mbar_wait(&bar[kDrain], 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ============================== softmax ==============================
        const int wt = (warp - 4) >> 2;          // the query tile of this warpgroup
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const uint32_t sp_col = lane_base + wt * 256;   // S / P
        const uint32_t o_col = sp_col + 128;
        const float c2 = p.scale_log2;
        uint32_t sc = 0;     // S tiles of this warpgroup so far
        uint32_t pvc = 0;    // commits on kPvDone + wt waited for so far
        uint32_t vbase = 0;  // key tiles of the CTA's earlier items (V ring position)
        // Waits for the next commit on this tile's kPvDone: every commit is
        // waited for once and in order (key tile j waits for the product of
        // tile j - 1 after it has computed its own P), so the parity wait is
        // always one phase ahead.
        auto wait_pv = [&]() {
            const bool ok = warp_wait(&bar[kPvDone + wt], pvc & 1, dead);
            ++pvc;
            return ok;
        };
        for (int32_t r = 0;; ++r) {
            const int32_t w = cta_item(r);
            if (w >= W) break;
            const Item it = item_at<kBF16>(p, prefix, w);
            const uint32_t vb0 = vbase;
            vbase += it.nkt_all;
            if (it.nkt[wt] == 0) continue;   // no tile for this warpgroup in the item
            const bool valid = row < (it.tok[wt] << p.log_g);
            const int32_t lim_min = it.n - it.qlen + it.t0[wt];   // the tile's first row
            const int32_t lim = valid ? lim_min + (row >> p.log_g) : -1;
            const bool residual = it.residual[wt];
            float m_used = -INFINITY, l = 0.f;
            bool ok = true;
            for (int32_t j = 0; j < it.nkt[wt]; ++j) {
                if (!warp_wait(&bar[kSFull + wt], sc & 1, dead)) {
                    ok = false;
                    break;
                }
                ++sc;
                pa::tc_fence_after();
                const int32_t key0 = j * kN;
                // tiles wholly below every row's causal limit need no mask
                const bool full = key0 + kN - 1 <= lim_min;
                // pass 1: the row's largest unmasked score
                float mx = -INFINITY;
                if (full) {
#pragma unroll 1
                    for (int c = 0; c < 4; c += 2) {
                        uint32_t s0[32], s1[32];
                        pa::tmem_ld32(sp_col + c * 32, s0);
                        pa::tmem_ld32(sp_col + c * 32 + 32, s1);
                        pa::tmem_ld_wait();
                        pa::reg_fence32(s0);
                        pa::reg_fence32(s1);
                        float m2[2] = {mx, -INFINITY};
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            m2[0] = fmaxf(m2[0], __uint_as_float(s0[e]));
                            m2[1] = fmaxf(m2[1], __uint_as_float(s1[e]));
                        }
                        mx = fmaxf(m2[0], m2[1]);
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t s[32];
                        pa::tmem_ld32(sp_col + c * 32, s);
                        pa::tmem_ld_wait();
                        pa::reg_fence32(s);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (key0 + c * 32 + e <= lim) mx = fmaxf(mx, __uint_as_float(s[e]));
                    }
                }
                mx *= c2;   // base-2 logit (scale > 0)
                const bool grow = mx > m_used + kRescaleLog2;   // false for -inf
                const float m_new = grow ? mx : m_used;
                const float base = m_new == -INFINITY ? 0.f : m_new;
                // pass 2: P = 2^(s c2 - m) rounded to 16 bits, stored over S's
                // first 64 columns as it goes (keys 64 h .. read before written)
                float lsum = 0.f;
                uint32_t rl[64];   // bf16 P's rounding residual (residual tiles only)
                if (full && !residual) {
                    // unmasked tiles: straight-line math, no per-key branches
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t s0[32], s1[32];
                        pa::tmem_ld32(sp_col + hh * 64, s0);
                        pa::tmem_ld32(sp_col + hh * 64 + 32, s1);
                        pa::tmem_ld_wait();
                        pa::reg_fence32(s0);
                        pa::reg_fence32(s1);
                        uint32_t pk[32];
                        float la = 0.f, lb = 0.f;
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float p0 = pa::fast_exp2(fmaf(__uint_as_float(s0[e]), c2, -base));
                            const float p1 =
                                pa::fast_exp2(fmaf(__uint_as_float(s0[e + 1]), c2, -base));
                            const float p2 = pa::fast_exp2(fmaf(__uint_as_float(s1[e]), c2, -base));
                            const float p3 =
                                pa::fast_exp2(fmaf(__uint_as_float(s1[e + 1]), c2, -base));
                            la += p0 + p1;
                            lb += p2 + p3;
                            pk[e >> 1] = pa::pack2<kBF16>(p0, p1);
                            pk[16 + (e >> 1)] = pa::pack2<kBF16>(p2, p3);
                        }
                        lsum += la + lb;
                        pa::tmem_st32(sp_col + hh * 32, pk);
                    }
                } else {
                    // the causal edge, the context's end, residual tiles
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t s0[32], s1[32];
                        pa::tmem_ld32(sp_col + hh * 64, s0);
                        pa::tmem_ld32(sp_col + hh * 64 + 32, s1);
                        pa::tmem_ld_wait();
                        pa::reg_fence32(s0);
                        pa::reg_fence32(s1);
                        uint32_t pk[32];
                        float la = 0.f, lb = 0.f;
                        const int32_t kl = lim - key0 - hh * 64;   // keys 0 .. kl of this half
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            float p0 = pa::fast_exp2(fmaf(__uint_as_float(s0[e]), c2, -base));
                            float p1 = pa::fast_exp2(fmaf(__uint_as_float(s0[e + 1]), c2, -base));
                            float p2 = pa::fast_exp2(fmaf(__uint_as_float(s1[e]), c2, -base));
                            float p3 = pa::fast_exp2(fmaf(__uint_as_float(s1[e + 1]), c2, -base));
                            p0 = e <= kl ? p0 : 0.f;
                            p1 = e + 1 <= kl ? p1 : 0.f;
                            p2 = e + 32 <= kl ? p2 : 0.f;
                            p3 = e + 33 <= kl ? p3 : 0.f;
                            la += p0 + p1;
                            lb += p2 + p3;
                            const uint32_t h01 = pa::pack2<kBF16>(p0, p1);
                            const uint32_t h23 = pa::pack2<kBF16>(p2, p3);
                            pk[e >> 1] = h01;
                            pk[16 + (e >> 1)] = h23;
                            rl[hh * 32 + (e >> 1)] = pa::bf16x2_residual(h01, p0, p1);
                            rl[hh * 32 + 16 + (e >> 1)] = pa::bf16x2_residual(h23, p2, p3);
                        }
                        lsum += la + lb;
                        pa::tmem_st32(sp_col + hh * 32, pk);
                    }
                }
                // The previous key tile's product done (O holds every earlier
                // tile) before O moves to the new maximum; P V of this tile is
                // only issued after the hand-over below.
                if (j >= 1) {
                    if (!wait_pv()) {
                        ok = false;
                        break;
                    }
                    pa::tc_fence_after();
                    if (__any_sync(0xffffffffu, grow)) {
                        const float f = grow ? pa::fast_exp2(m_used - m_new) : 1.f;
                        l *= f;
#pragma unroll 1
                        for (int c = 0; c < 4; ++c) {
                            uint32_t o[32];
                            pa::tmem_ld32(o_col + c * 32, o);
                            pa::tmem_ld_wait();
                            pa::reg_fence32(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                            pa::tmem_st32(o_col + c * 32, o);
                        }
                    }
                }
                pa::tmem_st_wait();
                m_used = m_new;
                // l sums the fp32 P (rows of unmasked tiles have 256+ keys and
                // the others carry P's residual, so rounding does not bias l)
                l += lsum;
                // The last key tile may reach past the context: zero those V
                // rows (both halves) once the tile has landed -- by the first
                // warpgroup whose tile reads it.
                if (key0 + kN > it.n && (wt == 0 || j >= it.nkt[0])) {
                    const uint32_t vt = vb0 + j;
                    const uint32_t vs = vt % kVStages;
                    if (!warp_wait(&bar[kVFull + vs], (vt / kVStages) & 1, dead)) {
                        ok = false;
                        break;
                    }
                    if (key0 + row >= it.n) {
                        unsigned char* vrow = smem + kOffV + vs * kTileBytes +
                                              (uint32_t)(row >> 3) * 2048 + (uint32_t)(row & 7) * 128;
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                            for (int c16 = 0; c16 < 8; ++c16)
                                *reinterpret_cast<uint4*>(vrow + hf * 1024 + c16 * 16) =
                                    make_uint4(0, 0, 0, 0);
                    }
                    pa::fence_proxy_async_smem();
                }
                pa::tc_fence_before();
                __syncwarp();
                if (lane == 0) pa::mbar_arrive(&bar[kPFull + wt]);
                if (residual) {
                    // second product: P's rounding residual, once the first is read
                    if (!wait_pv()) {
                        ok = false;
                        break;
                    }
                    pa::tc_fence_after();
                    uint32_t a[32], b[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        a[e] = rl[e];
                        b[e] = rl[32 + e];
                    }
                    pa::tmem_st32(sp_col, a);
                    pa::tmem_st32(sp_col + 32, b);
                    pa::tmem_st_wait();
                    pa::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) pa::mbar_arrive(&bar[kPFull + wt]);
                }
            }
            if (!ok) break;
            // ---- epilogue: O / l, once the last product is done
            if (!wait_pv()) break;
            pa::tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int32_t t = it.t0[wt] + (row >> p.log_g);
            const int32_t hq = it.g * p.G + (row & (p.G - 1));
            uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)(it.q0 + t) * p.H + hq) * kD);
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                pa::tmem_ld32(o_col + c * 32, o);
                pa::tmem_ld_wait();
                pa::reg_fence32(o);
                if (valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 v;
                        v.x = pa::pack2<kBF16>(__uint_as_float(o[e]) * inv,
                                               __uint_as_float(o[e + 1]) * inv);
                        v.y = pa::pack2<kBF16>(__uint_as_float(o[e + 2]) * inv,
                                               __uint_as_float(o[e + 3]) * inv);
                        v.z = pa::pack2<kBF16>(__uint_as_float(o[e + 4]) * inv,
                                               __uint_as_float(o[e + 5]) * inv);
                        v.w = pa::pack2<kBF16>(__uint_as_float(o[e + 6]) * inv,
                                               __uint_as_float(o[e + 7]) * inv);
                        dst[(c * 32 + e) >> 3] = v;
                    }
                }
            }
            pa::tc_fence_before();
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(&bar[kOFree + wt]);
        }
        if (*dead && row == 0) pa::raise_error(p.err, PA_DEVERR_TIMEOUT);
    }
    pa::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        pa::tc_fence_after();
        pa::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---- one query tile per (sequence, KV head): the split mode -------------------------
// Launches in which every sequence's rows fit one 128-row tile (max_q_len * G
// <= 128: speculative verification, decode-like batches; any G up to 128)
// split the work like the decode: the flattened list of (sequence i, KV head g,
// 128-key tile) is cut into equal contiguous shares over the CTAs.  Every key
// tile's scores land in one of two S buffers in TMEM, so the next tile's are
// computed while this one is worked on; the two softmax warpgroups take one
// half of the tile's keys each (trading row maxima through shared memory)
// and, at a segment's end, one half of O, which alternates between two TMEM
// buffers so that the next segment's products need not wait for the store.
// A pair split between CTAs leaves its (M, L, O) rows in one of the CTA's two
// workspace slots; the last CTA to finish the pair -- an acquire-release
// ticket, never a wait -- folds them.

constexpr int kMinTilesPerCta = 2;
// Work units a (sequence, KV head) pair costs beyond its key tiles (the
// segment's start and end: pipeline refill, the last product's latency), so
// a share of many short pairs gets fewer tiles.  The units sit before the
// pair's first tile on the flattened line the CTAs split evenly.
constexpr int kPairUnits = 4;
constexpr int kFoldRows = 8;   // rows a warp folds at once
// TMEM: two S / P buffers of 128 key columns, then two O buffers of d columns
// (segment r accumulates in O buffer r % 2: the next segment's first
// products need not wait for this one's read-out)
constexpr uint32_t kSBufCols = kN;
constexpr uint32_t kOCol = 2 * kSBufCols;
constexpr uint32_t kSOffQ = 0;                                   // two Q stages
constexpr uint32_t kSOffK = kSOffQ + 2 * kTileBytes;
constexpr uint32_t kSOffV = kSOffK + kKStages * kTileBytes;
constexpr uint32_t kSOffRow = kSOffV + kVStages * kTileBytes;   // warpgroup exchanges, fold values
constexpr uint32_t kSOffBar = kSOffRow + 6 * kM * 4;
constexpr uint32_t kSOffMisc = kSOffBar + kNumBars * 8;   // TMEM base, dead flag, flags per warpgroup
constexpr uint32_t kSOffPrefix = kSOffMisc + 32;
constexpr size_t kSlotFloats = (size_t)kM * (kD + 2);            // O rows, then M, then L

__host__ __device__ constexpr uint32_t split_smem_total(int B) {
    return 1024 + kSOffPrefix + (uint32_t)(B + 1) * 4;
}

struct SParams {
    const int32_t* q_start;
    uint16_t* out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t* counters;   // [B * Hkv] tickets of split pairs
    float* partials;     // [2 * gridDim.x] slots of kSlotFloats
    unsigned int* err;
    int32_t max_blocks, B, H, Hkv, G, tm, bs, num_blocks, max_q_len;
    float scale_log2;
};

struct SSeg {
    int32_t i, g, kt0, len, nkt;
    int32_t a;      // the pair's first unit on the flattened line (its tile 0 at a + kPairUnits)
    int32_t next;   // the line position after the segment
    int32_t n, qlen, q0;
};

__device__ __forceinline__ int32_t s_begin(int64_t c, int64_t F, int64_t C) {
    return (int32_t)(c * F / C);
}

// The segment of the share [pos, hi) that begins at the first key tile at or
// after pos (len = 0: no tile left in the share).
__device__ __forceinline__ SSeg s_segment(const SParams& p, const int32_t* prefix, int32_t pos,
                                          int32_t hi) {
    int32_t lo = 0, hb = p.B;   // largest i with prefix[i] <= pos
    while (hb - lo > 1) {
        const int32_t mid = (lo + hb) >> 1;
        if (prefix[mid] <= pos) lo = mid; else hb = mid;
    }
    SSeg s;
    s.i = lo;
    const int32_t units = (prefix[lo + 1] - prefix[lo]) / p.Hkv;
    s.nkt = units - kPairUnits;
    const int32_t local = pos - prefix[lo];
    s.g = local / units;
    s.a = prefix[lo] + s.g * units;
    const int32_t start = max(pos, s.a + kPairUnits);
    s.kt0 = start - s.a - kPairUnits;
    s.len = max(0, min(hi - start, s.nkt - s.kt0));
    s.next = start + s.len;
    s.n = clamp_len(__ldg(p.context_lens + lo), p.max_blocks * p.bs);
    s.q0 = __ldg(p.q_start + lo);
    s.qlen = __ldg(p.q_start + lo + 1) - s.q0;
    return s;
}

// A TMA producer warp's walk over its CTA's share: per segment (the Q tile
// first when with_q), the key tiles kt0 .. kt0 + len - 1 of pair (i, g).
__device__ __forceinline__ void s_produce(const SParams& p, const int32_t* prefix, int32_t lo,
                                          int32_t hi, const CUtensorMap* map,
                                          const CUtensorMap* qmap, bool with_q,
                                          unsigned char* smem, uint32_t ring_off, uint64_t* full,
                                          uint64_t* empty, int stages, uint64_t* bar,
                                          volatile int* dead, int lane) {
    const uint64_t kv_policy = pa::l2_policy_evict_first();   // streamed once
    const uint64_t q_policy = pa::l2_policy_evict_first();
    const int32_t oob_row = p.num_blocks * p.bs;
    const int32_t nb_shift = 31 - __clz(p.bs);
    const int32_t bpt = kN >> nb_shift;
    uint32_t kt = 0;
    int32_t r = 0, q_issued = 0;
    for (int32_t pos = lo; pos < hi; ++r) {
        const SSeg sg = s_segment(p, prefix, pos, hi);
        if (sg.len == 0) break;
        pos = sg.next;
        if (with_q) {
            // Q stage r % 2: the next segment's Q travels while this one computes
            const int qs = r & 1;
            uint64_t* qfull = &bar[qs ? kQFull1 : kQFull];
            if (r >= 2 && !warp_wait(&bar[qs ? kQEmpty1 : kQEmpty], (uint32_t)(((r >> 1) - 1) & 1),
                                     dead))
                break;
            if (lane == 0) {
                // two boxes of tm tokens x G heads x 128 bytes (126 rows for G = 7;
                // the tile's last rows then keep stale values, never stored)
                pa::mbar_arrive_expect_tx(qfull, 2u * p.tm * p.G * 128u);
                for (int h = 0; h < 2; ++h)
                    pa::tma_load_4d(smem + kSOffQ + qs * kTileBytes + h * kHalfBytes, qmap, qfull,
                                    0, sg.g * p.G, sg.q0, h, q_policy);
            }
            q_issued = r + 1;
        }
        const int32_t* trow = p.block_tables + (int64_t)sg.i * p.max_blocks;
        const int32_t nblk = (sg.n + p.bs - 1) >> nb_shift;
        auto entry = [&](int32_t j) {
            const int32_t jb = j * bpt + lane;
            if (lane >= bpt || jb >= nblk) return -1;
            const int32_t e = __ldg(trow + jb);
            if (e < 0 || e >= p.num_blocks) {
                pa::raise_error(p.err, PA_DEVERR_BLOCK_ID);
                return -1;
            }
            return e;
        };
        int32_t blk = entry(sg.kt0);
        bool ok_all = true;
        for (int32_t j = 0; j < sg.len; ++j) {
            const int32_t blk_next = j + 1 < sg.len ? entry(sg.kt0 + j + 1) : -1;
            int32_t rows[16];
#pragma unroll
            for (int q8 = 0; q8 < 16; ++q8) {
                const int32_t e = __shfl_sync(0xffffffffu, blk, (q8 * 8) >> nb_shift);
                rows[q8] = e >= 0 ? e * p.bs + ((q8 * 8) & (p.bs - 1)) : oob_row;
            }
            const uint32_t st = kt % stages;
            if (kt >= (uint32_t)stages && !warp_wait(&empty[st], (kt / stages - 1) & 1, dead)) {
                ok_all = false;
                break;
            }
            if (lane == 0) {
                pa::mbar_arrive_expect_tx(&full[st], kTileBytes);
                unsigned char* dst = smem + ring_off + st * kTileBytes;
#pragma unroll
                for (int q8 = 0; q8 < 16; ++q8)
                    pa::tma_load_3d(dst + q8 * 2048, map, &full[st], 0, rows[q8], sg.g * 2,
                                    kv_policy);
            }
            ++kt;
            __syncwarp();
            blk = blk_next;
        }
        if (!ok_all) break;
    }
    if (*dead && lane == 0) pa::raise_error(p.err, PA_DEVERR_TIMEOUT);
    for (int32_t u = q_issued > 2 ? q_issued - 2 : 0; u < q_issued; ++u)
        pa::mbar_wait(&bar[(u & 1) ? kQFull1 : kQFull], (uint32_t)((u >> 1) & 1), kWaitLimitNs);
    for (uint32_t u = kt > (uint32_t)stages ? kt - stages : 0; u < kt; ++u)
        pa::mbar_wait(&full[u % stages], (u / stages) & 1, kWaitLimitNs);
}

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
multi_query_tc_split_kernel(const __grid_constant__ CUtensorMap qmap,
                            const __grid_constant__ CUtensorMap kmap,
                            const __grid_constant__ CUtensorMap vmap, const SParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kSOffBar);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSOffMisc);
    volatile int* dead = reinterpret_cast<volatile int*>(smem + kSOffMisc + 4);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + kSOffMisc + 8);
    float* xch = reinterpret_cast<float*>(smem + kSOffRow);   // [parity][warpgroup][128]
    float* fold_ml = xch + 4 * kM;                            // [max, 1 / sum][128]
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + kSOffPrefix);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t B = p.B;
    const int32_t max_len = p.max_blocks * p.bs;

    // ---- prefix of work units: prefix[i] = Hkv * sum_{i' < i} u_i', with
    // u = ceil(n / 128) + kPairUnits for a sequence with query rows and keys,
    // else 0; by warp 0 (lane l sums a contiguous slice, then a scan)
    if (warp == 0) {
        const int32_t per = (B + 31) / 32;
        const int32_t beg = min(lane * per, B), end = min(beg + per, B);
        auto tiles_of = [&](int32_t i, bool flag) {
            const int32_t raw = __ldg(p.context_lens + i);
            const int32_t n = clamp_len(raw, max_len);
            const int32_t ql = __ldg(p.q_start + i + 1) - __ldg(p.q_start + i);
            const bool bad = raw < 0 || ql < 0 || ql > n || ql > p.max_q_len;
            if (flag && blockIdx.x == 0) {
                if (raw > max_len) pa::raise_error(p.err, PA_DEVERR_TABLE_WIDTH);
                if (bad) pa::raise_error(p.err, PA_DEVERR_CONTEXT);
            }
            return (ql > 0 && !bad) ? p.Hkv * ((n + kN - 1) / kN + kPairUnits) : 0;
        };
        int32_t local = 0;
        for (int32_t i = beg; i < end; ++i) local += tiles_of(i, true);
        int32_t x = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        int32_t run = x - local;
        for (int32_t i = beg; i < end; ++i) {
            prefix[i] = run;
            run += tiles_of(i, false);
        }
        if (lane == 31) prefix[B] = x;
    }
    if (tid == 0) {
        for (int b = 0; b < kNumBars; ++b) pa::mbar_init(&bar[b], 1);
        for (int b = 0; b < 2; ++b) {
            pa::mbar_init(&bar[kPFull + b], 8);
            pa::mbar_init(&bar[kOFree + b], 8);
        }
        for (int q = 0; q < 4; ++q) pa::mbar_init(&bar[kXch + q], 2);
        pa::mbar_init(&bar[kAll8], 8);
        pa::fence_barrier_init();
        *dead = 0;
    }
    __syncthreads();
    const int64_t F = prefix[B];
    int64_t C = F / kMinTilesPerCta;
    if (C > (int64_t)gridDim.x) C = gridDim.x;
    if (C < 1) C = 1;
    if ((int64_t)blockIdx.x >= C || F == 0) return;   // no work: no TMEM taken
    const int32_t lo = s_begin(blockIdx.x, F, C), hi = s_begin(blockIdx.x + 1, F, C);
    if (warp == 1) {
        pa::tmem_alloc(tmem_slot, kTmemCols);
        pa::tmem_relinquish();
    }
    pa::tc_fence_before();
    __syncthreads();
    pa::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            pa::prefetch_tensormap(&qmap);
            pa::prefetch_tensormap(&kmap);
        }
        s_produce(p, prefix, lo, hi, &kmap, &qmap, true, smem, kSOffK, &bar[kKFull],
                  &bar[kKEmpty], kKStages, bar, dead, lane);
    } else if (warp == 2) {
        if (lane == 0) pa::prefetch_tensormap(&vmap);
        s_produce(p, prefix, lo, hi, &vmap, &qmap, false, smem, kSOffV, &bar[kVFull],
                  &bar[kVEmpty], kVStages, bar, dead, lane);
    } else if (warp == 1) {
        // ============================ MMA issuer ============================
        // Per segment: S(0) -> buffer 0, S(1) -> buffer 1, then for each key
        // tile j: PV(j) into the segment's O buffer (r % 2), and S(j + 2) into
        // buffer j % 2 -- after PV(j), which reads P(j) from those columns.
        if (lane == 0) {
            constexpr uint32_t idS = pa::idesc_f16(kBF16, false, kM, kN);
            constexpr uint32_t idPV = pa::idesc_f16(kBF16, true, kM, kD);
            const uint32_t sQ = pa::smem_addr(smem + kSOffQ);
            const uint32_t sK = pa::smem_addr(smem + kSOffK);
            const uint32_t sV = pa::smem_addr(smem + kSOffV);
            uint32_t kc = 0, vc = 0;
            uint32_t pc[2] = {0, 0};
            bool alive = true;
            auto s_mma = [&](int b, uint32_t qb) {   // S into buffer b for the next K tile
                if (!wait_bar(&bar[kKFull + kc % kKStages], (kc / kKStages) & 1, dead)) return false;
                pa::tc_fence_after();
                const uint32_t kb = sK + (kc % kKStages) * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                    const uint64_t a =
                        pa::smem_desc_sw128(qb + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd =
                        pa::smem_desc_sw128(kb + (kk >> 2) * 1024 + (kk & 3) * 32, 16, 2048);
                    pa::umma_f16(tmem + b * kSBufCols, a, bd, idS, kk > 0 ? 1u : 0u);
                }
                pa::umma_commit(&bar[kSFull + b]);
                pa::umma_commit(&bar[kKEmpty + kc % kKStages]);
                ++kc;
                return true;
            };
            auto pv_mma = [&](uint32_t o_tmem, int b, uint32_t vb, bool accumulate) {
#pragma unroll
                for (int kk = 0; kk < kN / 16; ++kk) {
                    const uint64_t bd = pa::smem_desc_sw128(vb + kk * 4096, 1024, 2048);
                    pa::umma_f16_tmem_a(o_tmem, tmem + b * kSBufCols + kk * 8, bd, idPV,
                                        (accumulate || kk > 0) ? 1u : 0u);
                }
            };
            int32_t r = 0;
            // the CTA's shares, grid-stride (C <= gridDim.x: one share)
            for (int32_t c = blockIdx.x; c < C && alive; c += gridDim.x) {
                const int32_t hi_c = s_begin(c + 1, F, C);
                for (int32_t pos = s_begin(c, F, C); pos < hi_c && alive; ++r) {
                const SSeg sg = s_segment(p, prefix, pos, hi_c);
                if (sg.len == 0) break;
                pos = sg.next;
                const bool residual =
                    kBF16 && (sg.n - sg.qlen + 1 < kResidualKeys);   // the first row's keys
                const int qs = r & 1;
                const uint32_t qb = sQ + qs * kTileBytes;
                const uint32_t o_tmem = tmem + kOCol + (uint32_t)(r & 1) * kD;
                if (!wait_bar(&bar[qs ? kQFull1 : kQFull], (uint32_t)((r >> 1) & 1), dead)) break;
                for (int b = 0; b < 2 && b < sg.len; ++b)
                    if (!s_mma(b, qb)) {
                        alive = false;
                        break;
                    }
                for (int32_t j = 0; j < sg.len && alive; ++j) {
                    const int b = j & 1;
                    // this O buffer's previous segment (r - 2) read out first
                    if (j == 0 && r >= 2 &&
                        !wait_bar(&bar[kOFree + (r & 1)], (uint32_t)(((r >> 1) - 1) & 1), dead)) {
                        alive = false;
                        break;
                    }
                    if (!wait_bar(&bar[kPFull + b], pc[b] & 1, dead)) {
                        alive = false;
                        break;
                    }
                    ++pc[b];
                    if (!wait_bar(&bar[kVFull + vc % kVStages], (vc / kVStages) & 1, dead)) {
                        alive = false;
                        break;
                    }
                    pa::tc_fence_after();
                    const uint32_t vb = sV + (vc % kVStages) * kTileBytes;
                    pv_mma(o_tmem, b, vb, j > 0);
                    if (residual) {
                        pa::umma_commit(&bar[kPvDone]);   // P's high part read
                        if (!wait_bar(&bar[kPFull + b], pc[b] & 1, dead)) {
                            alive = false;
                            break;
                        }
                        ++pc[b];
                        pa::tc_fence_after();
                        pv_mma(o_tmem, b, vb, true);
                    }
                    pa::umma_commit(&bar[kPvDone]);
                    pa::umma_commit(&bar[kVEmpty + vc % kVStages]);
                    ++vc;
                    if (j + 2 < sg.len && !s_mma(b, qb)) {
                        alive = false;
                        break;
                    }
                }
                if (!alive) break;
                pa::umma_commit(&bar[qs ? kQEmpty1 : kQEmpty]);
                }
            }
            pa::umma_commit(&bar[kDrain]);
            pa::mbar_wait(&bar[kDrain], 0, kWaitLimitNs);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ============================== softmax ==============================
        // Warpgroup h takes keys [64 h, 64 h + 64) of every tile (P columns
        // [32 h, 32 h + 32), O columns [64 h, 64 h + 64)); the two warps that
        // share a row quarter trade their row maxima once per tile and their
        // row sums once per segment.  At a segment's end both read their half
        // of O out and store it; for a split pair, the ticket and the fold.
        const int h = (warp - 4) >> 2;
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16);
        const float c2 = p.scale_log2;
        uint32_t sc[2] = {0, 0}, pvc = 0, xc = 0, ac = 0;
        uint32_t vbase = 0;   // key tiles of the share's earlier segments (V ring position)
        auto wait_pv = [&]() {
            const bool ok = warp_wait(&bar[kPvDone], pvc & 1, dead);
            ++pvc;
            return ok;
        };
        // this row's value from the other warpgroup (bounded pair barrier;
        // the slot's parity alternates, so a slot is rewritten only after the
        // partner has passed the next exchange, i.e. read this one)
        auto exchange = [&](float v, float& other) {
            float* slot = xch + (xc & 1) * 2 * kM;
            slot[h * kM + row] = v;
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(&bar[kXch + wq]);
            const bool ok = warp_wait(&bar[kXch + wq], xc & 1, dead);
            ++xc;
            other = slot[(h ^ 1) * kM + row];
            return ok;
        };
        auto all8 = [&]() {   // the eight softmax warps meet (bounded)
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(&bar[kAll8]);
            return warp_wait(&bar[kAll8], (ac++) & 1, dead);
        };
        int32_t r = 0;
        for (int32_t pos = lo; pos < hi; ++r) {
            const SSeg sg = s_segment(p, prefix, pos, hi);
            if (sg.len == 0) break;
            pos = sg.next;
            const uint32_t vb0 = vbase;
            vbase += (uint32_t)sg.len;
            const int32_t rows = sg.qlen * p.G;
            const bool valid = row < rows;
            const int32_t t_row = row / p.G;
            const int32_t lim_min = sg.n - sg.qlen;                 // the first row's limit
            const int32_t lim = valid ? lim_min + t_row : -1;
            const bool residual = kBF16 && (sg.n - sg.qlen + 1 < kResidualKeys);
            const uint32_t o_col = lane_base + kOCol + (uint32_t)(r & 1) * kD + h * 64;
            float m_used = -INFINITY, l = 0.f;
            bool ok = true;
            for (int32_t j = 0; j < sg.len; ++j) {
                const int b = j & 1;
                const uint32_t s_col = lane_base + b * kSBufCols + h * 64;   // this half's scores
                const uint32_t p_col = lane_base + b * kSBufCols + h * 32;   // this half's P pairs
                if (!warp_wait(&bar[kSFull + b], sc[b] & 1, dead)) {
                    ok = false;
                    break;
                }
                ++sc[b];
                pa::tc_fence_after();
                const int32_t key0 = (sg.kt0 + j) * kN + h * 64;   // this half's first key
                const bool full = key0 + 63 <= lim_min;
                uint32_t s0[32], s1[32];
                pa::tmem_ld32(s_col, s0);
                pa::tmem_ld32(s_col + 32, s1);
                pa::tmem_ld_wait();
                pa::reg_fence32(s0);
                pa::reg_fence32(s1);
                float mx = -INFINITY;
                if (full) {
                    float m2[2] = {-INFINITY, -INFINITY};
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        m2[0] = fmaxf(m2[0], __uint_as_float(s0[e]));
                        m2[1] = fmaxf(m2[1], __uint_as_float(s1[e]));
                    }
                    mx = fmaxf(m2[0], m2[1]);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        if (key0 + e <= lim) mx = fmaxf(mx, __uint_as_float(s0[e]));
                        if (key0 + 32 + e <= lim) mx = fmaxf(mx, __uint_as_float(s1[e]));
                    }
                }
                float mx_o;
                if (!exchange(mx, mx_o)) {
                    ok = false;
                    break;
                }
                mx = fmaxf(mx, mx_o) * c2;   // the same value in both warpgroups
                const bool grow = mx > m_used + kRescaleLog2;
                const float m_new = grow ? mx : m_used;
                const float base = m_new == -INFINITY ? 0.f : m_new;
                float lsum;
                uint32_t pk[32], rl[32];
                if (full && !residual) {
                    float la = 0.f, lb = 0.f;
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float p0 = pa::fast_exp2(fmaf(__uint_as_float(s0[e]), c2, -base));
                        const float p1 = pa::fast_exp2(fmaf(__uint_as_float(s0[e + 1]), c2, -base));
                        const float p2 = pa::fast_exp2(fmaf(__uint_as_float(s1[e]), c2, -base));
                        const float p3 = pa::fast_exp2(fmaf(__uint_as_float(s1[e + 1]), c2, -base));
                        la += p0 + p1;
                        lb += p2 + p3;
                        pk[e >> 1] = pa::pack2<kBF16>(p0, p1);
                        pk[16 + (e >> 1)] = pa::pack2<kBF16>(p2, p3);
                    }
                    lsum = la + lb;
                } else {
                    float la = 0.f, lb = 0.f;
                    const int32_t kl = lim - key0;
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float p0 = pa::fast_exp2(fmaf(__uint_as_float(s0[e]), c2, -base));
                        float p1 = pa::fast_exp2(fmaf(__uint_as_float(s0[e + 1]), c2, -base));
                        float p2 = pa::fast_exp2(fmaf(__uint_as_float(s1[e]), c2, -base));
                        float p3 = pa::fast_exp2(fmaf(__uint_as_float(s1[e + 1]), c2, -base));
                        p0 = e <= kl ? p0 : 0.f;
                        p1 = e + 1 <= kl ? p1 : 0.f;
                        p2 = e + 32 <= kl ? p2 : 0.f;
                        p3 = e + 33 <= kl ? p3 : 0.f;
                        la += p0 + p1;
                        lb += p2 + p3;
                        const uint32_t h01 = pa::pack2<kBF16>(p0, p1);
                        const uint32_t h23 = pa::pack2<kBF16>(p2, p3);
                        pk[e >> 1] = h01;
                        pk[16 + (e >> 1)] = h23;
                        rl[e >> 1] = pa::bf16x2_residual(h01, p0, p1);
                        rl[16 + (e >> 1)] = pa::bf16x2_residual(h23, p2, p3);
                    }
                    lsum = la + lb;
                }
                pa::tmem_st32(p_col, pk);
                // the previous tile's product done before O moves
                if (j >= 1) {
                    if (!wait_pv()) {
                        ok = false;
                        break;
                    }
                    pa::tc_fence_after();
                    if (__any_sync(0xffffffffu, grow)) {
                        const float f = grow ? pa::fast_exp2(m_used - m_new) : 1.f;
                        l *= f;
#pragma unroll 1
                        for (int c = 0; c < 2; ++c) {
                            uint32_t o[32];
                            pa::tmem_ld32(o_col + c * 32, o);
                            pa::tmem_ld_wait();
                            pa::reg_fence32(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                            pa::tmem_st32(o_col + c * 32, o);
                        }
                    }
                }
                pa::tmem_st_wait();
                m_used = m_new;
                l += lsum;
                if ((sg.kt0 + j) * kN + kN > sg.n) {
                    // keys past the context: their V rows zeroed (this warpgroup
                    // the 128-byte half h of each row) once the tile has landed
                    const uint32_t vt = vb0 + (uint32_t)j;
                    const uint32_t vs = vt % kVStages;
                    if (!warp_wait(&bar[kVFull + vs], (vt / kVStages) & 1, dead)) {
                        ok = false;
                        break;
                    }
                    if ((sg.kt0 + j) * kN + row >= sg.n) {
                        unsigned char* vrow = smem + kSOffV + vs * kTileBytes +
                                              (uint32_t)(row >> 3) * 2048 + (uint32_t)(row & 7) * 128 +
                                              (uint32_t)h * 1024;
#pragma unroll
                        for (int c16 = 0; c16 < 8; ++c16)
                            *reinterpret_cast<uint4*>(vrow + c16 * 16) = make_uint4(0, 0, 0, 0);
                    }
                    pa::fence_proxy_async_smem();
                }
                pa::tc_fence_before();
                __syncwarp();
                if (lane == 0) pa::mbar_arrive(&bar[kPFull + b]);
                if (residual) {
                    // the bf16 rounding residual of P, a second product over V
                    if (!wait_pv()) {
                        ok = false;
                        break;
                    }
                    pa::tc_fence_after();
                    pa::tmem_st32(p_col, rl);
                    pa::tmem_st_wait();
                    pa::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) pa::mbar_arrive(&bar[kPFull + b]);
                }
            }
            if (!ok) break;
            // ---- the segment's end: the last product, the row sums, then O
            if (!wait_pv()) break;
            pa::tc_fence_after();
            float l_o;
            if (!exchange(l, l_o)) break;
            const float L = h == 0 ? l + l_o : l_o + l;   // the same sum in both warpgroups
            const float M = m_used;
            const bool whole = sg.kt0 == 0 && sg.len == sg.nkt;
            const int32_t hq = sg.g * p.G + (row - t_row * p.G);
            uint16_t* orow = p.out + ((int64_t)(sg.q0 + t_row) * p.H + hq) * kD + h * 64;
            float* ps = nullptr;
            if (!whole) {
                const int64_t c = blockIdx.x;
                const int64_t slot = s_begin(c, F, C) >= sg.a ? 2 * c : 2 * c + 1;
                ps = p.partials + slot * kSlotFloats;
            }
            const float inv = whole && L > 0.f ? 1.f / L : 1.f;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                uint32_t o[32];
                pa::tmem_ld32(o_col + c * 32, o);
                pa::tmem_ld_wait();
                pa::reg_fence32(o);
                if (!valid) continue;
                if (whole) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 x;
                        x.x = pa::pack2<kBF16>(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                        x.y = pa::pack2<kBF16>(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                        x.z = pa::pack2<kBF16>(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                        x.w = pa::pack2<kBF16>(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                        reinterpret_cast<uint4*>(orow)[(c * 32 + e) >> 3] = x;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(ps + (size_t)row * kD + h * 64 + c * 32 + e) =
                            make_float4(__uint_as_float(o[e]), __uint_as_float(o[e + 1]),
                                        __uint_as_float(o[e + 2]), __uint_as_float(o[e + 3]));
                }
            }
            if (!whole && valid && h == 0) {
                ps[(size_t)kM * kD + row] = M;
                ps[(size_t)kM * kD + kM + row] = L;
            }
            pa::tc_fence_before();
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(&bar[kOFree + (r & 1)]);
            if (whole) continue;
            // Publish: the meeting orders every thread's partial stores before
            // thread 0's release; the ticket names the pair's last CTA and, for
            // it, acquires every other CTA's partial.
            if (!all8()) break;
            // the CTAs holding the pair's first and last key tiles
            const int64_t t0 = (int64_t)sg.a + kPairUnits;
            const int64_t c_first = ((t0 + 1) * C - 1) / F;
            const int64_t c_last = ((t0 + sg.nkt) * C - 1) / F;
            if (row == 0 && h == 0) {
                int32_t* ctr = p.counters + (int64_t)sg.i * p.Hkv + sg.g;
                const int prev = pa::atomic_add_acq_rel_gpu(ctr, 1);
                const int last = prev == (int)(c_last - c_first);
                if (last) atomicExch(ctr, 0);
                *last_flag = last;
            }
            if (!all8()) break;
            if (!*last_flag) continue;
            // The pair's last CTA folds every covering CTA's rows.  The first
            // covering CTA holds the pair in its first slot when the pair is its
            // first segment; every later one holds it in its first slot.
            const int ncov = (int)(c_last - c_first + 1);
            const int64_t slot0 = 2 * c_first + (s_begin(c_first, F, C) >= sg.a ? 0 : 1);
            auto slot_ptr = [&](int c) {
                return p.partials + (c ? 2 * (c_first + c) : slot0) * kSlotFloats;
            };
            // per row (warpgroup 0, thread = row): the common maximum and 1 / sum
            if (h == 0) {
                float Mx = -INFINITY;
                for (int c = 0; c < ncov; ++c)
                    Mx = fmaxf(Mx, __ldcg(slot_ptr(c) + (size_t)kM * kD + row));
                const float Mxs = Mx == -INFINITY ? 0.f : Mx;
                float Ls = 0.f;
                for (int c = 0; c < ncov; ++c) {
                    const float* q = slot_ptr(c);
                    Ls += pa::fast_exp2(__ldcg(q + (size_t)kM * kD + row) - Mxs) *
                          __ldcg(q + (size_t)kM * kD + kM + row);
                }
                fold_ml[row] = Mxs;
                fold_ml[kM + row] = Ls > 0.f ? 1.f / Ls : 0.f;
            }
            if (!all8()) break;
            // per row (warp w8 of the eight: rows w8, w8 + 8, ...; lane = 4 of
            // the row's 128 values): coalesced 512-byte reads, kFoldRows rows in
            // flight per covering CTA
            const int w8 = h * 4 + wq;
#pragma unroll 1
            for (int r0 = 0; r0 + w8 < rows; r0 += 8 * kFoldRows) {
                float4 acc[kFoldRows];
#pragma unroll
                for (int k = 0; k < kFoldRows; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
                for (int c = 0; c < ncov; ++c) {
                    const float* q = slot_ptr(c);
                    float4 v[kFoldRows];
                    float mc[kFoldRows];
#pragma unroll
                    for (int k = 0; k < kFoldRows; ++k) {
                        const int rr = min(r0 + 8 * k + w8, kM - 1);
                        v[k] = __ldcg(reinterpret_cast<const float4*>(q + (size_t)rr * kD) + lane);
                        mc[k] = __ldcg(q + (size_t)kM * kD + rr);
                    }
#pragma unroll
                    for (int k = 0; k < kFoldRows; ++k) {
                        const int rr = min(r0 + 8 * k + w8, kM - 1);
                        const float f = pa::fast_exp2(mc[k] - fold_ml[rr]) * fold_ml[kM + rr];
                        acc[k].x += f * v[k].x;
                        acc[k].y += f * v[k].y;
                        acc[k].z += f * v[k].z;
                        acc[k].w += f * v[k].w;
                    }
                }
#pragma unroll
                for (int k = 0; k < kFoldRows; ++k) {
                    const int rr = r0 + 8 * k + w8;
                    if (rr >= rows) break;
                    const int32_t tr = rr / p.G;
                    uint16_t* o = p.out + ((int64_t)(sg.q0 + tr) * p.H + sg.g * p.G + (rr - tr * p.G)) * kD;
                    uint2 x;
                    x.x = pa::pack2<kBF16>(acc[k].x, acc[k].y);
                    x.y = pa::pack2<kBF16>(acc[k].z, acc[k].w);
                    reinterpret_cast<uint2*>(o)[lane] = x;
                }
            }
            // the fold's reads of fold_ml done before a later fold rewrites it
            if (!all8()) break;
        }
        if (*dead && row == 0 && h == 0) pa::raise_error(p.err, PA_DEVERR_TIMEOUT);
    }
    pa::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        pa::tc_fence_after();
        pa::tmem_dealloc(tmem, kTmemCols);
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

CUtensorMapDataType tma_type(pa_dtype dtype) {
    return dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// Cache view {64 elements, token rows of the pool, 64-column half over all KV
// heads}; box {64, 8, 2}: 8 rows of one KV head, both halves, landing as
// [half][8 rows][128 B] -- two swizzle atoms.
bool encode_kv_map(CUtensorMap* map, const void* base, int32_t rows, int32_t Hkv, pa_dtype dtype) {
    auto encode = get_encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)Hkv * 2};
    const cuuint64_t strides[2] = {(cuuint64_t)Hkv * kD * 2, 128};
    const cuuint32_t box[3] = {64, 8, 2};
    const cuuint32_t elem[3] = {1, 1, 1};
    return encode(map, tma_type(dtype), 3, const_cast<void*>(base), dims, strides, box, elem,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Query view {64 elements, head, query row, 64-column half}; box {64, G,
// 128 / G, 1}: one half of a tile's 128 rows (token-major, the group's heads
// inside), landing as [row][128 B].  Rows past the last query read zeros.
bool encode_q_map(CUtensorMap* map, const void* q, int32_t rows, int32_t H, int32_t G,
                  pa_dtype dtype) {
    auto encode = get_encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[4] = {64, (cuuint64_t)H, (cuuint64_t)rows, 2};
    const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2, 128};
    const cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)(kM / G), 1};
    const cuuint32_t elem[4] = {1, 1, 1, 1};
    return encode(map, tma_type(dtype), 4, const_cast<void*>(q), dims, strides, box, elem,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kBF16>
pa_status launch(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                 const Params& prm, size_t smem, int grid, cudaStream_t stream) {
    auto kern = multi_query_tc_kernel<kBF16>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem_total(kMaxBatch));
    });
    if (attr_err != cudaSuccess) return PA_ERR_CUDA;
    kern<<<grid, kThreads, smem, stream>>>(qm, km, vm, prm);
    return pa::cuda_status(cudaGetLastError());
}

size_t split_counters_bytes(int32_t B, int32_t Hkv) {
    return (((size_t)B * Hkv * sizeof(int32_t)) + 255) & ~size_t(255);
}

template <bool kBF16>
pa_status launch_split(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm,
                       const SParams& prm, size_t smem, int grid, cudaStream_t stream) {
    auto kern = multi_query_tc_split_kernel<kBF16>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)split_smem_total(kMaxBatch));
    });
    if (attr_err != cudaSuccess) return PA_ERR_CUDA;
    kern<<<grid, kThreads, smem, stream>>>(qm, km, vm, prm);
    return pa::cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" {

PA_API size_t pa_multi_query_tc_workspace_size(int32_t B, int32_t H, int32_t Hkv, int32_t d) {
    if (B < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || d != kD) return 0;
    const int sms = pa::device_sm_count();
    if (sms <= 0) return 0;
    return split_counters_bytes(B, Hkv) + 2 * (size_t)sms * kSlotFloats * sizeof(float);
}

PA_API pa_status pa_multi_query_tc(const void* q, const int32_t* q_start, int32_t q_rows,
                                   const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int32_t max_blocks,
                                   const int32_t* context_lens, int32_t max_q_len, int32_t B,
                                   int32_t H, int32_t Hkv, int32_t d, int32_t block_size,
                                   int32_t num_blocks, float scale, pa_dtype dtype, void* out,
                                   void* workspace, size_t ws_bytes, void* stream) {
    if (B < 0 || H <= 0 || Hkv <= 0 || max_blocks <= 0 || num_blocks <= 0 || q_rows < 0 ||
        max_q_len < 0 || !std::isfinite(scale))
        return PA_ERR_INVALID;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (H % Hkv != 0 || d != kD) return PA_ERR_UNSUPPORTED;
    const int G = H / Hkv;
    if (G > kM) return PA_ERR_UNSUPPORTED;
    // Every sequence's rows in one query tile: the split mode, any grouping.
    // Otherwise pairs of query tiles, G a power of two (128 / G tokens a tile).
    const bool split = (int64_t)max_q_len * G <= kM;
    if (!split && (G & (G - 1)) != 0) return PA_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
    if (B > kMaxBatch) return PA_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
    // flattened indices are int32: every sequence's 128-row tiles (or 128-key
    // tiles) times Hkv
    if ((int64_t)B * Hkv * (((int64_t)max_blocks * block_size * (split ? 1 : G) + kM - 1) / kM) >=
        ((int64_t)1 << 30))
        return PA_ERR_UNSUPPORTED;
    if (B == 0 || q_rows == 0 || max_q_len == 0) return PA_OK;
    if (!q || !q_start || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return PA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
         reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15u)
        return PA_ERR_INVALID;
    unsigned int* err = pa::device_error_word();
    const int sms = pa::device_sm_count();
    if (!err || !sms) return PA_ERR_CUDA;
    if (split) {
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return PA_ERR_INVALID;
        if (ws_bytes < pa_multi_query_tc_workspace_size(B, H, Hkv, d)) return PA_ERR_INVALID;
    }

    CUtensorMap qm, km, vm;
    const int32_t rows = num_blocks * block_size;
    if (!encode_q_map(&qm, q, q_rows, H, G, dtype) ||
        !encode_kv_map(&km, k_cache, rows, Hkv, dtype) ||
        !encode_kv_map(&vm, v_cache, rows, Hkv, dtype))
        return PA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (split) {
        SParams sp;
        sp.q_start = q_start;
        sp.out = static_cast<uint16_t*>(out);
        sp.block_tables = block_tables;
        sp.context_lens = context_lens;
        sp.counters = static_cast<int32_t*>(workspace);
        sp.partials = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) +
                                               split_counters_bytes(B, Hkv));
        sp.err = err;
        sp.max_blocks = max_blocks;
        sp.B = B;
        sp.H = H;
        sp.Hkv = Hkv;
        sp.G = G;
        sp.tm = kM / G;
        sp.bs = block_size;
        sp.num_blocks = num_blocks;
        sp.max_q_len = max_q_len;
        sp.scale_log2 = scale * kLog2e;
        const size_t smem = split_smem_total(B);
        return dtype == PA_BF16 ? launch_split<true>(qm, km, vm, sp, smem, sms, st)
                                : launch_split<false>(qm, km, vm, sp, smem, sms, st);
    }
    Params prm;
    prm.q_start = q_start;
    prm.out = static_cast<uint16_t*>(out);
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.err = err;
    prm.max_blocks = max_blocks;
    prm.B = B;
    prm.H = H;
    prm.Hkv = Hkv;
    prm.G = G;
    prm.log_g = 31 - __builtin_clz((unsigned)G);
    prm.bs = block_size;
    prm.num_blocks = num_blocks;
    prm.scale_log2 = scale * kLog2e;
    const size_t smem = smem_total(B);
    return dtype == PA_BF16 ? launch<true>(qm, km, vm, prm, smem, sms, st)
                            : launch<false>(qm, km, vm, prm, smem, sms, st);
}

}  // extern "C"
