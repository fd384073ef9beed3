// Several query tokens per sequence over the paged cache (pa_multi_query):
// chunked prefill and speculative verification ("vLLM 深度拆解：当大模型推理学会
// 「分页注意力」", section 5: a long prompt's prefill is cut into chunks that run
// between decode steps, and a draft model's N tokens are verified by one
// forward pass of the main model).  Sequence i's queries are its last qlen_i
// cached tokens (rows q_start[i] .. q_start[i+1]-1 of q); query r attends to
// cached tokens 0 .. n_i - qlen_i + r (causal), as the decode does to all n_i.
//
//  * Work items are (sequence, KV head, tile of 64 rows), a row being one
//    (query token, query head of the KV head's group) pair in token-major
//    order, so one K/V chunk serves the whole GQA group.  An item reads the
//    64-key chunks of its context up to its last row's causal limit.  The
//    list of (item, chunk) pairs is cut into equal contiguous shares over the
//    persistent CTAs (two per SM); an item inside one share finishes in one
//    pass, an item split between shares leaves per-row partials (m, l, O) and
//    the last CTA to finish it -- an atomic ticket per item and warp, never a
//    wait -- merges them.
//  * A producer warp streams the K and V chunks of its share through a
//    shared-memory ring with the decode's 3-D TMA boxes; the table is read 32
//    entries at a time, the next window and the next segment's first window
//    one step ahead.
//  * Four consumer warps own 16 rows each and run FlashAttention-style over
//    the chunks in 32-key halves: S = Q K^T and O += P V as m16n8k16
//    tensor-core MMAs (P stays in registers as the A operand; a bf16 P carries
//    its rounding residual as a second operand in warps that hold a row of
//    fewer than 256 keys), online softmax in base 2 with
//    the per-row causal limit, normalisation once at the end.  V rows past the
//    context are zeroed in shared memory before use (unwritten slots may hold
//    NaN).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "pa.h"
#include "pa_common.cuh"

namespace {

constexpr int kMaxRows = 64;        // query rows per item at most (4 consumer warps x 16)
constexpr int kKv = 64;             // keys per pipeline stage (a "chunk")
constexpr int kMaxWarps = 4;        // consumer warps per CTA at most
constexpr int kMaxStages = 8;
constexpr int kMaxBatch = 4096;
constexpr int kMaxCtas = 512;
constexpr int kMinChunksPerCta = 4;
// A bf16 P keeps 8 significant bits; warps with a row of fewer keys than this
// add P's rounding residual as a second product (about 16 bits).  Over more
// keys the rounding errors of P average out.
constexpr int kResidualKeys = 256;

// Launch shapes: NW consumer warps of 16 rows each plus one producer warp per
// CTA.  Four run two CTAs per SM with 113 KB of shared memory each; three
// (items of at most 48 rows, e.g. a few draft tokens of a GQA group, where a
// fourth warp would idle) run three CTAs per SM with 75 KB each.
template <int NW>
struct Shape {
    static constexpr int kRows = 16 * NW;
    static constexpr int kThreads = (NW + 1) * 32;
    static constexpr int kCtasPerSm = NW == 4 ? 2 : 3;
    static constexpr uint32_t kSmemBudget = NW == 4 ? 113 * 1024 : 75 * 1024;
};
constexpr uint64_t kWaitLimitNs = 1ull << 30;
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
    const uint16_t* q;
    const int32_t* q_start;
    uint16_t* out;
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t* counters;   // [items_cap][kWarps] arrival tickets of split items
    float* partials;     // [2 * kMaxCtas][kRows * (D + 2)] per-CTA partial rows
    unsigned int* err;
    int32_t max_blocks, B, H, Hkv, G, bs, num_blocks, stages, items_cap;
    int32_t rows;        // query rows per item: 16 per consumer warp
    float scale_log2;
};

struct Layout {
    uint32_t stage_bytes, bars, prefix, total;
};

// Stages, barriers, then prefix[B + 1] (chunks), iprefix[B + 1] (items), scan[64].
__host__ __device__ inline Layout make_layout(int D, int B, int stages) {
    Layout L;
    L.stage_bytes = 2u * kKv * D * 2;                      // K then V, 16-bit
    L.bars = stages * L.stage_bytes;                       // full[], empty[]
    L.prefix = L.bars + 2 * kMaxStages * 8;
    L.total = 1024 + L.prefix + (uint32_t)(B + 1) * 8 + 64 * 4;
    return L;
}

__device__ __forceinline__ int32_t clamp_len(int32_t n, int32_t cap) {
    return n < 0 ? 0 : (n > cap ? cap : n);
}

// Byte offset of (token t, 64-column half h, 16-byte column c) in a tensor's
// chunk: [box][half][rows][128 B], TMA 128-byte swizzle.
__device__ __forceinline__ uint32_t tile_offset(uint32_t t, uint32_t h, uint32_t c,
                                                uint32_t halves, uint32_t rows_shift) {
    const uint32_t b = t >> rows_shift, r = t & ((1u << rows_shift) - 1u);
    return ((((b * halves + h) << rows_shift) + r) << 7) + ((c ^ (t & 7u)) << 4);
}

struct SeqInfo {
    int32_t n, qlen, q0, tiles;   // context, queries, first query row, 64-row tiles
};

__device__ __forceinline__ SeqInfo seq_info(const Params& p, int32_t i, int32_t max_len) {
    SeqInfo s;
    s.n = clamp_len(__ldg(p.context_lens + i), max_len);
    s.q0 = __ldg(p.q_start + i);
    s.qlen = __ldg(p.q_start + i + 1) - s.q0;
    s.tiles = (s.qlen < 0 || s.qlen > s.n) ? 0 : (s.qlen * p.G + p.rows - 1) / p.rows;
    return s;
}

// Chunks tile t (of `rows` rows) reads: keys 0 .. n - qlen + r_max, r_max its
// last query token.
__device__ __forceinline__ int32_t tile_chunks(const SeqInfo& s, int32_t t, int32_t G,
                                               int32_t rows) {
    const int32_t rows_end = min((t + 1) * rows, s.qlen * G);
    const int32_t r_max = (rows_end - 1) / G;
    return (s.n - s.qlen + r_max + 1 + kKv - 1) / kKv;
}

// The flattened work list is every (sequence i, KV head g, tile t, chunk c)
// in that order; a segment is the part of one item (i, g, t) inside [pos, hi).
struct Seg {
    int32_t i, g, t;
    SeqInfo s;
    int32_t c0, len, nc;   // first chunk, chunks in the segment, chunks of the item
    int32_t a;             // flattened index of the item's first chunk
    int32_t item;          // item id (counter index)
};

__device__ __forceinline__ Seg find_seg(const int32_t* prefix, const int32_t* iprefix,
                                        const Params& p, int32_t pos, int32_t hi,
                                        int32_t max_len) {
    int32_t lo_i = 0, hi_i = p.B;
    while (hi_i - lo_i > 1) {
        const int32_t mid = (lo_i + hi_i) >> 1;
        if (prefix[mid] <= pos) lo_i = mid; else hi_i = mid;
    }
    Seg sg;
    sg.i = lo_i;
    sg.s = seq_info(p, lo_i, max_len);
    const int32_t per_g = (prefix[lo_i + 1] - prefix[lo_i]) / p.Hkv;
    const int32_t local = pos - prefix[lo_i];
    sg.g = local / per_g;
    const int32_t lg = local - sg.g * per_g;
    int32_t t = 0, acc = 0, ct = tile_chunks(sg.s, 0, p.G, p.rows);
    while (acc + ct <= lg) {
        acc += ct;
        ++t;
        ct = tile_chunks(sg.s, t, p.G, p.rows);
    }
    sg.t = t;
    sg.nc = ct;
    sg.c0 = lg - acc;
    sg.a = pos - sg.c0;
    sg.len = min(hi - pos, ct - sg.c0);
    sg.item = iprefix[lo_i] + sg.g * sg.s.tiles + t;
    return sg;
}

__device__ __forceinline__ int32_t cta_begin(int64_t c, int64_t W, int64_t C) {
    return (int32_t)(c * W / C);
}

// Slot of the partial CTA c leaves for the item starting at a: its first slot
// if the item is where its share begins, else its second.
__device__ __forceinline__ int64_t partial_slot(int64_t c, int64_t W, int64_t C, int32_t a) {
    return cta_begin(c, W, C) >= a ? 2 * c : 2 * c + 1;
}

// Two CTAs of five warps per SM put three warps on two of the four SM
// sub-partitions, whose register files hold 16K registers each: 168 per
// thread at most (three CTAs of four warps: three warps on every one).
template <int D, bool kBF16, int NW>
__global__ void __maxnreg__(168)
multi_query_kernel(const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const Params p) {
    constexpr int kWarps = NW;
    constexpr int kRows = Shape<NW>::kRows;
    constexpr int kThreads = Shape<NW>::kThreads;
    constexpr uint32_t kHalves = D / 64;
    constexpr int kSlotFloats = kRows * (D + 2);
    const int32_t B = p.B, Hkv = p.Hkv, G = p.G, bs = p.bs, S = p.stages;
    const Layout L = make_layout(D, B, S);
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* empty = full + kMaxStages;
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + L.prefix);
    int32_t* iprefix = prefix + (B + 1);
    int32_t* scan = iprefix + (B + 1);   // [32] chunks, [32] items

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t max_len = p.max_blocks * bs;
    const uint32_t rows_shift = (uint32_t)(31 - __clz(bs < 32 ? bs : 32));

    // ---- prefixes: prefix[i] = Hkv * chunks of sequence i's tiles before i,
    //      iprefix[i] = Hkv * tiles before i
    {
        const int per = (B + kThreads - 1) / kThreads;
        const int beg = min(tid * per, B), end = min(beg + per, B);
        auto count = [&](int i, int32_t& chunks, int32_t& tiles) {
            const SeqInfo s = seq_info(p, i, max_len);
            if (blockIdx.x == 0) {
                const int32_t raw = __ldg(p.context_lens + i);
                if (s.qlen != 0 && s.tiles == 0) pa::raise_error(p.err, PA_DEVERR_CONTEXT);
                if (raw > max_len) pa::raise_error(p.err, PA_DEVERR_TABLE_WIDTH);
            }
            tiles = s.tiles;
            chunks = 0;
            for (int32_t t = 0; t < s.tiles; ++t) chunks += tile_chunks(s, t, G, kRows);
        };
        int32_t lc = 0, lt = 0;
        for (int i = beg; i < end; ++i) {
            int32_t c, t;
            count(i, c, t);
            lc += c;
            lt += t;
        }
        int32_t xc = lc, xt = lt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t yc = __shfl_up_sync(0xffffffffu, xc, off);
            const int32_t yt = __shfl_up_sync(0xffffffffu, xt, off);
            if (lane >= off) {
                xc += yc;
                xt += yt;
            }
        }
        if (lane == 31) {
            scan[warp] = xc;
            scan[32 + warp] = xt;
        }
        if (tid == 0) {
            for (int s = 0; s < S; ++s) {
                pa::mbar_init(&full[s], 1);
                pa::mbar_init(&empty[s], kWarps);
            }
            pa::fence_barrier_init();
        }
        __syncthreads();
        int32_t rc = xc - lc, rt = xt - lt;
        for (int w = 0; w < warp; ++w) {
            rc += scan[w];
            rt += scan[32 + w];
        }
        for (int i = beg; i < end; ++i) {
            prefix[i] = rc * Hkv;
            iprefix[i] = rt * Hkv;
            int32_t c, t;
            count(i, c, t);
            rc += c;
            rt += t;
        }
        if (tid == 0) {
            int32_t tc = 0, tt = 0;
            for (int w = 0; w < kThreads / 32; ++w) {
                tc += scan[w];
                tt += scan[32 + w];
            }
            prefix[B] = tc * Hkv;
            iprefix[B] = tt * Hkv;
            if (blockIdx.x == 0 && iprefix[B] > p.items_cap) pa::raise_error(p.err, PA_DEVERR_CONTEXT);
        }
        __syncthreads();
    }
    if (iprefix[B] > p.items_cap) return;   // more queries than max_q_len promised
    const int64_t W = prefix[B];
    // every CTA gets at least kMinChunksPerCta chunks of a balanced contiguous share
    int64_t C = W / kMinChunksPerCta;
    if (C > (int64_t)gridDim.x) C = gridDim.x;
    if (C < 1) C = 1;
    if ((int64_t)blockIdx.x >= C) return;
    const int32_t lo = cta_begin(blockIdx.x, W, C);
    const int32_t hi = cta_begin(blockIdx.x + 1, W, C);

    if (warp == kWarps) {
        // =============================== producer ===============================
        if (lane == 0) {
            pa::prefetch_tensormap(&kmap);
            pa::prefetch_tensormap(&vmap);
        }
        const uint64_t policy = pa::l2_policy_evict_first();
        const int bs_shift = 31 - __clz(bs);
        const int bpc = kKv >> rows_shift;             // blocks (boxes per tensor) per chunk
        const int32_t oob_row = p.num_blocks * bs;
        auto load_window = [&](int32_t i, int32_t base) {
            const int32_t j = base + lane;
            return j < p.max_blocks ? __ldg(p.block_tables + (int64_t)i * p.max_blocks + j) : -1;
        };
        int stage = 0;
        uint32_t use = 0;
        int32_t kglob = 0;       // chunks issued so far
        bool dead = false;
        Seg cur{}, nxt{};
        int32_t went = -1, wnext = -1, nwent = -1, nwnext = -1;
        if (lo < hi) {
            cur = find_seg(prefix, iprefix, p, lo, hi, max_len);
            const int32_t b0 = (cur.c0 * kKv) >> bs_shift;
            went = load_window(cur.i, b0);
            wnext = load_window(cur.i, b0 + 32);
        }
        for (int32_t pos = lo; pos < hi && !dead;) {
            const int32_t npos = pos + cur.len;
            if (npos < hi) {                                 // the next segment's windows
                nxt = find_seg(prefix, iprefix, p, npos, hi, max_len);
                const int32_t b0 = (nxt.c0 * kKv) >> bs_shift;
                nwent = load_window(nxt.i, b0);
                nwnext = load_window(nxt.i, b0 + 32);
            }
            const int32_t nb = (cur.s.n + bs - 1) >> bs_shift;
            int32_t wbase = (cur.c0 * kKv) >> bs_shift;      // windows start at multiples of bpc
            for (int32_t c = cur.c0; c < cur.c0 + cur.len; ++c, ++kglob) {
                const int32_t j0 = (c * kKv) >> bs_shift;
                if (j0 + bpc > wbase + 32) {
                    wbase += 32;
                    went = wnext;
                    wnext = load_window(cur.i, wbase + 32);
                }
                if (kglob >= S &&
                    !__all_sync(0xffffffffu, pa::mbar_wait(&empty[stage], use ^ 1u, kWaitLimitNs))) {
                    dead = true;
                    if (lane == 0) pa::raise_error(p.err, PA_DEVERR_TIMEOUT);
                    break;
                }
                int32_t blk[8];
#pragma unroll
                for (int b = 0; b < 8; ++b)
                    blk[b] = __shfl_sync(0xffffffffu, went, (j0 - wbase + b) & 31);
                if (lane == 0) {
                    pa::mbar_arrive_expect_tx(&full[stage], L.stage_bytes);
                    unsigned char* kdst = smem + stage * L.stage_bytes;
#pragma unroll
                    for (int b = 0; b < 8; ++b) {
                        if (b >= bpc) break;
                        bool ok = j0 + b < nb;
                        if (ok && (blk[b] < 0 || blk[b] >= p.num_blocks)) {
                            ok = false;
                            pa::raise_error(p.err, PA_DEVERR_BLOCK_ID);
                        }
                        const uint32_t off = ((uint32_t)b * kHalves << rows_shift) * 128;
                        const int32_t row = ok ? blk[b] * bs : oob_row;
                        const int32_t z = cur.g * (int32_t)kHalves;
                        pa::tma_load_3d(kdst + off, &kmap, &full[stage], 0, row, z, policy);
                        pa::tma_load_3d(kdst + L.stage_bytes / 2 + off, &vmap, &full[stage], 0,
                                        row, z, policy);
                    }
                }
                __syncwarp();
                if (++stage == S) {
                    stage = 0;
                    use ^= 1u;
                }
            }
            cur = nxt;
            went = nwent;
            wnext = nwnext;
            pos = npos;
        }
        // every issued load has landed before the CTA may exit
        for (int s = 0; s < S && s < kglob; ++s) {
            const int32_t last_use = (kglob - 1 - s) / S;
            pa::mbar_wait(&full[s], (uint32_t)(last_use & 1), kWaitLimitNs);
        }
        return;
    }

    // ================================ consumers ================================
    const int qr = lane >> 2;        // fragment row (and +8)
    const int qc = 2 * (lane & 3);   // fragment column pair
    const int mi = lane >> 3, rr = lane & 7;
    const uint32_t smem_base = pa::smem_addr(smem);
    int stage = 0;
    uint32_t use = 0;
    bool dead = false;

    for (int32_t pos = lo; pos < hi;) {
        const Seg sg = find_seg(prefix, iprefix, p, pos, hi, max_len);
        pos += sg.len;
        const int32_t row0 = sg.t * kRows;
        const int32_t nrows = min(kRows, sg.s.qlen * G - row0);
        // this lane's two rows: (token r, head hg) and its causal limit
        int32_t lim[2];
        int64_t qoff[2];
        bool valid[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int32_t row = warp * 16 + qr + 8 * h2;
            valid[h2] = row < nrows;
            const int32_t ra = row0 + row;
            const int32_t r = ra / G, hg = ra - (ra / G) * G;
            lim[h2] = valid[h2] ? sg.s.n - sg.s.qlen + r : -1;
            qoff[h2] = ((int64_t)(sg.s.q0 + r) * p.H + sg.g * G + hg) * D + qc;
        }
        uint32_t qa[D / 16][4];   // Q as A fragments
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const unsigned int* qp = reinterpret_cast<const unsigned int*>(p.q + qoff[h2] + 16 * ks);
                qa[ks][h2] = valid[h2] ? __ldg(qp) : 0u;
                qa[ks][2 + h2] = valid[h2] ? __ldg(qp + 4) : 0u;
            }
        float o[D / 8][4];
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
        const int32_t warp_lim = __reduce_max_sync(0xffffffffu, max(lim[0], lim[1]));
        // keys up to the smallest limit of the warp's valid rows are visible to all
        // of them (rows past the tile are never read)
        const int32_t warp_min_lim = __reduce_min_sync(
            0xffffffffu, (int)min(valid[0] ? lim[0] : INT32_MAX, valid[1] ? lim[1] : INT32_MAX));
        const bool residual = kBF16 && warp_min_lim < kResidualKeys - 1;

        for (int32_t c = sg.c0; c < sg.c0 + sg.len; ++c) {
            const bool ready = dead || pa::mbar_wait(&full[stage], use, kWaitLimitNs);
            if (!__all_sync(0xffffffffu, ready)) {
                dead = true;
                if (lane == 0) pa::raise_error(p.err, PA_DEVERR_TIMEOUT);
            }
            const int32_t key0 = c * kKv;
            if (!dead && key0 <= warp_lim) {
                const uint32_t kt = smem_base + stage * L.stage_bytes;
                const uint32_t vt = kt + L.stage_bytes / 2;
                const int32_t valid_keys = min(sg.s.n - key0, kKv);
                if (valid_keys < kKv) {
                    // zero V rows past the context (every warp, before its own use)
                    unsigned char* vbytes = smem + stage * L.stage_bytes + L.stage_bytes / 2;
                    const int per_half = (kKv - valid_keys) * 8;
                    for (int e = lane; e < per_half * (int)kHalves; e += 32) {
                        const int hh = e / per_half, rem = e - hh * per_half;
                        const uint32_t tok = (uint32_t)(valid_keys + (rem >> 3));
                        *reinterpret_cast<uint4*>(
                            vbytes + tile_offset(tok, hh, rem & 7, kHalves, rows_shift)) =
                            make_uint4(0, 0, 0, 0);
                    }
                    pa::fence_proxy_async_smem();
                    __syncwarp();
                }
                // The chunk in two halves of 32 keys (fewer live registers: two
                // CTAs per SM); a half past every row's causal limit is skipped.
#pragma unroll 1
                for (int kh = 0; kh < 2; ++kh) {
                    const int32_t hkey0 = key0 + 32 * kh;
                    if (hkey0 > warp_lim) break;
                    // S = Q K^T: 16 rows x 32 keys (4 n-tiles)
                    float s[4][4];
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t d = 16 * ks + (mi & 1) * 8;
#pragma unroll
                        for (int np = 0; np < 2; ++np) {
                            const uint32_t key = 32 * kh + 16 * np + (mi >> 1) * 8 + rr;
                            uint32_t b[4];
                            pa::ldsm_x4(kt + tile_offset(key, d >> 6, (d & 63) >> 3, kHalves,
                                                         rows_shift),
                                        b[0], b[1], b[2], b[3]);
                            pa::mma_16816<kBF16>(s[2 * np], qa[ks], b[0], b[1]);
                            pa::mma_16816<kBF16>(s[2 * np + 1], qa[ks], b[2], b[3]);
                        }
                    }
                    // causal mask, online softmax (rows qr and qr + 8 of this warp);
                    // a half every valid row sees whole needs no mask (rows past
                    // the tile have zero q and are never stored)
                    float mx[2] = {-INFINITY, -INFINITY};
                    if (hkey0 + 31 <= warp_min_lim) {
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float x = s[nt][e] * p.scale_log2;
                                s[nt][e] = x;
                                mx[e >> 1] = fmaxf(mx[e >> 1], x);
                            }
                    } else {
#pragma unroll
                        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int32_t key = hkey0 + 8 * nt + qc + (e & 1);
                                const float x =
                                    key <= lim[e >> 1] ? s[nt][e] * p.scale_log2 : -INFINITY;
                                s[nt][e] = x;
                                mx[e >> 1] = fmaxf(mx[e >> 1], x);
                            }
                    }
                    float alpha[2], msafe[2];
                    bool grew = false;
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        float v = mx[h2];
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
                        const float m_new = fmaxf(m_run[h2], v);
                        grew |= m_new > m_run[h2];
                        msafe[h2] = m_new == -INFINITY ? 0.f : m_new;
                        alpha[h2] = pa::fast_exp2(m_run[h2] - msafe[h2]);
                        m_run[h2] = m_new;
                        l_run[h2] *= alpha[h2];
                    }
                    // O needs the rescale only when some row's maximum grew (a
                    // row whose maximum stays has alpha = 1 exactly)
                    if (__any_sync(0xffffffffu, grew)) {
#pragma unroll
                        for (int nt = 0; nt < D / 8; ++nt) {
                            o[nt][0] *= alpha[0];
                            o[nt][1] *= alpha[0];
                            o[nt][2] *= alpha[1];
                            o[nt][3] *= alpha[1];
                        }
                    }
                    // P as A fragments (k-step = 16 keys = n-tiles 2 ks2, 2 ks2 + 1).
                    // bf16 keeps 8 bits of P: for warps with a short row a
                    // second, residual part (pl) restores about 16, so a row of
                    // a few keys whose V terms cancel stays within the
                    // tolerance; f16 P (11 bits) needs none.
                    uint32_t pa_[2][4], pl[2][4];
#pragma unroll
                    for (int nt = 0; nt < 4; ++nt) {
                        float e4[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            e4[e] = pa::fast_exp2(s[nt][e] - msafe[e >> 1]);
                            l_run[e >> 1] += e4[e];
                        }
                        const uint32_t h01 = pa::pack2<kBF16>(e4[0], e4[1]);
                        const uint32_t h23 = pa::pack2<kBF16>(e4[2], e4[3]);
                        pa_[nt >> 1][(nt & 1) * 2] = h01;
                        pa_[nt >> 1][(nt & 1) * 2 + 1] = h23;
                        if (residual) {
                            pl[nt >> 1][(nt & 1) * 2] = pa::bf16x2_residual(h01, e4[0], e4[1]);
                            pl[nt >> 1][(nt & 1) * 2 + 1] = pa::bf16x2_residual(h23, e4[2], e4[3]);
                        }
                    }
                    // O += P V: 16 rows x D (D/8 n-tiles), 32 keys (2 k-steps)
#pragma unroll
                    for (int ks2 = 0; ks2 < 2; ++ks2) {
                        const uint32_t key = 32 * kh + 16 * ks2 + (mi & 1) * 8 + rr;
                        const uint32_t a[4] = {pa_[ks2][0], pa_[ks2][1], pa_[ks2][2], pa_[ks2][3]};
                        const uint32_t al[4] = {pl[ks2][0], pl[ks2][1], pl[ks2][2], pl[ks2][3]};
#pragma unroll
                        for (int np2 = 0; np2 < D / 16; ++np2) {
                            const uint32_t d = 16 * np2 + (mi >> 1) * 8;
                            uint32_t b[4];
                            pa::ldsm_x4_trans(vt + tile_offset(key, d >> 6, (d & 63) >> 3, kHalves,
                                                               rows_shift),
                                              b[0], b[1], b[2], b[3]);
                            pa::mma_16816<kBF16>(o[2 * np2], a, b[0], b[1]);
                            pa::mma_16816<kBF16>(o[2 * np2 + 1], a, b[2], b[3]);
                            if (residual) {
                                pa::mma_16816<kBF16>(o[2 * np2], al, b[0], b[1]);
                                pa::mma_16816<kBF16>(o[2 * np2 + 1], al, b[2], b[3]);
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) pa::mbar_arrive(&empty[stage]);
            if (++stage == S) {
                stage = 0;
                use ^= 1u;
            }
        }
        if (dead) continue;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            float v = l_run[h2];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            l_run[h2] = v;
        }
        auto store_row_pair = [&](int h2, int nt, float x, float y) {
            *reinterpret_cast<uint32_t*>(p.out + qoff[h2] + 8 * nt) = pa::pack2<kBF16>(x, y);
        };
        if (sg.c0 == 0 && sg.len == sg.nc) {
            // the whole item is in this CTA's share: normalise and store
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                if (!valid[h2]) continue;
                const float inv = l_run[h2] > 0.f ? 1.f / l_run[h2] : 0.f;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt)
                    store_row_pair(h2, nt, o[nt][2 * h2] * inv, o[nt][2 * h2 + 1] * inv);
            }
            continue;
        }
        // A split item: this warp's 16 rows go to the CTA's partial slot; the
        // last CTA to finish them (per-warp ticket) merges all partials.
        const int64_t c_first = ((int64_t)(sg.a + 1) * C - 1) / W;
        const int64_t c_last = ((int64_t)(sg.a + sg.nc) * C - 1) / W;
        float* ps = p.partials + partial_slot(blockIdx.x, W, C, sg.a) * kSlotFloats;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int row = warp * 16 + qr + 8 * h2;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt)
                *reinterpret_cast<float2*>(&ps[row * D + 8 * nt + qc]) =
                    make_float2(o[nt][2 * h2], o[nt][2 * h2 + 1]);
            if ((lane & 3) == 0) {
                ps[kRows * D + row] = m_run[h2];
                ps[kRows * D + kRows + row] = l_run[h2];
            }
        }
        // Publish: __syncwarp orders the lanes' stores before lane 0's release
        // (cumulativity); the acquire-release ticket names the last CTA and,
        // for it, acquires the other CTAs' partials.
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            int32_t* ctr = p.counters + (int64_t)sg.item * kWarps + warp;
            last = pa::atomic_add_acq_rel_gpu(ctr, 1) == (int)(c_last - c_first);
            if (last) atomicExch(ctr, 0);   // ready for the next launch
        }
        if (!__shfl_sync(0xffffffffu, last, 0)) continue;
        __syncwarp();
        const int ncov = (int)(c_last - c_first + 1);
        const int64_t slot0 = 2 * c_first + (cta_begin(c_first, W, C) == sg.a ? 0 : 1);
        // Each lane folds, for its 4 output values, the ncov partials
        // (m_c, l_c, O_c) eight at a time with all eight loads in flight.
        for (int e = lane; e < 16 * (D / 4); e += 32) {
            const int row = warp * 16 + e / (D / 4), d4 = (e % (D / 4)) * 4;
            if (row >= nrows) continue;
            float M = -INFINITY, Ls = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int c0 = 0; c0 < ncov; c0 += 8) {
                float pm[8], pl[8];
                float4 po[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int cc = c0 + j;
                    if (cc < ncov) {
                        const float* q =
                            p.partials + (cc ? 2 * (c_first + cc) : slot0) * kSlotFloats;
                        pm[j] = __ldcg(q + kRows * D + row);
                        pl[j] = __ldcg(q + kRows * D + kRows + row);
                        po[j] = __ldcg(reinterpret_cast<const float4*>(q + row * D + d4));
                    } else {
                        pm[j] = -INFINITY;
                        pl[j] = 0.f;
                        po[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                float Mb = M;
#pragma unroll
                for (int j = 0; j < 8; ++j) Mb = fmaxf(Mb, pm[j]);
                if (Mb == -INFINITY) continue;   // rows with no key so far
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
            const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
            const int32_t ra = row0 + row;
            const int32_t r = ra / G, hg = ra - (ra / G) * G;
            uint2 packed;
            packed.x = pa::pack2<kBF16>(acc.x * inv, acc.y * inv);
            packed.y = pa::pack2<kBF16>(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(p.out + ((int64_t)(sg.s.q0 + r) * p.H + sg.g * G + hg) * D +
                                      d4) = packed;
        }
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

// The decode's 3-D cache view: {64 elements, token rows of the pool, 64-column
// half over all KV heads}; box {64, min(block_size, 32), d / 64}.
bool encode_cache_map(CUtensorMap* map, const void* base, int32_t rows, int32_t Hkv, int32_t d,
                      int32_t block_size, pa_dtype dtype) {
    auto encode = get_encode_fn();
    if (!encode) return false;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)Hkv * d / 64};
    const cuuint64_t strides[2] = {(cuuint64_t)Hkv * d * 2, 128};
    const cuuint32_t box[3] = {64, (cuuint32_t)(block_size < 32 ? block_size : 32),
                               (cuuint32_t)(d / 64)};
    const cuuint32_t elem[3] = {1, 1, 1};
    return encode(map,
                  dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                  3, const_cast<void*>(base), dims, strides, box, elem,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int choose_stages(int D, int B, uint32_t budget) {
    const Layout L0 = make_layout(D, B, 0);
    if (L0.total >= budget) return 0;
    int s = (int)((budget - L0.total) / L0.stage_bytes);
    return s > kMaxStages ? kMaxStages : s;
}

// Upper bound of the work items under either launch shape: every sequence's
// tiles (of 48 rows, the smaller tile) times Hkv.
int64_t items_cap(int32_t B, int32_t H, int32_t Hkv, int32_t max_q_len) {
    const int64_t G = H / Hkv;
    const int64_t rows = Shape<3>::kRows;
    return (int64_t)B * Hkv * (((int64_t)max_q_len * G + rows - 1) / rows);
}

size_t counters_bytes(int64_t items) {
    return (((size_t)items * kMaxWarps * sizeof(int32_t)) + 255) & ~size_t(255);
}

size_t partials_bytes(int32_t d) {
    return (size_t)2 * kMaxCtas * kMaxRows * (d + 2) * sizeof(float);
}

template <int D, bool kBF16, int NW>
pa_status launch(const CUtensorMap& km, const CUtensorMap& vm, const Params& prm, size_t smem,
                 int grid, cudaStream_t stream) {
    auto kern = multi_query_kernel<D, kBF16, NW>;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)Shape<NW>::kSmemBudget);
        if (attr_err == cudaSuccess)   // the largest shared-memory carve-out
            attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                            100);
    });
    if (attr_err != cudaSuccess) return PA_ERR_CUDA;
    kern<<<grid, Shape<NW>::kThreads, smem, stream>>>(km, vm, prm);
    return pa::cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" {

PA_API size_t pa_multi_query_workspace_size(int32_t B, int32_t H, int32_t Hkv, int32_t d,
                                            int32_t max_q_len) {
    if (B < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || max_q_len < 0 || (d != 64 && d != 128))
        return 0;
    return counters_bytes(items_cap(B, H, Hkv, max_q_len)) + partials_bytes(d);
}

PA_API pa_status pa_multi_query(const void* q, const int32_t* q_start, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                int32_t max_blocks, const int32_t* context_lens,
                                int32_t max_q_len, int32_t B, int32_t H, int32_t Hkv, int32_t d,
                                int32_t block_size, int32_t num_blocks, float scale,
                                pa_dtype dtype, void* out, void* workspace, size_t ws_bytes,
                                void* stream) {
    if (B < 0 || H <= 0 || Hkv <= 0 || max_blocks <= 0 || num_blocks <= 0 || max_q_len < 0 ||
        !std::isfinite(scale))
        return PA_ERR_INVALID;
    if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (H % Hkv != 0) return PA_ERR_UNSUPPORTED;
    if (d != 64 && d != 128) return PA_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PA_ERR_UNSUPPORTED;
    if (B > kMaxBatch) return PA_ERR_UNSUPPORTED;
    if ((int64_t)num_blocks * block_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
    const int G = H / Hkv;
    // flattened chunk indices are int32: every tile's chunks times Hkv
    const int64_t cap = items_cap(B, H, Hkv, max_q_len);
    const int64_t max_chunks = ((int64_t)max_blocks * block_size + kKv - 1) / kKv;
    if (cap * max_chunks >= ((int64_t)1 << 30)) return PA_ERR_UNSUPPORTED;
    if (B == 0 || max_q_len == 0) return PA_OK;
    if (!q || !q_start || !k_cache || !v_cache || !block_tables || !context_lens || !out ||
        !workspace)
        return PA_ERR_INVALID;
    if (ws_bytes < pa_multi_query_workspace_size(B, H, Hkv, d, max_q_len)) return PA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
         reinterpret_cast<uintptr_t>(workspace)) & 15u)
        return PA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 7u)
        return PA_ERR_INVALID;
    // Items of at most 48 rows (a few query tokens of a group) run the
    // three-warp shape when its smaller ring still holds two stages.
    const int stages3 = choose_stages(d, B, Shape<3>::kSmemBudget);
    const bool narrow = (int64_t)max_q_len * G <= Shape<3>::kRows && stages3 >= 2;
    const int stages = narrow ? stages3 : choose_stages(d, B, Shape<4>::kSmemBudget);
    if (stages < 2) return PA_ERR_UNSUPPORTED;
    unsigned int* err = pa::device_error_word();
    const int sms = pa::device_sm_count();
    if (!err || !sms) return PA_ERR_CUDA;

    CUtensorMap km, vm;
    const int32_t rows = num_blocks * block_size;
    if (!encode_cache_map(&km, k_cache, rows, Hkv, d, block_size, dtype) ||
        !encode_cache_map(&vm, v_cache, rows, Hkv, d, block_size, dtype))
        return PA_ERR_CUDA;

    Params prm;
    prm.q = static_cast<const uint16_t*>(q);
    prm.q_start = q_start;
    prm.out = static_cast<uint16_t*>(out);
    prm.block_tables = block_tables;
    prm.context_lens = context_lens;
    prm.counters = static_cast<int32_t*>(workspace);
    prm.partials = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) +
                                            counters_bytes(cap));
    prm.err = err;
    prm.max_blocks = max_blocks;
    prm.B = B;
    prm.H = H;
    prm.Hkv = Hkv;
    prm.G = G;
    prm.bs = block_size;
    prm.num_blocks = num_blocks;
    prm.stages = stages;
    prm.items_cap = (int32_t)cap;
    prm.rows = narrow ? Shape<3>::kRows : Shape<4>::kRows;
    prm.scale_log2 = scale * kLog2e;
    const size_t smem = make_layout(d, B, stages).total;
    int grid = sms * (narrow ? Shape<3>::kCtasPerSm : Shape<4>::kCtasPerSm);
    if (grid > kMaxCtas) grid = kMaxCtas;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool bf = dtype == PA_BF16;
    if (narrow) {
        if (d == 128)
            return bf ? launch<128, true, 3>(km, vm, prm, smem, grid, st)
                      : launch<128, false, 3>(km, vm, prm, smem, grid, st);
        return bf ? launch<64, true, 3>(km, vm, prm, smem, grid, st)
                  : launch<64, false, 3>(km, vm, prm, smem, grid, st);
    }
    if (d == 128)
        return bf ? launch<128, true, 4>(km, vm, prm, smem, grid, st)
                  : launch<128, false, 4>(km, vm, prm, smem, grid, st);
    return bf ? launch<64, true, 4>(km, vm, prm, smem, grid, st)
              : launch<64, false, 4>(km, vm, prm, smem, grid, st);
}

}  // extern "C"
