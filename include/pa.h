/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged KV-cache decode library.
 *
 * The operations follow five web pages on vLLM's PagedAttention, cited by
 * title and section:
 *   [P1] "LLM推理优化：vLLM PagedAttention深度解析与工程实践" (lpnh.cn/news/754185)
 *   [P2] "vLLM推理加速深度解析：从PagedAttention原理到生产部署实战" (kwkr.cn/news/169259)
 *   [P3] "vLLM 深度拆解：当大模型推理学会「分页注意力」——PagedAttention、连续批处理与
 *        V1 引擎如何重写 GPU 推理服务的心智模型" (chenxutan.com/d/4834.html)
 *   [P4] "LLM推理优化技术地图：从KV Cache到量化与投机解码" (qwbw.cn/news/280730)
 *   [P5] the untitled Qwen2.5-7B-on-vLLM deployment page (mhpq.cn/news/468822)
 *
 * Conventions
 *   - Every call returns a pa_status; nothing throws across the ABI.
 *   - Host pointers are marked (host), device pointers (device).  The caller
 *     owns every buffer; the library allocates no device memory.
 *   - Device calls are asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and never synchronise.  Errors found by a kernel
 *     (a block id outside the pool, a slot outside the cache, a context longer
 *     than its table row) set bits in a per-device error word; the offending
 *     access is skipped, never performed.  pa_check_device_errors() reads and
 *     clears that word.
 *   - KV cache layout ([P1] section 4.1): one K and one V tensor per layer,
 *     each [num_blocks][block_size][num_kv_heads][head_dim], row-major,
 *     16-byte aligned.  A token's slot is physical_block * block_size +
 *     offset_in_block.
 *   - Supported shapes: head_dim 64 or 128; block_size 8, 16 or 32;
 *     num_heads % num_kv_heads == 0; for pa_decode and pa_decode_fp8 the
 *     group G = num_heads / num_kv_heads is at most 16 or a multiple of 16
 *     (wider groups, e.g. multi-query attention, are processed 16 query heads
 *     at a time); fp16 or bf16 elements.  Other shapes return
 *     PA_ERR_UNSUPPORTED.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID = 1,      /* bad argument or an operation the state forbids */
    PA_ERR_OOM = 2,          /* the free block list cannot cover the request */
    PA_ERR_NOT_FOUND = 3,    /* unknown sequence id */
    PA_ERR_BOUNDS = 4,       /* a kernel met an index outside its buffers */
    PA_ERR_CUDA = 5,         /* a CUDA runtime call failed */
    PA_ERR_UNSUPPORTED = 6,  /* shape or dtype outside the supported set */
    PA_ERR_TIMEOUT = 7       /* a kernel's bounded wait ran out */
} pa_status;

typedef enum pa_dtype { PA_F16 = 0, PA_BF16 = 1 } pa_dtype;

/* Bits of the device error word (pa_check_device_errors). */
#define PA_DEVERR_BLOCK_ID 0x1u     /* table entry < 0 or >= num_blocks */
#define PA_DEVERR_TABLE_WIDTH 0x2u  /* context_len needs more blocks than max_blocks */
#define PA_DEVERR_SLOT 0x4u         /* slot >= num_blocks * block_size */
#define PA_DEVERR_TIMEOUT 0x8u      /* a bounded pipeline wait gave up */
#define PA_DEVERR_PAIR 0x10u        /* copy pair outside the pool */
#define PA_DEVERR_CONTEXT 0x20u     /* negative context length */

PA_API const char* pa_status_str(pa_status s);
PA_API int32_t pa_version(void);

/* ------------------------------------------------------------------------
 * Host block allocator.  [P1] section 3.2 (BlockManager): the free list starts
 * in block order (or in the caller's order), blocks are taken from its front
 * and returned to its back in table order, and an allocation checks the free
 * list before taking anything.  [P3] section 3.3 (BlockSpaceManager):
 * append_slot writes into the last block while it has room and takes a new
 * block when it is full; free returns all blocks; sequences with the same
 * prefix share physical blocks, and a shared block is copied only when a
 * sharer writes into it (copy-on-write).  [P2] section 2.2 gives the same
 * workflow.  Shared blocks carry a reference count; a block returns to the
 * free list when its count reaches zero.
 *
 * A pa_allocator is host-only and not thread-safe; the caller owns it
 * (create/destroy).  Sequence ids are arbitrary int64 keys.
 * ---------------------------------------------------------------------- */
typedef struct pa_allocator pa_allocator;

typedef struct pa_alloc_stats {
    int32_t num_blocks;     /* pool size */
    int32_t block_size;     /* tokens per block */
    int32_t free_blocks;    /* blocks on the free list */
    int32_t used_blocks;    /* blocks with reference count >= 1 */
    int32_t shared_blocks;  /* blocks with reference count >= 2 */
    int32_t num_seqs;       /* live sequences */
    int64_t num_tokens;     /* sum of the live sequences' lengths */
} pa_alloc_stats;

/* Creates a pool of num_blocks blocks of block_size tokens.  init_free_order
 * (host, num_blocks int32, nullable) is the initial free list and must be a
 * permutation of 0..num_blocks-1; NULL means 0..num_blocks-1. */
PA_API pa_status pa_alloc_create(int32_t num_blocks, int32_t block_size,
                                 const int32_t* init_free_order, pa_allocator** out);
PA_API void pa_alloc_destroy(pa_allocator* a);

/* [P1] section 3.2 allocate(seq_id, num_tokens): grows the sequence (creating
 * it if new) so that its blocks hold num_tokens tokens, taking
 * ceil((num_tokens - held_slots) / block_size) blocks from the front of the
 * free list; the sequence's length becomes max(length, num_tokens).  All or
 * nothing: PA_ERR_OOM leaves every state unchanged.  Growing a sequence whose
 * partially filled last block is shared returns PA_ERR_INVALID (use
 * pa_append_slot, which copies on write). */
PA_API pa_status pa_alloc(pa_allocator* a, int64_t seq_id, int32_t num_tokens);

/* [P3] section 3.3 append_slot(): reserves the slot of the sequence's next
 * token (position = current length) and returns it in *slot_out (host).  If
 * that position opens a new block, a block is taken from the front of the free
 * list.  If it falls in a partially filled block shared with other sequences,
 * a new block is taken, the sequence's table points to it, the old block's
 * count drops by one, and (*cow_src, *cow_dst) name the copy the caller must
 * make (pa_copy_blocks) before writing the token; otherwise both are -1.
 * cow_src / cow_dst may be NULL.  PA_ERR_OOM leaves state unchanged. */
PA_API pa_status pa_append_slot(pa_allocator* a, int64_t seq_id, int64_t* slot_out,
                                int32_t* cow_src, int32_t* cow_dst);

/* One decode step's appends: pa_append_slot for seq_ids[0..B) in that order,
 * all or nothing.  slot_mapping (host, B int64) receives each new token's
 * slot, cow_pairs (host, capacity B pairs of int32 {src, dst}) the copies to
 * make, *num_cow their count.  Duplicate ids return PA_ERR_INVALID. */
PA_API pa_status pa_append_batch(pa_allocator* a, const int64_t* seq_ids, int32_t B,
                                 int64_t* slot_mapping, int32_t* cow_pairs, int32_t* num_cow);

/* Shares parent's blocks with a new sequence child: the table is copied and
 * every block's count rises by one; no KV data moves ([P4] section 3.3, [P3]
 * section 3.3). */
PA_API pa_status pa_fork(pa_allocator* a, int64_t parent, int64_t child);

/* [P1] section 3.2 free(seq_id): drops the sequence; each block's count
 * falls by one and blocks reaching zero go to the back of the free list in
 * table order. */
PA_API pa_status pa_free(pa_allocator* a, int64_t seq_id);

/* Fills block_tables (host, [B][max_blocks] int32, unused entries -1) and
 * context_lens (host, [B] int32) for seq_ids[0..B).  A table longer than
 * max_blocks returns PA_ERR_INVALID. */
PA_API pa_status pa_export(const pa_allocator* a, const int64_t* seq_ids, int32_t B,
                           int32_t max_blocks, int32_t* block_tables, int32_t* context_lens);

/* Slots (host, count int64) of token positions [start, start+count) of a
 * sequence, e.g. to write a prompt's K/V with pa_reshape_and_cache. */
PA_API pa_status pa_seq_slots(const pa_allocator* a, int64_t seq_id, int32_t start,
                              int32_t count, int64_t* slots);
PA_API pa_status pa_seq_info(const pa_allocator* a, int64_t seq_id, int32_t* length,
                             int32_t* num_table_blocks);
PA_API pa_status pa_block_ref(const pa_allocator* a, int32_t block, int32_t* ref);
/* Copies the free list, front first, into out (host, capacity cap). */
PA_API pa_status pa_free_list(const pa_allocator* a, int32_t* out, int32_t cap, int32_t* n);
PA_API pa_status pa_alloc_stats_get(const pa_allocator* a, pa_alloc_stats* out);

/* ------------------------------------------------------------------------
 * Automatic prefix caching ([P5] section 3.2: a prompt is cut into blocks of
 * block_size tokens, each block's KV is cached under a hash of its token ids,
 * and a request reuses the cached KV of a prefix that matches token for token
 * and is aligned to block boundaries; [P1] section 4.2: reuse across requests,
 * e.g. the turns of a conversation).
 *
 * A full block is cached under the key (id of the cache entry holding the
 * previous block's content, or 0 for the first block, the block's token ids),
 * so a key names the whole prefix up to the block; entry ids are never reused.
 * A freed block keeps its entry while it waits on the free list, and a hit
 * takes it back off the list; a block the free list hands out again (from its
 * front, oldest freed first) loses its entry.  Only sequences created by
 * pa_alloc_prompt and grown by pa_append_token / pa_append_batch_tokens know
 * their token ids; pa_alloc, pa_append_slot and pa_append_batch on a sequence
 * stop its registering.  The cache costs host memory only (one entry of
 * block_size token ids per cached block).
 * ---------------------------------------------------------------------- */
typedef struct pa_prefix_stats {
    int64_t lookups;      /* prompt blocks looked up (each walk stops at its first miss) */
    int64_t hits;         /* of which found */
    int64_t registered;   /* blocks entered into the cache */
    int64_t evicted;      /* entries dropped because their block was handed out again */
    int64_t entries;      /* entries now in the cache */
    int64_t cached_free;  /* free-list blocks that still hold an entry */
} pa_prefix_stats;

/* Creates sequence seq_id (which must be new) holding the prompt
 * tokens[0..num_tokens) (host int32 token ids).  The prompt's full blocks are
 * looked up in order; each one found is shared (count +1, taken off the free
 * list if it was there) until the first miss.  The remaining blocks come from
 * the front of the free list, and each new full block is entered into the
 * cache (its K/V must be written, e.g. by pa_reshape_and_cache at the slots
 * of pa_seq_slots, before another sequence reads it).  *cached_tokens
 * (nullable) receives the number of leading tokens whose K/V is already in
 * the cache (a multiple of block_size): the caller computes and writes only
 * the rest.  All or nothing: PA_ERR_OOM leaves every state unchanged. */
PA_API pa_status pa_alloc_prompt(pa_allocator* a, int64_t seq_id, const int32_t* tokens,
                                 int32_t num_tokens, int32_t* cached_tokens);

/* pa_append_slot that also records the appended token's id: when the token
 * fills its block, the block is entered into the cache (unless the same key
 * is cached already, in which case the sequence's chain continues from that
 * entry). */
PA_API pa_status pa_append_token(pa_allocator* a, int64_t seq_id, int32_t token,
                                 int64_t* slot_out, int32_t* cow_src, int32_t* cow_dst);

/* pa_append_batch with one token id per sequence (tokens: host, B int32). */
PA_API pa_status pa_append_batch_tokens(pa_allocator* a, const int64_t* seq_ids,
                                        const int32_t* tokens, int32_t B, int64_t* slot_mapping,
                                        int32_t* cow_pairs, int32_t* num_cow);

PA_API pa_status pa_prefix_stats_get(const pa_allocator* a, pa_prefix_stats* out);

/* ------------------------------------------------------------------------
 * Swap space ([P1] section 3.2: an allocation that finds too few free blocks
 * calls for swap or preemption; [P2] section 4: with swap space enabled the
 * KV cache moves to CPU memory, at a cost in speed).
 *
 * The allocator keeps a host pool of num_host_blocks blocks with its own free
 * list (taken from the front, returned to the back).  A swapped-out sequence
 * holds host blocks instead of device blocks; it cannot be appended to,
 * forked, grown or exported until it is swapped back in; pa_free releases its
 * host blocks.  The caller moves the data with pa_swap_blocks (device pool ->
 * host pool before the device blocks are reused; host -> device after a swap
 * in, before the sequence is read).
 * ---------------------------------------------------------------------- */
typedef struct pa_swap_stats {
    int32_t host_blocks;   /* host pool size */
    int32_t host_free;     /* host blocks on the host free list */
    int32_t swapped_seqs;  /* sequences now swapped out */
} pa_swap_stats;

/* Sets the host pool size (once; host blocks 0..num_host_blocks-1 in order). */
PA_API pa_status pa_alloc_set_swap_pool(pa_allocator* a, int32_t num_host_blocks);

/* Swaps a sequence out: each block of its table, in order, takes a host block
 * from the front of the host free list; pairs (host, capacity cap pairs of
 * int32) receives {device block, host block} per block and *n their count.
 * Each device block's count then drops by one (blocks reaching zero go to the
 * back of the device free list, as in pa_free), so a block still shared with
 * live sequences stays on the device and the swapped sequence keeps its own
 * host copy.  All or nothing: PA_ERR_OOM (host pool full) leaves every state
 * unchanged. */
PA_API pa_status pa_swap_out(pa_allocator* a, int64_t seq_id, int32_t* pairs, int32_t cap,
                             int32_t* n);

/* Swaps a sequence back in: one device block from the front of the free list
 * per host block, in table order; pairs receives {host block, device block};
 * the host blocks return to the back of the host free list.  All or nothing
 * (PA_ERR_OOM).  The sequence's blocks are private afterwards. */
PA_API pa_status pa_swap_in(pa_allocator* a, int64_t seq_id, int32_t* pairs, int32_t cap,
                            int32_t* n);

PA_API pa_status pa_swap_stats_get(const pa_allocator* a, pa_swap_stats* out);
/* Copies the host free list, front first, into out (host, capacity cap). */
PA_API pa_status pa_host_free_list(const pa_allocator* a, int32_t* out, int32_t cap, int32_t* n);

/* ------------------------------------------------------------------------
 * Device operations.
 * ---------------------------------------------------------------------- */

/* KV append ([P2] section 2.2: each generated token's K/V is stored in the
 * physical block its current logical block points to; [P3] section 3.3).
 * For t in [0, T): if slot_mapping[t] >= 0,
 *   k_cache[slot / block_size][slot % block_size][h][:] = k_new[t][h][:]
 * and the same for V, for every KV head h.  A negative slot is padding and is
 * skipped.  A slot >= num_blocks * block_size is skipped and sets
 * PA_DEVERR_SLOT.  Bit-exact copy.
 *   k_new, v_new   (device) [T][Hkv][d] fp16/bf16
 *   slot_mapping   (device) [T] int64
 *   k_cache, v_cache (device) [num_blocks][block_size][Hkv][d], updated in place */
PA_API pa_status pa_reshape_and_cache(const void* k_new, const void* v_new,
                                      const int64_t* slot_mapping, int32_t T, void* k_cache,
                                      void* v_cache, int32_t num_blocks, int32_t block_size,
                                      int32_t Hkv, int32_t d, pa_dtype dtype, void* stream);

/* FP8 KV append ([P4] section 4.3: quantising the KV cache to 8 bits halves
 * its bytes; the pages fix no format, so this library takes OCP FP8 E4M3 with
 * one fp32 scale per (token, KV head) row).  For t in [0, T) with
 * slot = slot_mapping[t] >= 0 and every KV head h, with x = k_new[t][h][:]
 * widened to fp32:
 *   s = fl32(max_i |x_i| / 448)
 *   k_cache[slot / bs][slot % bs][h][i] = E4M3(fl32(x_i / s))   (RNE, saturating)
 *   k_scale[slot / bs][h][slot % bs] = s
 * (IEEE fp32 divisions); an all-zero row stores s = 0 and zero codes.  Rows
 * holding NaN or infinity are outside this contract (their scale is not
 * defined by the formula above; codes and scale are unspecified).  The
 * same for V.  A negative slot is padding and is skipped; a slot >=
 * num_blocks * block_size is skipped and sets PA_DEVERR_SLOT.
 *   k_new, v_new     (device) [T][Hkv][d] fp16/bf16 (dtype), d = 128
 *   slot_mapping     (device) [T] int64
 *   k_cache, v_cache (device) [num_blocks][block_size][Hkv][d] uint8 codes
 *   k_scale, v_scale (device) [num_blocks][Hkv][block_size] fp32, 16-byte aligned */
PA_API pa_status pa_reshape_and_cache_fp8(const void* k_new, const void* v_new,
                                          const int64_t* slot_mapping, int32_t T, void* k_cache,
                                          void* v_cache, float* k_scale, float* v_scale,
                                          int32_t num_blocks, int32_t block_size, int32_t Hkv,
                                          int32_t d, pa_dtype dtype, void* stream);

/* INT8 KV append (the other 8-bit format of [P4] section 4.3; the pages fix
 * none, so this library takes symmetric INT8 with one fp32 scale per (token,
 * KV head) row).  As pa_reshape_and_cache_fp8 with
 *   s = fl32(max_i |x_i| / 127)
 *   k_cache[slot / bs][slot % bs][h][i] = clamp(rint(fl32(x_i / s)), -127, 127)
 * (nearest integer, ties to even; the byte of the two's-complement int8); an
 * all-zero row stores s = 0 and zero codes.  INT8 has no NaN or infinity
 * code: rows holding either are outside this contract (their codes and scale
 * are unspecified).  Same arguments and errors. */
PA_API pa_status pa_reshape_and_cache_int8(const void* k_new, const void* v_new,
                                           const int64_t* slot_mapping, int32_t T, void* k_cache,
                                           void* v_cache, float* k_scale, float* v_scale,
                                           int32_t num_blocks, int32_t block_size, int32_t Hkv,
                                           int32_t d, pa_dtype dtype, void* stream);

/* Copy-on-write block copies ([P3] section 3.3): for every layer l and pair p,
 * block pairs[p][1] of k_caches[l] and v_caches[l] becomes a bit copy of
 * block pairs[p][0].  block_bytes = block_size * Hkv * d * element size and
 * must be a multiple of 16.  A pair outside [0, num_blocks) is skipped and
 * sets PA_DEVERR_PAIR.  Destinations must be distinct and must not be sources.
 *   k_caches, v_caches (host) arrays of num_layers device pointers
 *   pairs              (device) [num_pairs][2] int32 {src, dst} */
PA_API pa_status pa_copy_blocks(void* const* k_caches, void* const* v_caches,
                                int32_t num_layers, const int32_t* pairs, int32_t num_pairs,
                                int64_t block_bytes, int32_t num_blocks, void* stream);

/* Block copies between two pools, for swapping: for each pool pair l in
 * [0, num_pools) (a layer's K or V) and each pair p, block pairs[p][1] of
 * dst_pools[l] becomes a bit copy of block pairs[p][0] of src_pools[l].  A
 * pool is device memory or pinned (page-locked) host memory the device can
 * address (e.g. cudaHostAlloc / torch pin_memory); the kernel moves the data
 * itself, so one launch covers every block of every layer.  block_bytes is
 * the bytes of one block of one pool (block_size * Hkv * d * element size,
 * a multiple of 16); pointers must be 16-byte aligned.  A pair whose source
 * is outside [0, src_blocks) or destination outside [0, dst_blocks) is
 * skipped and sets PA_DEVERR_PAIR.  Destinations must be distinct.
 *   src_pools, dst_pools (host) arrays of num_pools pointers
 *   pairs                (device or pinned host) [num_pairs][2] int32 {src, dst} */
PA_API pa_status pa_swap_blocks(const void* const* src_pools, void* const* dst_pools,
                                int32_t num_pools, const int32_t* pairs, int32_t num_pairs,
                                int64_t block_bytes, int32_t src_blocks, int32_t dst_blocks,
                                void* stream);

/* Bytes of workspace pa_decode needs for batch B, H query heads and head dim
 * d; 0 for unsupported sizes.  The workspace holds per-(sequence, KV head)
 * arrival counters and per-CTA partial results of split contexts. */
PA_API size_t pa_decode_workspace_size(int32_t B, int32_t H, int32_t d);

/* Zeroes a workspace (async on stream).  Call once after allocating it; every
 * pa_decode call leaves the counters at zero again.  A workspace serves one
 * stream at a time: pa_decode calls that overlap on the GPU must not share one.
 * A call whose bounded waits ran out (PA_DEVERR_TIMEOUT) may leave counters
 * set: zero the workspace again before reusing it. */
PA_API pa_status pa_decode_workspace_init(void* workspace, size_t bytes, void* stream);

/* Paged decode attention ([P1] section 二: attn = softmax(Q K^T / sqrt(d)) V;
 * [P3] section 1.1: the new token's query attends to every cached K/V;
 * [P1] sections 3.1 and 4.1, [P3] section 2.1: K/V reached through the block
 * table; [P4] section 2.3: query heads grouped, G = H / Hkv heads per KV head,
 * query head h reads KV head h / G).  For each sequence i with
 * n = context_lens[i] and query head h:
 *   s_j = scale * q[i][h] . K_j,  K_j = k_cache[block_tables[i][j / bs]][j % bs][h / G]
 *   out[i][h] = sum_j softmax(s)_j V_j       over j in [0, n)
 * with fp32 accumulation, rounded once to the output dtype; n == 0 gives a
 * zero row.  The caller passes scale (1/sqrt(d) for the pages' formula).
 *   q            (device) [B][H][d]
 *   k_cache, v_cache (device) [num_blocks][block_size][Hkv][d]
 *   block_tables (device) [B][max_blocks] int32
 *   context_lens (device) [B] int32, each <= max_context_len
 *   max_context_len (host) an upper bound of context_lens (sizes the split)
 *   out          (device) [B][H][d], same dtype as q
 *   workspace    (device) >= pa_decode_workspace_size(B, H, d) bytes, zeroed
 *                once by pa_decode_workspace_init
 * Blocks past a context's end are never read; a table entry outside the pool
 * is read as zeros and sets PA_DEVERR_BLOCK_ID. */
PA_API pa_status pa_decode(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int32_t max_blocks,
                           const int32_t* context_lens, int32_t max_context_len, int32_t B,
                           int32_t H, int32_t Hkv, int32_t d, int32_t block_size,
                           int32_t num_blocks, float scale, pa_dtype dtype, void* out,
                           void* workspace, size_t ws_bytes, void* stream);

/* Several query tokens per sequence over the paged cache: chunked prefill and
 * speculative verification ([P3] section 5: a long prompt's prefill is cut
 * into chunks that run between decode steps; a draft model's N tokens are
 * verified by one forward pass).  Sequence i's queries are its LAST
 * qlen_i = q_start[i+1] - q_start[i] cached tokens (their K/V already written
 * by pa_reshape_and_cache); with n = context_lens[i], query r (0-based) of
 * sequence i and query head h attend causally to tokens 0 .. n - qlen_i + r:
 *   out[q_start[i] + r][h] = sum_j softmax_j(scale * q[q_start[i] + r][h] . K_j) V_j
 * with K_j, V_j as in pa_decode (KV head h / G), fp32 accumulation, rounded
 * once to the output dtype.  qlen_i = 1 is the decode of one token; qlen_i = n
 * is the prefill of a whole prompt.  The work (64-row query tiles x 64-key
 * chunks) is split evenly over the CTAs, so a tile whose context is long is
 * shared by several CTAs whose partial results the last one merges; the
 * workspace holds their arrival tickets and partials.
 *   q            (device) [T][H][d], T = q_start[B]; out (device) [T][H][d]
 *   q_start      (device) [B + 1] int32, q_start[0] = 0, non-decreasing
 *   max_q_len    (host) an upper bound of every qlen_i (sizes the workspace)
 *   workspace    (device) >= pa_multi_query_workspace_size(B, H, Hkv, d,
 *                max_q_len) bytes, zeroed once (pa_decode_workspace_init);
 *                every call leaves the tickets at zero (zero it again after a
 *                call that set PA_DEVERR_TIMEOUT)
 *   other arguments as in pa_decode
 * qlen_i > n (or < 0), or a batch with more query rows than max_q_len allows,
 * skips the sequence (or the call) and sets PA_DEVERR_CONTEXT; a context
 * longer than its table row is cut to it and sets PA_DEVERR_TABLE_WIDTH; a
 * table entry outside the pool reads zeros and sets PA_DEVERR_BLOCK_ID. */
PA_API size_t pa_multi_query_workspace_size(int32_t B, int32_t H, int32_t Hkv, int32_t d,
                                            int32_t max_q_len);
PA_API pa_status pa_multi_query(const void* q, const int32_t* q_start, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                int32_t max_blocks, const int32_t* context_lens,
                                int32_t max_q_len, int32_t B, int32_t H, int32_t Hkv, int32_t d,
                                int32_t block_size, int32_t num_blocks, float scale,
                                pa_dtype dtype, void* out, void* workspace, size_t ws_bytes,
                                void* stream);

/* pa_multi_query on the 5th-generation tensor cores (tcgen05, accumulators in
 * tensor memory): the same result as pa_multi_query ([P3] section 5: chunked
 * prefill, speculative verification).  Rows are (query token, query head of a
 * KV head's group) pairs, token-major, in 128-row tiles against 128-key tiles.
 * Two modes, chosen per call:
 *  - max_q_len * (H / Hkv) <= 128 (every sequence's rows fit one tile:
 *    speculative verification, decode-like batches; any grouping up to 128):
 *    the (sequence, KV head, key tile) list is split evenly over one CTA per
 *    SM; pairs split between CTAs are merged through the workspace;
 *  - otherwise (prefill chunks; H / Hkv a power of two): two query tiles of a
 *    (sequence, KV head) share each key tile; no workspace is used.
 *   q_rows       rows of q and out (= q_start[B]); rows past it read as zeros
 *   max_q_len    (host) an upper bound of every qlen_i; a sequence above it is
 *                skipped and sets PA_DEVERR_CONTEXT
 *   d            128 only
 *   q, out       16-byte aligned
 *   workspace    (device, 256-byte aligned) >= pa_multi_query_tc_workspace_size
 *                bytes, zeroed once (pa_decode_workspace_init); every call leaves
 *                its tickets at zero (zero it again after a call that set
 *                PA_DEVERR_TIMEOUT); unused (may be NULL) in the second mode
 *   other arguments as in pa_multi_query
 * Errors as pa_multi_query; PA_ERR_UNSUPPORTED for other head dims or
 * groupings.  A bf16 P is rounded to 8 bits; tiles whose first row has fewer
 * than 256 keys add P's rounding residual as a second product. */
PA_API size_t pa_multi_query_tc_workspace_size(int32_t B, int32_t H, int32_t Hkv, int32_t d);
PA_API pa_status pa_multi_query_tc(const void* q, const int32_t* q_start, int32_t q_rows,
                                   const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int32_t max_blocks,
                                   const int32_t* context_lens, int32_t max_q_len, int32_t B,
                                   int32_t H, int32_t Hkv, int32_t d, int32_t block_size,
                                   int32_t num_blocks, float scale, pa_dtype dtype, void* out,
                                   void* workspace, size_t ws_bytes, void* stream);

/* pa_decode over an FP8 cache written by pa_reshape_and_cache_fp8 ([P4]
 * section 4.3).  Computes what pa_decode computes with
 *   K_j = k_scale[b][h / G][j % bs] * E4M3(k_cache[b][j % bs][h / G][:]),
 *   V_j likewise,  b = block_tables[i][j / bs],
 * for d = 128 only.  q and out are fp16/bf16 (dtype).  Both products run on
 * f16 tensor-core MMAs with fp32 accumulation: the codes widen exactly; a bf16
 * q is scaled by a power of two into f16 range first (exact for its elements
 * down to 2^-29 of its largest).  A table entry outside the pool reads zero
 * codes and scales and sets PA_DEVERR_BLOCK_ID.  Other arguments, the
 * workspace and the errors are those of pa_decode.
 *   k_cache, v_cache (device) [num_blocks][block_size][Hkv][128] uint8
 *   k_scale, v_scale (device) [num_blocks][Hkv][block_size] fp32, 16-byte aligned */
PA_API pa_status pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                               const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, int32_t max_blocks,
                               const int32_t* context_lens, int32_t max_context_len, int32_t B,
                               int32_t H, int32_t Hkv, int32_t d, int32_t block_size,
                               int32_t num_blocks, float scale, pa_dtype dtype, void* out,
                               void* workspace, size_t ws_bytes, void* stream);

/* pa_decode_fp8 over an INT8 cache (codes from pa_reshape_and_cache_int8):
 * each element is code * scale; the int8 code is widened to f16 exactly and
 * the scales are applied as for E4M3.  Otherwise as pa_decode_fp8. */
PA_API pa_status pa_decode_int8(const void* q, const void* k_cache, const void* v_cache,
                                const float* k_scale, const float* v_scale,
                                const int32_t* block_tables, int32_t max_blocks,
                                const int32_t* context_lens, int32_t max_context_len, int32_t B,
                                int32_t H, int32_t Hkv, int32_t d, int32_t block_size,
                                int32_t num_blocks, float scale, pa_dtype dtype, void* out,
                                void* workspace, size_t ws_bytes, void* stream);

/* pa_decode without a caller-supplied workspace, for callers that cannot
 * allocate device memory: code running inside an allocator's own hooks, or in
 * a process whose device memory is pre-partitioned by a host framework that
 * forbids further cudaMalloc calls.  The paper has no counterpart to this
 * entry point.  Arguments are those of pa_decode minus
 * the workspace.  Scratch lives in one file-scope device array of
 * PA_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU loading the library holds
 * until the process exits; a batch whose pa_decode_workspace_size(B, H, d)
 * exceeds it returns PA_ERR_UNSUPPORTED.  The call allocates nothing: the
 * first call on a device looks up the array's device address (so make that
 * first call before any stream capture); the address is kept per device and
 * context, so the first call after a device reset (a new context) looks it
 * up again.  Every call clears the arrival
 * counters with an async memset on `stream`.  All calls share the one array,
 * which keeps the last call's partial results: calls that overlap on the GPU
 * (different streams, or different host threads) race and must be serialised
 * by the caller. */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)
PA_API pa_status pa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int32_t max_blocks,
                                   const int32_t* context_lens, int32_t max_context_len,
                                   int32_t B, int32_t H, int32_t Hkv, int32_t d,
                                   int32_t block_size, int32_t num_blocks, float scale,
                                   pa_dtype dtype, void* out, void* stream);

/* ------------------------------------------------------------------------
 * Decode step executor: one call per step for one layer's whole hot path --
 * the block manager's bookkeeping on the host ([P1] section 3.2: a slot for
 * each new token, block tables for the kernel; [P3] section 3.3: a shared
 * last block is copied before it is written), one host->device copy of the
 * step's inputs and tables, pa_copy_blocks when copy-on-write arises,
 * pa_reshape_and_cache, pa_decode and one device->host copy of the output
 * (their _fp8 / _int8 forms over an 8-bit cache).
 * The two kernels are captured once per slot, at creation, into a CUDA graph
 * owned by the executor and replayed every step on the caller's stream; the
 * input copy runs on the executor's own copy-in stream and the output copy on
 * its copy-out stream, so a step's inputs travel while the previous step's
 * decode runs and its output travels while the next one's does.  The caller
 * owns the staging buffers: a page-locked host buffer (cudaHostAlloc, or a pinned
 * torch tensor) and a device buffer, each desc.depth slots of
 * pa_step_layout.total bytes (slot i at byte i * total), 256-byte aligned.
 * In a slot the caller writes a step's q [B][H][d] and new k / v [B][Hkv][d]
 * (dtype) at offsets q, k_new, v_new of the host buffer; the executor writes
 * slot_mapping, block_tables, context_lens and cow_pairs there itself and
 * leaves the output [B][H][d] at offset out.  Step n uses slot n % depth; with
 * two slots a step can be submitted while the one before it still runs.  The
 * paper has no counterpart to the executor object; it exists so that a
 * serving loop pays one launch per step and its host bookkeeping can overlap
 * the device work.  Like the allocator it drives, an executor is not
 * thread-safe: one host thread submits and waits at a time.
 * ---------------------------------------------------------------------- */
typedef struct pa_step pa_step;

typedef struct pa_step_desc {
    int32_t B;                /* sequences per step, 1 .. 4096 */
    int32_t H, Hkv, d;        /* query heads, KV heads, head dim (64 or 128) */
    int32_t block_size;       /* 8, 16 or 32 */
    int32_t num_blocks;       /* blocks of the cache pool */
    int32_t max_blocks;       /* table width exported every step */
    int32_t max_context_len;  /* bound of every context length, <= max_blocks * block_size */
    pa_dtype dtype;           /* of q, k_new, v_new, the output and a 16-bit cache */
    float scale;              /* attention scale, 1/sqrt(d) for the pages' formula */
    int32_t q8;               /* 8-bit cache with per-(token, KV head) scales (d = 128):
                                 0 none, 1 E4M3 (pa_decode_fp8), 2 INT8 (pa_decode_int8) */
    int32_t depth;            /* staging slots (and graphs): 1 or 2 */
} pa_step_desc;

typedef struct pa_step_layout {  /* byte offsets inside one slot of either staging buffer */
    size_t q, k_new, v_new, slot_mapping, block_tables, context_lens;
    size_t in_bytes;             /* [0, in_bytes) is copied host->device each step */
    size_t cow_pairs, out;       /* copy-on-write pairs [B][2] int32; output [B][H][d] */
    size_t total;                /* bytes of one slot */
} pa_step_layout;

/* Layout of the staging buffers for desc; PA_ERR_INVALID for a bad desc. */
PA_API pa_status pa_step_layout_get(const pa_step_desc* desc, pa_step_layout* out);

/* Creates an executor for one layer's caches k_cache / v_cache (device,
 * [num_blocks][block_size][Hkv][d], dtype or, with q8, uint8 codes plus
 * k_scale / v_scale [num_blocks][Hkv][block_size] fp32; the scales are NULL
 * otherwise) and the allocator alloc (all must outlive it).  workspace (device, >= pa_decode_workspace_size(B, H, d) bytes, zeroed
 * once) is the decode's.  Captures the graph on a private stream; nothing
 * runs.  PA_ERR_INVALID for bad arguments, misaligned staging, or an allocator
 * whose pool size or block size differs from desc's. */
PA_API pa_status pa_step_create(const pa_step_desc* desc, pa_allocator* alloc, void* k_cache,
                                void* v_cache, float* k_scale, float* v_scale, void* host_stage,
                                void* dev_stage, void* workspace, size_t ws_bytes,
                                pa_step** out);

/* Submits one decode step for the B sequences seq_ids (host) without waiting
 * for it, in slot n % depth (n = steps submitted so far; *slot receives it,
 * nullable), after waiting for the step that last used that slot: appends one
 * token to each sequence (pa_append_batch), exports the tables, copies the
 * slot's inputs to the device on the copy-in stream, and on `stream` -- once
 * they are there -- issues the copy-on-write copies the appends need and
 * launches the slot's graph; the output copy follows on the copy-out stream.
 * Work the caller later orders on `stream` runs after the step's decode but
 * not necessarily after its output copy: pa_step_wait is what guarantees the
 * output is on the host.  Steps may be submitted on different streams: every
 * step's copy-on-write, append and decode wait for the previous step's decode
 * (they share the cache and the decode workspace), so alternating streams
 * orders the kernels as one stream would.  A sequence whose length after the append would
 * exceed max_context_len or max_blocks * block_size returns PA_ERR_BOUNDS
 * before anything changes; allocator errors are those of pa_append_batch (all
 * or nothing).  After the appends, a slot, table entry or copy pair outside
 * the pool (an allocator that does not match the cache) returns PA_ERR_BOUNDS
 * and a failed CUDA call PA_ERR_CUDA, both before any launch, with the appends
 * done.  Write a step's inputs into its slot before submitting it, and only
 * once the slot's previous step is done (pa_step_wait). */
PA_API pa_status pa_step_submit(pa_step* s, const int64_t* seq_ids, void* stream, int32_t* slot);

/* Waits for the last step submitted in `slot`; its output is then in the
 * slot's host region.  PA_ERR_INVALID for a slot outside 0 .. depth - 1. */
PA_API pa_status pa_step_wait(pa_step* s, int32_t slot);

/* pa_step_submit followed by pa_step_wait of its slot. */
PA_API pa_status pa_step_run(pa_step* s, const int64_t* seq_ids, void* stream);

/* Waits for every submitted step's output and for the executor's own copy
 * streams, then frees the executor (graphs, streams, events); the staging
 * buffers and workspace stay the caller's.  After a submit that failed with
 * PA_ERR_CUDA, kernels it did launch on the caller's stream are the caller's
 * to wait for (a stream synchronize) before freeing what they use. */
PA_API void pa_step_destroy(pa_step* s);

/* Synchronises `stream`, returns the current device's error word in *flags
 * (host, nullable) and clears it.  Returns PA_ERR_BOUNDS or PA_ERR_TIMEOUT if
 * any bit was set, PA_ERR_CUDA if the stream reports an error, else PA_OK. */
PA_API pa_status pa_check_device_errors(void* stream, uint32_t* flags);

/* Failure-path check: launches one CTA that waits, with the same bounded wait
 * the decode pipeline uses on its mbarriers, on an mbarrier that nothing ever
 * arrives on.  After limit_us microseconds (1 .. 1,000,000) the wait gives up
 * and sets PA_DEVERR_TIMEOUT in the device error word; the context stays
 * usable.  The paper has no counterpart; it lets a test exercise the timeout
 * path without stalling a real pipeline. */
PA_API pa_status pa_selftest_wait_timeout(uint32_t limit_us, void* stream);

/* Measurement aid: the throughput ceiling of the legacy tensor-core path the
 * attention kernels use (mma.sync m16n8k16, f16 or -- bf16 != 0 -- bf16
 * operands, fp32 accumulation).  Launches two CTAs of eight warps per SM; each
 * warp issues `iters` (1 .. 2^20) rounds of 8 independent MMAs from registers
 * and writes one float per thread to sink (device, >= SMs x 2 x 256 floats,
 * contents meaningless).  *flops (host) receives the launch's floating-point
 * operations (2 per multiply-add); time the launch with events on `stream`.
 * PA_ERR_INVALID for bad arguments or a small sink.  The paper has no
 * counterpart; it gives the kernels' MMA-bound work a denominator measured on
 * the same path. */
PA_API pa_status pa_measure_mma_ceiling(int32_t bf16, int32_t iters, float* sink,
                                        size_t sink_bytes, int64_t* flops, void* stream);

/* Number of decode CTAs pa_decode launches on the current device (one per SM
 * times the resident CTAs per SM), for launch accounting; 0 on error. */
PA_API int32_t pa_decode_grid_size(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
