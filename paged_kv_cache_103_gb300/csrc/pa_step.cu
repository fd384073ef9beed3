// Decode step executor: one C-ABI call per step runs the whole hot path of one
// layer.  The host part is the block manager's per-step bookkeeping
// ("LLM推理优化：vLLM PagedAttention深度解析与工程实践", section 3.2: a slot
// per new token, block tables handed to the kernel; "vLLM 深度拆解：当大模型
// 推理学会「分页注意力」", section 3.3: copy-on-write of a shared last block);
// the device part is one host->device copy of the step's inputs and tables,
// the append (pa_reshape_and_cache), the attention (pa_decode) and one
// device->host copy of the output.  The two kernels are captured once per
// staging slot into a CUDA graph and replayed every step on the caller's
// stream; the copies run on the executor's own copy-in and copy-out streams,
// ordered against the graph by events.  With two staging slots a step can be
// submitted while the previous one still runs: the host bookkeeping and the
// input copy of step n + 1 overlap the decode of step n, and the output copy
// of step n overlaps the decode of step n + 1.
#include <cuda_runtime.h>

#include <new>

#include "pa.h"
#include "pa_common.cuh"

namespace {

constexpr int kMaxDepth = 2;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool desc_ok(const pa_step_desc* d) {
    return d && d->B > 0 && d->B <= 4096 && d->H > 0 && d->Hkv > 0 && d->H % d->Hkv == 0 &&
           (d->d == 64 || d->d == 128) &&
           (d->block_size == 8 || d->block_size == 16 || d->block_size == 32) &&
           d->num_blocks > 0 && d->max_blocks > 0 && d->max_context_len > 0 &&
           (int64_t)d->max_context_len <= (int64_t)d->max_blocks * d->block_size &&
           (d->dtype == PA_F16 || d->dtype == PA_BF16) && d->q8 >= 0 && d->q8 <= 2 &&
           (d->q8 == 0 || d->d == 128) && d->depth >= 1 && d->depth <= kMaxDepth;
}

}  // namespace

struct pa_step {
    pa_step_desc desc;
    pa_step_layout lay;     // offsets inside one slot; slot i starts at i * lay.total
    pa_allocator* alloc;
    void* k_cache;
    void* v_cache;
    float* k_scale;         // 8-bit caches only
    float* v_scale;
    unsigned char* host;    // pinned staging, depth slots
    unsigned char* dev;     // device staging, depth slots
    int64_t block_bytes;    // one block of one cache (codes for FP8)
    int64_t submitted;      // steps submitted so far (the next uses slot submitted % depth)
    cudaStream_t in_stream;   // host->device copies of the inputs
    cudaStream_t out_stream;  // device->host copies of the outputs
    cudaGraphExec_t exec[kMaxDepth];  // per slot: the append and the decode
    cudaEvent_t in_done[kMaxDepth];   // the slot's inputs are on the device
    cudaEvent_t comp_done[kMaxDepth]; // the slot's decode has finished
    cudaEvent_t done[kMaxDepth];      // the slot's output is on the host
    bool pending[kMaxDepth];
};

namespace {

void release(pa_step* s) {
    // Copies of a submit that failed half way are not marked pending: drain the
    // copy streams too, so that nothing still reads or writes the caller's
    // staging once this returns.
    if (s->in_stream) cudaStreamSynchronize(s->in_stream);
    if (s->out_stream) cudaStreamSynchronize(s->out_stream);
    for (int i = 0; i < kMaxDepth; ++i) {
        if (s->pending[i]) cudaEventSynchronize(s->done[i]);
        if (s->exec[i]) cudaGraphExecDestroy(s->exec[i]);
        if (s->in_done[i]) cudaEventDestroy(s->in_done[i]);
        if (s->comp_done[i]) cudaEventDestroy(s->comp_done[i]);
        if (s->done[i]) cudaEventDestroy(s->done[i]);
    }
    if (s->in_stream) cudaStreamDestroy(s->in_stream);
    if (s->out_stream) cudaStreamDestroy(s->out_stream);
    delete s;
}

// Captures slot i's graph on the private stream cap: the append and the
// decode over the slot's device staging.  The copies in and out are issued
// per step on the executor's copy streams (pa_step_submit), so that the next
// step's inputs travel while this step's decode runs.
pa_status capture(pa_step* s, int i, void* workspace, size_t ws_bytes, cudaStream_t cap) {
    const pa_step_desc* d = &s->desc;
    const pa_step_layout& L = s->lay;
    unsigned char* g = s->dev + (size_t)i * L.total;
    pa_status st = PA_OK;
    cudaGraph_t graph = nullptr;
    if (cudaStreamBeginCapture(cap, cudaStreamCaptureModeRelaxed) != cudaSuccess) return PA_ERR_CUDA;
    const int64_t* slots = reinterpret_cast<const int64_t*>(g + L.slot_mapping);
    const int32_t* tables = reinterpret_cast<const int32_t*>(g + L.block_tables);
    const int32_t* lens = reinterpret_cast<const int32_t*>(g + L.context_lens);
    if (st == PA_OK && d->q8)
        st = (d->q8 == 1 ? pa_reshape_and_cache_fp8 : pa_reshape_and_cache_int8)(g + L.k_new, g + L.v_new, slots, d->B, s->k_cache,
                                      s->v_cache, s->k_scale, s->v_scale, d->num_blocks,
                                      d->block_size, d->Hkv, d->d, d->dtype, cap);
    else if (st == PA_OK)
        st = pa_reshape_and_cache(g + L.k_new, g + L.v_new, slots, d->B, s->k_cache, s->v_cache,
                                  d->num_blocks, d->block_size, d->Hkv, d->d, d->dtype, cap);
    if (st == PA_OK && d->q8)
        st = (d->q8 == 1 ? pa_decode_fp8 : pa_decode_int8)(g + L.q, s->k_cache, s->v_cache, s->k_scale, s->v_scale, tables,
                           d->max_blocks, lens, d->max_context_len, d->B, d->H, d->Hkv, d->d,
                           d->block_size, d->num_blocks, d->scale, d->dtype, g + L.out, workspace,
                           ws_bytes, cap);
    else if (st == PA_OK)
        st = pa_decode(g + L.q, s->k_cache, s->v_cache, tables, d->max_blocks, lens,
                       d->max_context_len, d->B, d->H, d->Hkv, d->d, d->block_size, d->num_blocks,
                       d->scale, d->dtype, g + L.out, workspace, ws_bytes, cap);
    // End the capture whatever happened, so the stream is usable again.
    if (cudaStreamEndCapture(cap, &graph) != cudaSuccess && st == PA_OK) st = PA_ERR_CUDA;
    if (st == PA_OK && cudaGraphInstantiate(&s->exec[i], graph, 0) != cudaSuccess) st = PA_ERR_CUDA;
    if (graph) cudaGraphDestroy(graph);
    return st;
}

}  // namespace

extern "C" {

PA_API pa_status pa_step_layout_get(const pa_step_desc* d, pa_step_layout* out) {
    if (!desc_ok(d) || !out) return PA_ERR_INVALID;
    const size_t e = 2;
    pa_step_layout L;
    size_t at = 0;
    L.q = at;
    at = align256(at + (size_t)d->B * d->H * d->d * e);
    L.k_new = at;
    at = align256(at + (size_t)d->B * d->Hkv * d->d * e);
    L.v_new = at;
    at = align256(at + (size_t)d->B * d->Hkv * d->d * e);
    L.slot_mapping = at;
    at = align256(at + (size_t)d->B * sizeof(int64_t));
    L.block_tables = at;
    at = align256(at + (size_t)d->B * d->max_blocks * sizeof(int32_t));
    L.context_lens = at;
    at = align256(at + (size_t)d->B * sizeof(int32_t));
    L.in_bytes = at;
    L.cow_pairs = at;
    at = align256(at + (size_t)d->B * 2 * sizeof(int32_t));
    L.out = at;
    at = align256(at + (size_t)d->B * d->H * d->d * e);
    L.total = at;
    *out = L;
    return PA_OK;
}

PA_API pa_status pa_step_create(const pa_step_desc* d, pa_allocator* alloc, void* k_cache,
                                void* v_cache, float* k_scale, float* v_scale, void* host_stage,
                                void* dev_stage, void* workspace, size_t ws_bytes,
                                pa_step** out) {
    if (!desc_ok(d) || !alloc || !k_cache || !v_cache || !host_stage || !dev_stage ||
        !workspace || !out)
        return PA_ERR_INVALID;
    if (d->q8 && (!k_scale || !v_scale)) return PA_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(host_stage) | reinterpret_cast<uintptr_t>(dev_stage)) & 255u)
        return PA_ERR_INVALID;
    if (ws_bytes < pa_decode_workspace_size(d->B, d->H, d->d)) return PA_ERR_INVALID;
    // the allocator's pool must be the cache's: its blocks and slots index it
    pa_alloc_stats as;
    if (pa_alloc_stats_get(alloc, &as) != PA_OK || as.num_blocks != d->num_blocks ||
        as.block_size != d->block_size)
        return PA_ERR_INVALID;
    *out = nullptr;
    pa_step* s = new (std::nothrow) pa_step;
    if (!s) return PA_ERR_OOM;
    s->desc = *d;
    pa_step_layout_get(d, &s->lay);
    s->alloc = alloc;
    s->k_cache = k_cache;
    s->v_cache = v_cache;
    s->k_scale = d->q8 ? k_scale : nullptr;
    s->v_scale = d->q8 ? v_scale : nullptr;
    s->host = static_cast<unsigned char*>(host_stage);
    s->dev = static_cast<unsigned char*>(dev_stage);
    s->block_bytes = (int64_t)d->block_size * d->Hkv * d->d * (d->q8 ? 1 : 2);
    s->submitted = 0;
    s->in_stream = s->out_stream = nullptr;
    for (int i = 0; i < kMaxDepth; ++i) {
        s->exec[i] = nullptr;
        s->in_done[i] = s->comp_done[i] = s->done[i] = nullptr;
        s->pending[i] = false;
    }
    // One-time set-up of the device error word and SM count, outside the capture.
    if (!pa::device_error_word() || !pa::device_sm_count()) {
        release(s);
        return PA_ERR_CUDA;
    }
    // The graphs are captured on a private stream; they can be launched on any.
    cudaStream_t cap = nullptr;
    if (cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) != cudaSuccess) {
        release(s);
        return PA_ERR_CUDA;
    }
    pa_status st = PA_OK;
    if (cudaStreamCreateWithFlags(&s->in_stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&s->out_stream, cudaStreamNonBlocking) != cudaSuccess)
        st = PA_ERR_CUDA;
    for (int i = 0; i < d->depth && st == PA_OK; ++i) {
        if (cudaEventCreateWithFlags(&s->in_done[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&s->comp_done[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&s->done[i], cudaEventDisableTiming) != cudaSuccess)
            st = PA_ERR_CUDA;
        else
            st = capture(s, i, workspace, ws_bytes, cap);
    }
    cudaStreamDestroy(cap);
    if (st != PA_OK) {
        release(s);
        return st;
    }
    *out = s;
    return PA_OK;
}

PA_API pa_status pa_step_submit(pa_step* s, const int64_t* seq_ids, void* stream,
                                int32_t* slot_out) {
    if (!s || !seq_ids) return PA_ERR_INVALID;
    const pa_step_desc& d = s->desc;
    const pa_step_layout& L = s->lay;
    const int slot = (int)(s->submitted % d.depth);
    // The slot's staging is reused: the step that last used it must be done.
    if (s->pending[slot]) {
        if (cudaEventSynchronize(s->done[slot]) != cudaSuccess) return PA_ERR_CUDA;
        s->pending[slot] = false;
    }
    unsigned char* h = s->host + (size_t)slot * L.total;
    unsigned char* g = s->dev + (size_t)slot * L.total;
    // Every sequence must still fit the executor's bounds after the append;
    // checked first so that a refusal changes nothing.
    for (int32_t i = 0; i < d.B; ++i) {
        int32_t len = 0, nb = 0;
        const pa_status st = pa_seq_info(s->alloc, seq_ids[i], &len, &nb);
        if (st != PA_OK) return st;
        if (len + 1 > d.max_context_len || (len + d.block_size) / d.block_size > d.max_blocks)
            return PA_ERR_BOUNDS;
    }
    int32_t ncow = 0;
    int32_t* pairs = reinterpret_cast<int32_t*>(h + L.cow_pairs);
    pa_status st = pa_append_batch(s->alloc, seq_ids, d.B,
                                   reinterpret_cast<int64_t*>(h + L.slot_mapping), pairs, &ncow);
    if (st != PA_OK) return st;
    st = pa_export(s->alloc, seq_ids, d.B, d.max_blocks,
                   reinterpret_cast<int32_t*>(h + L.block_tables),
                   reinterpret_cast<int32_t*>(h + L.context_lens));
    if (st != PA_OK) return st;
    // What the graph will read, checked on the host before anything launches:
    // every new slot inside the pool, every used table entry a pool block.
    {
        const int64_t* sm = reinterpret_cast<const int64_t*>(h + L.slot_mapping);
        const int32_t* tb = reinterpret_cast<const int32_t*>(h + L.block_tables);
        const int32_t* ln = reinterpret_cast<const int32_t*>(h + L.context_lens);
        const int64_t nslots = (int64_t)d.num_blocks * d.block_size;
        for (int32_t i = 0; i < d.B; ++i) {
            if (sm[i] < 0 || sm[i] >= nslots || ln[i] < 1 || ln[i] > d.max_context_len)
                return PA_ERR_BOUNDS;
            const int32_t used = (ln[i] + d.block_size - 1) / d.block_size;
            for (int32_t j = 0; j < used; ++j) {
                const int32_t b = tb[(int64_t)i * d.max_blocks + j];
                if (b < 0 || b >= d.num_blocks) return PA_ERR_BOUNDS;
            }
        }
        for (int32_t p = 0; p < ncow; ++p)
            if (pairs[2 * p] < 0 || pairs[2 * p] >= d.num_blocks || pairs[2 * p + 1] < 0 ||
                pairs[2 * p + 1] >= d.num_blocks)
                return PA_ERR_BOUNDS;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    // Inputs in on the copy-in stream: nothing on the device still reads this
    // slot (its last step's output copy is done, waited above), so the copy
    // can run while the previous step's decode does.
    if (cudaMemcpyAsync(g, h, L.in_bytes, cudaMemcpyHostToDevice, s->in_stream) != cudaSuccess)
        return PA_ERR_CUDA;
    // From here on a failure returns with the copy queued: wait for it, so
    // the slot's host staging is free again when the caller retries.
    auto fail = [&](pa_status e) {
        cudaStreamSynchronize(s->in_stream);
        return e;
    };
    if (cudaEventRecord(s->in_done[slot], s->in_stream) != cudaSuccess ||
        cudaStreamWaitEvent(cs, s->in_done[slot], 0) != cudaSuccess)
        return fail(PA_ERR_CUDA);
    // Every step's kernels share the decode workspace and the cache: this
    // step's copy-on-write, append and decode start after the previous step's
    // decode, whichever stream that one was submitted on.
    if (s->submitted > 0 &&
        cudaStreamWaitEvent(cs, s->comp_done[(s->submitted - 1) % d.depth], 0) != cudaSuccess)
        return fail(PA_ERR_CUDA);
    if (ncow > 0) {
        // Copy-on-write before the step's append writes the new token.
        int32_t* dpairs = reinterpret_cast<int32_t*>(g + L.cow_pairs);
        if (cudaMemcpyAsync(dpairs, pairs, (size_t)ncow * 2 * sizeof(int32_t),
                            cudaMemcpyHostToDevice, cs) != cudaSuccess)
            return fail(PA_ERR_CUDA);
        void* kc = s->k_cache;
        void* vc = s->v_cache;
        st = pa_copy_blocks(&kc, &vc, 1, dpairs, ncow, s->block_bytes, d.num_blocks, cs);
        if (st != PA_OK) return fail(st);
        if (d.q8) {   // and the blocks' scales, [num_blocks][Hkv][block_size] fp32
            void* ks = s->k_scale;
            void* vs = s->v_scale;
            st = pa_copy_blocks(&ks, &vs, 1, dpairs, ncow, (int64_t)d.Hkv * d.block_size * 4,
                                d.num_blocks, cs);
            if (st != PA_OK) return fail(st);
        }
    }
    // The append and the decode, in order on the caller's stream (so one step's
    // copy-on-write and append follow the previous step's decode); then the
    // output out on the copy-out stream, while the next step's decode runs.
    if (cudaGraphLaunch(s->exec[slot], cs) != cudaSuccess ||
        cudaEventRecord(s->comp_done[slot], cs) != cudaSuccess ||
        cudaStreamWaitEvent(s->out_stream, s->comp_done[slot], 0) != cudaSuccess ||
        cudaMemcpyAsync(h + L.out, g + L.out, (size_t)d.B * d.H * d.d * 2, cudaMemcpyDeviceToHost,
                        s->out_stream) != cudaSuccess ||
        cudaEventRecord(s->done[slot], s->out_stream) != cudaSuccess)
        return fail(PA_ERR_CUDA);
    s->pending[slot] = true;
    ++s->submitted;
    if (slot_out) *slot_out = slot;
    return PA_OK;
}

PA_API pa_status pa_step_wait(pa_step* s, int32_t slot) {
    if (!s || slot < 0 || slot >= s->desc.depth) return PA_ERR_INVALID;
    if (!s->pending[slot]) return PA_OK;
    if (cudaEventSynchronize(s->done[slot]) != cudaSuccess) return PA_ERR_CUDA;
    s->pending[slot] = false;
    return PA_OK;
}

PA_API pa_status pa_step_run(pa_step* s, const int64_t* seq_ids, void* stream) {
    int32_t slot = 0;
    const pa_status st = pa_step_submit(s, seq_ids, stream, &slot);
    return st != PA_OK ? st : pa_step_wait(s, slot);
}

PA_API void pa_step_destroy(pa_step* s) {
    if (s) release(s);
}

}  // extern "C"
