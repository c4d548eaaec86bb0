// Two-slot VRAM pool fed from a pinned host store by the copy engine.
//
// "Can You Fine-Tune Llama 3.1 8B on a 4GB GPU? Soup's Layer Streaming Explained", section
// "How Soup's layer streaming actually works", steps 2-4: the frozen decoder weights live in
// page-locked host memory; the current layer is copied into a small pool of reusable VRAM
// buffers while the next one is prefetched into another; a finished layer's buffer is reused;
// the backward pass reads every layer again.  "Fine tune an 8B model on a 4GB laptop GPU
// (Soup setup)", section "Step 2, train": the pool is two buffers, prefetched one ahead.
//
// Per slot the pool keeps a copy-done event per chunk of the layer image (recorded on the
// copy stream after that chunk's cudaMemcpyAsync), which gates the compute stream in
// stream_pool_wait / stream_pool_wait_range, and a slot-free event (recorded on the compute
// stream by stream_pool_release), which gates the next copy into that slot.  With one chunk
// (the default) a layer is one copy.  With several, a layer's chunks are copied in ascending
// or descending order, so compute that needs only the first chunk in copy order can start
// while the others are still in flight ("Can You Fine-Tune Llama 3.1 8B on a 4GB GPU? Soup's
// Layer Streaming Explained", section "Did a correctness bug invalidate the Llama 3.1 8B
// result?" is about how a layer is split into transfers; here the split never changes what
// the kernels read, only when).  The host never blocks on the GPU except in the optional
// bounded poll of the waits.
#include <string.h>

#include <chrono>
#include <thread>
#include <vector>

#include "lsn_internal.h"

using namespace lsn;

namespace {

enum SlotState { kEmpty = 0, kLoading = 1, kInUse = 2, kReleased = 3 };
constexpr int kMaxChunks = 8;

struct Slot {
    void* dev = nullptr;
    int layer = -1;
    int state = kEmpty;
    bool free_recorded = false;
    bool reverse = false;                    // chunk copy order of the layer it holds
    cudaEvent_t copy_done[kMaxChunks] = {};  // per chunk
    cudaEvent_t slot_free = nullptr;
};

struct Timing {
    cudaEvent_t start, end;
    size_t bytes;
    int chunk;
};

void CUDART_CB sleep_host(void* arg) {
    const long us = (long)(reinterpret_cast<uintptr_t>(arg));
    std::this_thread::sleep_for(std::chrono::microseconds(us));
}

}  // namespace

struct lsn_pool {
    const uint8_t* store = nullptr;
    size_t store_bytes = 0;
    std::vector<size_t> offset;
    size_t layer_bytes = 0;
    int n_layers = 0;
    cudaStream_t copy = nullptr;
    Slot slot[2];
    int next_slot = 0;
    bool reuse = false;
    long delay_us = 0;
    std::vector<Timing> pending;
    std::vector<Timing> spare;
    lsn_pool_stats st{};
    int n_chunks = 1;
    size_t chunk_off[kMaxChunks + 1] = {0};   // chunk c = [chunk_off[c], chunk_off[c + 1])
    lsn_pool_stats chunk_st[kMaxChunks] = {};
};

static int harvest(lsn_pool* p, bool block) {
    size_t keep = 0;
    for (size_t i = 0; i < p->pending.size(); ++i) {
        Timing& t = p->pending[i];
        cudaError_t q = block ? cudaEventSynchronize(t.end) : cudaEventQuery(t.end);
        if (q == cudaErrorNotReady) {
            p->pending[keep++] = t;
            continue;
        }
        if (q != cudaSuccess) return cuda_fail(q, "stream pool: copy event");
        float ms = 0.f;
        LSN_CUDA_TRY(cudaEventElapsedTime(&ms, t.start, t.end));
        p->st.copy_ms += ms;
        p->st.bytes_copied += t.bytes;
        if (t.chunk == 0 || p->n_chunks == 1) p->st.copies += 1;   // one per layer copied
        lsn_pool_stats& cs = p->chunk_st[t.chunk];
        cs.copy_ms += ms;
        cs.bytes_copied += t.bytes;
        cs.copies += 1;
        p->spare.push_back(t);
    }
    p->pending.resize(keep);
    return LSN_OK;
}

static bool is_pinned(const void* ptr) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost;
}

extern "C" {

int stream_pool_create(const void* pinned_store, size_t store_bytes, const size_t* layer_offset,
                       size_t layer_bytes, int n_layers, void* slot0, void* slot1, void* copy_stream,
                       int first_slot, int reuse_resident, lsn_pool** out) {
    if (!out) return fail(LSN_EINVAL, "stream_pool_create: out is NULL");
    *out = nullptr;
    if (!pinned_store || !layer_offset || !slot0 || !slot1 || n_layers < 1 || layer_bytes == 0 ||
        store_bytes < layer_bytes || (first_slot != 0 && first_slot != 1))
        return fail(LSN_EINVAL, "stream_pool_create: bad arguments");
    if ((reinterpret_cast<uintptr_t>(slot0) & 255) || (reinterpret_cast<uintptr_t>(slot1) & 255))
        return fail(LSN_EINVAL, "stream_pool_create: slots must be 256-byte aligned");
    for (int l = 0; l < n_layers; ++l)
        if (layer_offset[l] > store_bytes || store_bytes - layer_offset[l] < layer_bytes)
            return fail(LSN_EINVAL, "stream_pool_create: layer %d lies outside the store", l);
    const uint8_t* s = static_cast<const uint8_t*>(pinned_store);
    if (!is_pinned(s) || !is_pinned(s + store_bytes - 1))
        return fail(LSN_EINVAL, "stream_pool_create: the host store is not page-locked");
    lsn_pool* p = new (std::nothrow) lsn_pool();
    if (!p) return fail(LSN_ENOMEM, "stream_pool_create: out of host memory");
    p->store = s;
    p->store_bytes = store_bytes;
    p->offset.assign(layer_offset, layer_offset + n_layers);
    p->layer_bytes = layer_bytes;
    p->n_layers = n_layers;
    p->copy = static_cast<cudaStream_t>(copy_stream);
    p->slot[0].dev = slot0;
    p->slot[1].dev = slot1;
    p->next_slot = first_slot;
    p->reuse = reuse_resident != 0;
    p->chunk_off[0] = 0;
    p->chunk_off[1] = layer_bytes;
    for (int i = 0; i < 2; ++i) {
        cudaError_t e = cudaSuccess;
        for (int c = 0; c < kMaxChunks && e == cudaSuccess; ++c)
            e = cudaEventCreateWithFlags(&p->slot[i].copy_done[c], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->slot[i].slot_free, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            stream_pool_destroy(p);
            return cuda_fail(e, "stream_pool_create: cudaEventCreate");
        }
    }
    *out = p;
    return LSN_OK;
}

int stream_pool_set_chunks(lsn_pool* p, int n_chunks, const size_t* chunk_offset) {
    if (!p || n_chunks < 1 || n_chunks > kMaxChunks || (n_chunks > 1 && !chunk_offset))
        return fail(LSN_EINVAL, "stream_pool_set_chunks: need 1..%d chunks and their offsets", kMaxChunks);
    for (int i = 0; i < 2; ++i)
        if (p->slot[i].state == kLoading || p->slot[i].state == kInUse)
            return fail(LSN_ESTATE, "stream_pool_set_chunks: a slot still holds layer %d", p->slot[i].layer);
    size_t off[kMaxChunks + 1];
    off[0] = 0;
    for (int c = 1; c < n_chunks; ++c) {
        off[c] = chunk_offset[c];
        if (off[c] <= off[c - 1] || off[c] >= p->layer_bytes || off[c] % 256)
            return fail(LSN_EINVAL, "stream_pool_set_chunks: chunk %d must start after chunk %d, inside the layer "
                                    "and on a 256-byte boundary", c, c - 1);
    }
    if (n_chunks > 1 && chunk_offset[0] != 0) return fail(LSN_EINVAL, "stream_pool_set_chunks: chunk 0 starts at 0");
    off[n_chunks] = p->layer_bytes;
    LSN_CUDA_TRY(cudaStreamSynchronize(p->copy));
    int rc = harvest(p, true);
    if (rc) return rc;
    p->n_chunks = n_chunks;
    memcpy(p->chunk_off, off, sizeof(size_t) * (n_chunks + 1));
    for (int i = 0; i < 2; ++i) {   // the bytes in the slots were copied under the old chunking
        p->slot[i].layer = -1;
        p->slot[i].state = kEmpty;
    }
    memset(p->chunk_st, 0, sizeof(p->chunk_st));
    return LSN_OK;
}

int stream_pool_prefetch_ex(lsn_pool* p, int layer, int reverse) {
    if (!p || layer < 0 || layer >= p->n_layers) return fail(LSN_EINVAL, "stream_pool_prefetch: bad layer");
    if (p->reuse) {
        for (int i = 0; i < 2; ++i) {
            Slot& sl = p->slot[i];
            if (sl.layer == layer && sl.state == kReleased) {
                sl.state = kLoading;          // bytes are already in the slot (every event recorded)
                p->next_slot = i ^ 1;
                p->st.skipped += 1;
                return LSN_OK;
            }
        }
    }
    const int si = p->next_slot;
    Slot& sl = p->slot[si];
    if (sl.state == kLoading || sl.state == kInUse)
        return fail(LSN_ESTATE, "stream_pool_prefetch: slot %d still holds layer %d (not released)", si, sl.layer);
    harvest(p, false);
    if (sl.free_recorded) LSN_CUDA_TRY(cudaStreamWaitEvent(p->copy, sl.slot_free, 0));
    if (p->delay_us > 0)
        LSN_CUDA_TRY(cudaLaunchHostFunc(p->copy, sleep_host, reinterpret_cast<void*>((uintptr_t)p->delay_us)));
    for (int j = 0; j < p->n_chunks; ++j) {
        const int c = reverse ? p->n_chunks - 1 - j : j;
        Timing t;
        if (!p->spare.empty()) {
            t = p->spare.back();
            p->spare.pop_back();
        } else {
            LSN_CUDA_TRY(cudaEventCreate(&t.start));
            cudaError_t e = cudaEventCreate(&t.end);
            if (e != cudaSuccess) {
                cudaEventDestroy(t.start);
                return cuda_fail(e, "cudaEventCreate");
            }
        }
        const size_t b0 = p->chunk_off[c], n = p->chunk_off[c + 1] - b0;
        t.bytes = n;
        t.chunk = c;
        LSN_CUDA_TRY(cudaEventRecord(t.start, p->copy));
        LSN_CUDA_TRY(cudaMemcpyAsync(static_cast<uint8_t*>(sl.dev) + b0, p->store + p->offset[layer] + b0, n,
                                     cudaMemcpyHostToDevice, p->copy));
        LSN_CUDA_TRY(cudaEventRecord(t.end, p->copy));
        LSN_CUDA_TRY(cudaEventRecord(sl.copy_done[c], p->copy));
        p->pending.push_back(t);
    }
    sl.layer = layer;
    sl.state = kLoading;
    sl.reverse = reverse != 0;
    p->next_slot = si ^ 1;
    return LSN_OK;
}

int stream_pool_prefetch(lsn_pool* p, int layer) { return stream_pool_prefetch_ex(p, layer, 0); }

int stream_pool_wait_range(lsn_pool* p, int layer, size_t begin, size_t end, void* compute_stream,
                           const void** dev_image, int timeout_ms) {
    if (!p || !dev_image || begin >= end || end > p->layer_bytes)
        return fail(LSN_EINVAL, "stream_pool_wait: bad arguments");
    int si = -1;
    for (int i = 0; i < 2; ++i)
        if (p->slot[i].layer == layer && (p->slot[i].state == kLoading || p->slot[i].state == kInUse)) si = i;
    if (si < 0) return fail(LSN_ESTATE, "stream_pool_wait: layer %d was not prefetched", layer);
    Slot& sl = p->slot[si];
    // the chunks are copied in order on one stream: the last of the covering chunks in copy
    // order has landed only once all of them have
    int c_lo = 0, c_hi = 0;
    while (c_lo + 1 < p->n_chunks && p->chunk_off[c_lo + 1] <= begin) ++c_lo;
    while (c_hi + 1 < p->n_chunks && p->chunk_off[c_hi + 1] < end) ++c_hi;
    cudaEvent_t done = sl.reverse ? sl.copy_done[c_lo] : sl.copy_done[c_hi];
    LSN_CUDA_TRY(cudaStreamWaitEvent(static_cast<cudaStream_t>(compute_stream), done, 0));
    if (timeout_ms > 0) {
        auto t0 = std::chrono::steady_clock::now();
        for (;;) {
            cudaError_t q = cudaEventQuery(done);
            if (q == cudaSuccess) break;
            if (q != cudaErrorNotReady) return cuda_fail(q, "stream_pool_wait: copy event");
            double el = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
            if (el > timeout_ms) {
                p->st.wait_ms += el;
                sl.state = kInUse;
                *dev_image = sl.dev;
                return fail(LSN_ETIMEOUT, "stream_pool_wait: layer %d copy not done after %d ms", layer, timeout_ms);
            }
            std::this_thread::sleep_for(std::chrono::microseconds(50));
        }
        p->st.wait_ms += std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
    }
    sl.state = kInUse;
    *dev_image = sl.dev;
    return LSN_OK;
}

int stream_pool_wait(lsn_pool* p, int layer, void* compute_stream, const void** dev_image, int timeout_ms) {
    if (!p) return fail(LSN_EINVAL, "stream_pool_wait: bad arguments");
    return stream_pool_wait_range(p, layer, 0, p->layer_bytes, compute_stream, dev_image, timeout_ms);
}

int stream_pool_chunk_stats(lsn_pool* p, int chunk, lsn_pool_stats* out) {
    if (!p || !out || chunk < 0 || chunk >= p->n_chunks) return fail(LSN_EINVAL, "stream_pool_chunk_stats: bad arguments");
    LSN_CUDA_TRY(cudaStreamSynchronize(p->copy));
    int rc = harvest(p, true);
    if (rc) return rc;
    *out = p->chunk_st[chunk];
    return LSN_OK;
}

int stream_pool_release(lsn_pool* p, int layer, void* compute_stream) {
    if (!p) return fail(LSN_EINVAL, "stream_pool_release: NULL pool");
    for (int i = 0; i < 2; ++i) {
        Slot& sl = p->slot[i];
        if (sl.layer == layer && sl.state == kInUse) {
            LSN_CUDA_TRY(cudaEventRecord(sl.slot_free, static_cast<cudaStream_t>(compute_stream)));
            sl.free_recorded = true;
            sl.state = kReleased;
            return LSN_OK;
        }
    }
    return fail(LSN_ESTATE, "stream_pool_release: layer %d is not in use", layer);
}

int stream_pool_stats(lsn_pool* p, lsn_pool_stats* out) {
    if (!p || !out) return fail(LSN_EINVAL, "stream_pool_stats: bad arguments");
    LSN_CUDA_TRY(cudaStreamSynchronize(p->copy));
    int rc = harvest(p, true);
    if (rc) return rc;
    *out = p->st;
    return LSN_OK;
}

int stream_pool_reset_stats(lsn_pool* p) {
    if (!p) return fail(LSN_EINVAL, "stream_pool_reset_stats: NULL pool");
    LSN_CUDA_TRY(cudaStreamSynchronize(p->copy));
    int rc = harvest(p, true);
    if (rc) return rc;
    memset(&p->st, 0, sizeof(p->st));
    memset(p->chunk_st, 0, sizeof(p->chunk_st));
    return LSN_OK;
}

int stream_pool_set_copy_delay_us(lsn_pool* p, int usec) {
    if (!p || usec < 0 || usec > 10000000) return fail(LSN_EINVAL, "stream_pool_set_copy_delay_us: bad arguments");
    p->delay_us = usec;
    return LSN_OK;
}

int stream_pool_destroy(lsn_pool* p) {
    if (!p) return LSN_OK;
    if (p->copy) cudaStreamSynchronize(p->copy);
    harvest(p, true);
    for (auto& t : p->pending) {
        cudaEventDestroy(t.start);
        cudaEventDestroy(t.end);
    }
    for (auto& t : p->spare) {
        cudaEventDestroy(t.start);
        cudaEventDestroy(t.end);
    }
    for (int i = 0; i < 2; ++i) {
        for (int c = 0; c < kMaxChunks; ++c)
            if (p->slot[i].copy_done[c]) cudaEventDestroy(p->slot[i].copy_done[c]);
        if (p->slot[i].slot_free) cudaEventDestroy(p->slot[i].slot_free);
    }
    delete p;
    return LSN_OK;
}

}  // extern "C"
