// cache.cpp -- host-resident experts with an HBM cache and prefetch (host code).
//
// A layer's experts live in page-locked host memory; a cache of `slots`
// expert-sized slots in HBM holds the ones in use.  The pages stream experts
// that do not fit on the GPU from host memory or disk and hide the copies
// behind compute ("在 8 GB 显卡上运行 510 GB 的 DeepSeek-V4.1-Flash",
// §提速之路：v1 到 v4; "把不支持 FP4 的 A100 拉到 673 tok/s", §但 CPU 也没那么快);
// on GB300 the host memory sits behind NVLink-C2C and the copy engines move it.
//
//   fetch(ids)     makes the experts of `ids` resident: a miss takes the least
//                  recently used slot that the request does not use, and its
//                  blob is copied there; the copies of a request go round-robin
//                  over kCopyStreams copy streams (several in flight), and a
//                  copy into a slot waits for the slot's previous fill, so a
//                  slot's fills stay in order; the caller's stream waits for the copies and
//                  then receives the layer's expert table (a device array of
//                  E pointers, NULL for experts not resident), written in
//                  stream order from a ring of page-locked staging buffers.
//   prefetch(ids)  the same copies without the wait and without a table: the
//                  experts a predictor expects next become resident while the
//                  current layer runs.
//
// A slot is never overwritten while work that may read it is pending: every
// call records an event on the caller's stream first, and that event
// "releases" the slots of the previous request; a copy into a victim slot
// waits for the victim's release event.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <vector>

#include "../../include/moe_ffn.h"
#include "internal.h"

namespace {
constexpr int kCopyStreams = 4;
}

struct moe_expert_cache_s {
    int device = 0;
    int E = 0, slots = 0;
    size_t blob = 0, stride = 0;
    std::vector<const uint8_t*> host;          // host blob of each expert
    uint8_t* dev = nullptr;                    // slots x stride bytes
    std::vector<int> slot_of;                  // expert -> slot or -1
    std::vector<int> expert_in;                // slot -> expert or -1
    std::vector<long long> last_use;           // slot -> request stamp
    std::vector<cudaEvent_t> released;         // slot -> free once this event completes
    std::vector<cudaEvent_t> filled;           // slot -> its last fill is done once this completes
    std::vector<char> ever_used;
    std::vector<int> prev_slots;               // slots of the previous request
    long long clock = 0;
    cudaStream_t copy[kCopyStreams] = {};
    cudaEvent_t copied[kCopyStreams] = {};
    int next_copy = 0;
    // the layer tables: one device array of E pointers, rewritten in stream
    // order; its host staging buffers form a ring guarded by events
    const uint8_t** dtable = nullptr;
    static constexpr int kRing = 8;
    const uint8_t** stage[kRing] = {};
    cudaEvent_t stage_ev[kRing] = {};
    int ring = 0;
    long long hits = 0, misses = 0, bytes = 0;     // hits and misses of fetches; bytes of all copies
};

namespace {

struct Guard {
    int prev = -1;
    explicit Guard(int dev)
    {
        cudaGetDevice(&prev);
        if (prev != dev) cudaSetDevice(dev);
    }
    ~Guard()
    {
        int cur = -1;
        cudaGetDevice(&cur);
        if (prev >= 0 && cur != prev) cudaSetDevice(prev);
    }
};

void destroy_cache(moe_expert_cache_s* c)
{
    if (!c) return;
    Guard g(c->device);
    for (cudaEvent_t e : c->released)
        if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : c->filled)
        if (e) cudaEventDestroy(e);
    for (int i = 0; i < kCopyStreams; i++) {
        if (c->copy[i]) cudaStreamDestroy(c->copy[i]);
        if (c->copied[i]) cudaEventDestroy(c->copied[i]);
    }
    for (int i = 0; i < moe_expert_cache_s::kRing; i++) {
        if (c->stage[i]) cudaFreeHost(c->stage[i]);
        if (c->stage_ev[i]) cudaEventDestroy(c->stage_ev[i]);
    }
    if (c->dtable) cudaFree(c->dtable);
    if (c->dev) cudaFree(c->dev);
    delete c;
}

// Records the caller's position: the slots of the previous request may be
// read by work enqueued up to here, so they are free once this event is.
cudaError_t mark_call(moe_expert_cache_s* c, cudaStream_t s)
{
    cudaError_t e = cudaSuccess;
    for (int slot : c->prev_slots)
        if (e == cudaSuccess) e = cudaEventRecord(c->released[slot], s);
    c->prev_slots.clear();
    return e;
}

bool valid_ids(const moe_expert_cache_s* c, const int32_t* ids, int n)
{
    if (n < 0 || (n > 0 && !ids)) return false;
    for (int i = 0; i < n; i++)
        if (ids[i] < -1 || ids[i] >= c->E) return false;
    return true;
}

// Makes ids resident (copies issued, not waited for).  Slots of the request
// are never victims of each other.  `count`: a fetch (hits and misses counted).
int make_resident(moe_expert_cache_s* c, const int32_t* ids, int n, bool count, std::vector<int>* req_slots)
{
    c->clock++;
    std::vector<char> in_req((size_t)c->slots, 0);
    // hits first, so that no miss evicts an expert of the same request
    for (int i = 0; i < n; i++) {
        const int e = ids[i];
        if (e < 0) continue;
        const int s = c->slot_of[e];
        if (s >= 0) in_req[s] = 1;
    }
    for (int i = 0; i < n; i++) {
        const int e = ids[i];
        if (e < 0) continue;
        int s = c->slot_of[e];
        if (s >= 0) {
            if (c->last_use[s] != c->clock) {
                if (count) c->hits++;
                c->last_use[s] = c->clock;
                if (req_slots) req_slots->push_back(s);
            }
            continue;
        }
        // miss: the least recently used slot outside the request (lowest number on ties)
        int victim = -1;
        for (int t = 0; t < c->slots; t++) {
            if (in_req[t]) continue;
            if (victim < 0 || c->last_use[t] < c->last_use[victim]) victim = t;
        }
        if (victim < 0) return MOE_ERR_INVALID_ARG;        // more distinct experts than slots
        const int old = c->expert_in[victim];
        if (old >= 0) c->slot_of[old] = -1;
        c->expert_in[victim] = e;
        c->slot_of[e] = victim;
        c->last_use[victim] = c->clock;
        in_req[victim] = 1;
        if (count) c->misses++;
        c->bytes += (long long)c->blob;
        cudaStream_t cs = c->copy[c->next_copy];
        c->next_copy = (c->next_copy + 1) % kCopyStreams;
        cudaError_t err = cudaSuccess;
        if (c->ever_used[victim]) {
            // after the work that may read the slot, and after its previous fill
            err = cudaStreamWaitEvent(cs, c->released[victim], 0);
            if (err == cudaSuccess) err = cudaStreamWaitEvent(cs, c->filled[victim], 0);
        }
        c->ever_used[victim] = 1;
        if (err == cudaSuccess)
            err = cudaMemcpyAsync(c->dev + (size_t)victim * c->stride, c->host[e], c->blob, cudaMemcpyHostToDevice,
                                  cs);
        if (err == cudaSuccess) err = cudaEventRecord(c->filled[victim], cs);
        if (err != cudaSuccess) return MOE_ERR_CUDA;
        if (req_slots) req_slots->push_back(victim);
    }
    return MOE_OK;
}

}  // namespace

extern "C" int moe_expert_cache_create(const moe_ffn_config* cfg, int device, const void* const* host_blobs, int slots,
                                       moe_expert_cache_t* out)
{
    if (!cfg || !host_blobs || !out || slots <= 0 || cfg->num_experts <= 0) return MOE_ERR_INVALID_ARG;
    const size_t blob = moe_ffn_packed_expert_bytes(cfg);
    if (blob == 0) return MOE_ERR_INVALID_ARG;
    for (int e = 0; e < cfg->num_experts; e++)
        if (!host_blobs[e] || ((uintptr_t)host_blobs[e] & 15)) return MOE_ERR_INVALID_ARG;
    Guard g(device);
    moe_expert_cache_s* c = new moe_expert_cache_s();
    c->device = device;
    c->E = cfg->num_experts;
    c->slots = slots;
    c->blob = blob;
    c->stride = (blob + 255) / 256 * 256;
    c->host.assign((const uint8_t* const*)host_blobs, (const uint8_t* const*)host_blobs + c->E);
    c->slot_of.assign((size_t)c->E, -1);
    c->expert_in.assign((size_t)slots, -1);
    c->last_use.assign((size_t)slots, 0);
    c->released.assign((size_t)slots, nullptr);
    c->filled.assign((size_t)slots, nullptr);
    c->ever_used.assign((size_t)slots, 0);
    bool ok = moe::lib_malloc((void**)&c->dev, c->stride * (size_t)slots) == cudaSuccess;
    ok = ok && moe::lib_malloc((void**)&c->dtable, sizeof(void*) * (size_t)c->E) == cudaSuccess;
    for (int i = 0; ok && i < kCopyStreams; i++) {
        ok = cudaStreamCreateWithFlags(&c->copy[i], cudaStreamNonBlocking) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&c->copied[i], cudaEventDisableTiming) == cudaSuccess;
    }
    for (int s = 0; ok && s < slots; s++) {
        ok = cudaEventCreateWithFlags(&c->released[s], cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&c->filled[s], cudaEventDisableTiming) == cudaSuccess;
    }
    for (int i = 0; ok && i < moe_expert_cache_s::kRing; i++) {
        ok = moe::lib_host_alloc((void**)&c->stage[i], sizeof(void*) * (size_t)c->E, cudaHostAllocDefault) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&c->stage_ev[i], cudaEventDisableTiming) == cudaSuccess;
        if (ok) ok = cudaEventRecord(c->stage_ev[i], 0) == cudaSuccess;
    }
    if (!ok) {
        cudaGetLastError();
        destroy_cache(c);
        return MOE_ERR_OOM;
    }
    *out = c;
    return MOE_OK;
}

extern "C" int moe_expert_cache_fetch(moe_expert_cache_t c, const int32_t* ids, int n, void* stream,
                                      moe_expert_table* tbl)
{
    if (!c || !tbl || !valid_ids(c, ids, n)) return MOE_ERR_INVALID_ARG;
    Guard g(c->device);
    cudaStream_t s = (cudaStream_t)stream;
    if (mark_call(c, s) != cudaSuccess) return MOE_ERR_CUDA;
    std::vector<int> req;
    int rc = make_resident(c, ids, n, true, &req);
    if (rc != MOE_OK) return rc;
    // the caller's stream waits for this request's copies (and earlier ones on
    // the same copy streams, which may be prefetches of these experts)
    for (int q = 0; q < kCopyStreams; q++) {
        if (cudaEventRecord(c->copied[q], c->copy[q]) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaStreamWaitEvent(s, c->copied[q], 0) != cudaSuccess) return MOE_ERR_CUDA;
    }
    // the table, staged in the next ring buffer once its previous copy is done
    const int r = c->ring;
    c->ring = (c->ring + 1) % moe_expert_cache_s::kRing;
    if (cudaEventSynchronize(c->stage_ev[r]) != cudaSuccess) return MOE_ERR_CUDA;
    for (int e = 0; e < c->E; e++)
        c->stage[r][e] = c->slot_of[e] >= 0 ? c->dev + (size_t)c->slot_of[e] * c->stride : nullptr;
    if (cudaMemcpyAsync(c->dtable, c->stage[r], sizeof(void*) * (size_t)c->E, cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaEventRecord(c->stage_ev[r], s) != cudaSuccess)
        return MOE_ERR_CUDA;
    c->prev_slots = req;
    tbl->experts = c->dtable;
    return MOE_OK;
}

extern "C" int moe_expert_cache_prefetch(moe_expert_cache_t c, const int32_t* ids, int n, void* stream)
{
    if (!c || !valid_ids(c, ids, n)) return MOE_ERR_INVALID_ARG;
    Guard g(c->device);
    cudaStream_t s = (cudaStream_t)stream;
    // the previous request's slots stay protected until the caller's work so far is done
    std::vector<int> keep = c->prev_slots;
    if (mark_call(c, s) != cudaSuccess) return MOE_ERR_CUDA;
    c->prev_slots = keep;
    return make_resident(c, ids, n, false, nullptr);
}

extern "C" int moe_expert_cache_slot(moe_expert_cache_t c, int expert)
{
    if (!c || expert < 0 || expert >= c->E) return -1;
    return c->slot_of[expert];
}

extern "C" int moe_expert_cache_stats(moe_expert_cache_t c, long long* hits, long long* misses, long long* bytes)
{
    if (!c) return MOE_ERR_INVALID_ARG;
    if (hits) *hits = c->hits;
    if (misses) *misses = c->misses;
    if (bytes) *bytes = c->bytes;
    return MOE_OK;
}

extern "C" void moe_expert_cache_destroy(moe_expert_cache_t c)
{
    if (!c) return;
    {
        Guard g(c->device);
        for (int q = 0; q < kCopyStreams; q++)
            if (c->copy[q]) cudaStreamSynchronize(c->copy[q]);
    }
    destroy_cache(c);
}
