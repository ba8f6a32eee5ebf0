// slots.cpp -- adapter slot manager: a host cache of prepared adapters
// feeding the GPU slots of the adapter stores.
//
// vLLM offline multi-LoRA page, step 2: max_loras adapters sit in GPU slots
// at once, max_cpu_loras prepared adapters wait in host memory, and the slot
// rank bounds every adapter ("limits": a higher rank cannot load).  TGI
// multi-LoRA page, "3. weight preprocessing": an adapter is prepared once,
// scale folded into B and ranks zero-padded, before it serves.
//
// Policy: the host cache drops its least recently used adapter that is not
// resident in a slot; a batch's adapters that are not resident go to free
// slots first, then to the least recently used slots the batch does not
// need.  The host cache is pinned and mapped into the device's address
// space, and one gather kernel per batch (slot_copy.cu) moves every piece
// of every adapter the batch loads, on the caller's stream; an event after
// it guards those host buffers against being overwritten or freed while the
// copy is still in flight.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <limits>
#include <new>
#include <unordered_map>
#include <vector>

#include "lora.h"
#include "slot_copy.h"

struct lora_slot_manager {
    struct Entry {
        std::vector<lora_bf16_t*> A, B;   // prepared [r_slot][h_in] and [width][r_slot], host
        std::vector<const void*> dA, dB;  // the same buffers' device addresses (device mode)
        uint64_t used = 0;                // last batch (tick) that named it
        int slot = -1;                    // resident slot, or -1
        bool stale = false;               // replaced while resident: reload at the next acquire
        cudaEvent_t copied = nullptr;     // recorded after its last load (device mode)
    };

    int n_proj = 0, n_slots = 0, r_slot = 0, max_cpu = 0;
    std::vector<int> h_in, width;
    std::vector<lora_bf16_t*> A_st, B_st;   // device stores (empty: policy only)
    std::unordered_map<int64_t, Entry> cache;
    std::vector<int64_t> slot_owner;        // slot -> adapter id, or -1
    std::vector<uint64_t> slot_used;        // slot -> last batch tick
    uint64_t tick = 0;
    lora_slot_stats_t stats{};

    bool device() const { return !A_st.empty(); }

    size_t a_elems(int p) const { return static_cast<size_t>(r_slot) * h_in[p]; }
    size_t b_elems(int p) const { return static_cast<size_t>(width[p]) * r_slot; }

    // Waits until no copy reads the entry's host buffers any more.
    void quiesce(Entry& e)
    {
        if (e.copied) cudaEventSynchronize(e.copied);
    }

    void release(Entry& e)
    {
        quiesce(e);
        for (auto* v : {&e.A, &e.B})
            for (lora_bf16_t* b : *v) {
                if (device()) cudaFreeHost(b);
                else delete[] b;
            }
        e.A.clear();
        e.B.clear();
        e.dA.clear();
        e.dB.clear();
        if (e.copied) cudaEventDestroy(e.copied);
        e.copied = nullptr;
    }

    // Host buffers for one adapter; false (nothing kept) when an allocation fails.
    bool allocate(Entry& e)
    {
        for (int p = 0; p < n_proj; ++p) {
            for (int ab = 0; ab < 2; ++ab) {
                const size_t n = ab == 0 ? a_elems(p) : b_elems(p);
                lora_bf16_t* b = nullptr;
                void* db = nullptr;
                if (device()) {
                    if (cudaHostAlloc(reinterpret_cast<void**>(&b), n * sizeof(lora_bf16_t), cudaHostAllocMapped) !=
                        cudaSuccess)
                        b = nullptr;
                    else if (cudaHostGetDevicePointer(&db, b, 0) != cudaSuccess) {
                        cudaFreeHost(b);
                        b = nullptr;
                    }
                } else {
                    b = new (std::nothrow) lora_bf16_t[n];
                }
                if (!b) {
                    release(e);
                    return false;
                }
                (ab == 0 ? e.A : e.B).push_back(b);
                (ab == 0 ? e.dA : e.dB).push_back(db);
            }
        }
        if (device() && cudaEventCreateWithFlags(&e.copied, cudaEventDisableTiming) != cudaSuccess) {
            e.copied = nullptr;
            release(e);
            return false;
        }
        return true;
    }
};

extern "C" {

lora_status_t lora_slots_create(int n_proj, const int* h_in, const int* width, lora_bf16_t* const* A_stores,
                                lora_bf16_t* const* B_stores, int n_slots, int r_slot, int max_cpu,
                                lora_slot_manager_t** out)
{
    if (!out || !h_in || !width || n_proj < 1 || n_proj > 16 || n_slots < 1 || r_slot < 1 || max_cpu < n_slots)
        return LORA_ERR_INVALID_ARG;
    if ((A_stores == nullptr) != (B_stores == nullptr)) return LORA_ERR_INVALID_ARG;
    if (r_slot > LORA_MAX_RANK) return LORA_ERR_RANK_EXCEEDS_SLOT;
    if (r_slot % 8 != 0) return LORA_ERR_ALIGNMENT;
    for (int p = 0; p < n_proj; ++p) {
        if (h_in[p] <= 0 || width[p] <= 0) return LORA_ERR_INVALID_ARG;
        if (h_in[p] % 8 != 0) return LORA_ERR_ALIGNMENT;
        if (A_stores) {
            if (!A_stores[p] || !B_stores[p]) return LORA_ERR_INVALID_ARG;
            if ((reinterpret_cast<uintptr_t>(A_stores[p]) | reinterpret_cast<uintptr_t>(B_stores[p])) & 15u)
                return LORA_ERR_ALIGNMENT;
        }
    }
    auto* m = new (std::nothrow) lora_slot_manager;
    if (!m) return LORA_ERR_INVALID_ARG;
    m->n_proj = n_proj;
    m->n_slots = n_slots;
    m->r_slot = r_slot;
    m->max_cpu = max_cpu;
    m->h_in.assign(h_in, h_in + n_proj);
    m->width.assign(width, width + n_proj);
    if (A_stores) {
        m->A_st.assign(A_stores, A_stores + n_proj);
        m->B_st.assign(B_stores, B_stores + n_proj);
    }
    m->slot_owner.assign(n_slots, -1);
    m->slot_used.assign(n_slots, 0);
    *out = m;
    return LORA_OK;
}

void lora_slots_destroy(lora_slot_manager_t* m)
{
    if (!m) return;
    for (auto& kv : m->cache) m->release(kv.second);
    delete m;
}

lora_status_t lora_slots_register(lora_slot_manager_t* m, int64_t adapter_id, const lora_bf16_t* const* A,
                                  const lora_bf16_t* const* B, int r, double alpha, int use_rslora)
{
    if (!m || !A || !B || adapter_id < 0 || r < 1) return LORA_ERR_INVALID_ARG;
    if (r > m->r_slot) return LORA_ERR_RANK_EXCEEDS_SLOT;
    for (int p = 0; p < m->n_proj; ++p)
        if (!A[p] || !B[p]) return LORA_ERR_INVALID_ARG;

    auto it = m->cache.find(adapter_id);
    lora_slot_manager::Entry fresh;
    lora_slot_manager::Entry* e = nullptr;
    if (it != m->cache.end()) {
        e = &it->second;
        m->quiesce(*e);   // a load from these buffers may still be in flight
    } else {
        // the victim, if the cache is full: least recently used, not resident
        int64_t victim = -1;
        if (static_cast<int>(m->cache.size()) >= m->max_cpu) {
            uint64_t oldest = std::numeric_limits<uint64_t>::max();
            for (auto& kv : m->cache)
                if (kv.second.slot < 0 && kv.second.used < oldest) {
                    oldest = kv.second.used;
                    victim = kv.first;
                }
            if (victim < 0) return LORA_ERR_SLOT_RANGE;
        }
        if (!m->allocate(fresh)) return LORA_ERR_CUDA;
        if (victim >= 0) {
            m->release(m->cache[victim]);
            m->cache.erase(victim);
            ++m->stats.host_evictions;
        }
        e = &m->cache.emplace(adapter_id, std::move(fresh)).first->second;
    }
    for (int p = 0; p < m->n_proj; ++p) {
        const lora_status_t st = lora_prepare_adapter(A[p], B[p], r, m->h_in[p], m->width[p], alpha, use_rslora,
                                                      m->r_slot, e->A[p], e->B[p]);
        if (st != LORA_OK) return st;   // unreachable after the checks above
    }
    e->used = ++m->tick;
    if (e->slot >= 0) e->stale = true;
    ++m->stats.registered;
    return LORA_OK;
}

lora_status_t lora_slots_acquire(lora_slot_manager_t* m, const int64_t* adapter_ids, int n, int32_t* slots_out,
                                 lora_stream_t stream)
{
    if (!m || n < 0 || (n > 0 && (!adapter_ids || !slots_out))) return LORA_ERR_INVALID_ARG;
    // distinct adapters of the batch, in order of first appearance
    std::vector<int64_t> distinct;
    for (int i = 0; i < n; ++i) {
        const int64_t id = adapter_ids[i];
        if (id == -1) continue;
        if (id < -1 || m->cache.find(id) == m->cache.end()) return LORA_ERR_INVALID_ARG;
        bool seen = false;
        for (int64_t d : distinct) seen |= d == id;
        if (!seen) distinct.push_back(id);
    }
    if (static_cast<int>(distinct.size()) > m->n_slots) return LORA_ERR_SLOT_RANGE;

    const uint64_t tick = ++m->tick;
    std::vector<int64_t> need;   // adapters to load
    for (int64_t id : distinct) {
        auto& e = m->cache[id];
        e.used = tick;
        if (e.slot >= 0) m->slot_used[e.slot] = tick;   // keep it: the batch needs it
        if (e.slot >= 0 && !e.stale) ++m->stats.hits;
        else need.push_back(id);
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (int64_t id : need) {
        auto& e = m->cache[id];
        int slot = e.slot;   // a stale resident copy reloads in place
        if (slot < 0) {
            // a free slot, else the least recently used one the batch does not need
            uint64_t best = std::numeric_limits<uint64_t>::max();
            for (int k = 0; k < m->n_slots; ++k) {
                if (m->slot_used[k] == tick) continue;
                const uint64_t key = m->slot_owner[k] < 0 ? 0 : m->slot_used[k] + 1;
                if (key < best) {
                    best = key;
                    slot = k;
                }
            }
            if (slot < 0) return LORA_ERR_SLOT_RANGE;   // unreachable: distinct <= n_slots
            const int64_t old = m->slot_owner[slot];
            if (old >= 0) {
                m->cache[old].slot = -1;
                ++m->stats.slot_evictions;
            }
            m->slot_owner[slot] = id;
            m->slot_used[slot] = tick;
            e.slot = slot;
        }
    }
    if (m->device() && !need.empty()) {
        // every piece of every adapter to load, gathered by one kernel per
        // kMaxCopySegs pieces; then one event per adapter
        std::vector<lora::CopySeg> segs;
        segs.reserve(need.size() * 2 * m->n_proj);
        for (int64_t id : need) {
            const auto& e = m->cache[id];
            for (int p = 0; p < m->n_proj; ++p) {
                segs.push_back({e.dA[p], m->A_st[p] + static_cast<size_t>(e.slot) * m->a_elems(p),
                                m->a_elems(p) * sizeof(lora_bf16_t)});
                segs.push_back({e.dB[p], m->B_st[p] + static_cast<size_t>(e.slot) * m->b_elems(p),
                                m->b_elems(p) * sizeof(lora_bf16_t)});
            }
        }
        cudaError_t ce = cudaSuccess;
        for (size_t i = 0; ce == cudaSuccess && i < segs.size(); i += lora::kMaxCopySegs)
            ce = lora::launch_slot_copy(segs.data() + i,
                                        static_cast<int>(std::min<size_t>(lora::kMaxCopySegs, segs.size() - i)), s);
        for (int64_t id : need)
            if (ce == cudaSuccess) ce = cudaEventRecord(m->cache[id].copied, s);
        if (ce != cudaSuccess) {   // leave the slots empty rather than half loaded
            for (int64_t id : need) {
                auto& e = m->cache[id];
                if (e.slot >= 0) m->slot_owner[e.slot] = -1;
                e.slot = -1;
            }
            return LORA_ERR_CUDA;
        }
    }
    for (int64_t id : need) {
        m->cache[id].stale = false;
        ++m->stats.loads;
    }
    for (int i = 0; i < n; ++i)
        slots_out[i] = adapter_ids[i] == -1 ? -1 : m->cache[adapter_ids[i]].slot;
    return LORA_OK;
}

int lora_slots_slot_of(const lora_slot_manager_t* m, int64_t adapter_id)
{
    if (!m) return -1;
    auto it = m->cache.find(adapter_id);
    return it == m->cache.end() ? -1 : it->second.slot;
}

lora_status_t lora_slots_stats(const lora_slot_manager_t* m, lora_slot_stats_t* out)
{
    if (!m || !out) return LORA_ERR_INVALID_ARG;
    *out = m->stats;
    return LORA_OK;
}

}  // extern "C"
