// stream.cu — routed experts streamed from host memory through an HBM expert
// cache.  chenxutan ds4 article §3.3 (routed experts are not all loaded onto
// the GPU but brought in as the router selects them), §3.5 (SSD streaming:
// when the model does not fit in memory the engine keeps running and pages
// weights in on demand) and
// the yudady DS-4 DwarfStar page, section "SSD Streaming" (the non-routed
// weights stay resident; a routed expert that misses the cache is loaded,
// used, and its space is later released).
//
// B300 form of that idea: the routed experts of any number of layers live in
// host memory (pinned, so copies are asynchronous DMA); a pool in HBM holds
// n_slots experts (gate + up + down each) and is managed least-recently-used
// first, keyed by (layer, expert).  A streamed forward reads the layer's
// expert ids back, copies only the experts that are not resident, points the
// layer's expert tables at the slots and runs the ordinary forward kernels,
// so its output is bit-identical to the resident path.
#include "ds4g_internal.cuh"

#include <list>
#include <new>
#include <unordered_map>
#include <vector>

namespace ds4g {

// Least-recently-used slot assignment, free of CUDA so that the policy can be
// checked on the host.  One call = one forward: its keys are assigned first
// (a key already resident is a hit and becomes most recent); misses then take
// free slots, else evict the least recent slot not used by the same call.
class ExpertLru {
  public:
    explicit ExpertLru(int n) : key_(n, -1), stamp_(n, 0), pos_(n) {
        for (int i = 0; i < n; ++i) pos_[i] = order_.insert(order_.end(), i);
    }
    int size() const { return (int)key_.size(); }

    // Assigns slots to the distinct keys of one call (keys < 0 are skipped,
    // slot -1).  slot[i] is key i's slot, miss[i] = 1 if it must be copied in
    // (only for the first occurrence of a key).  DS4G_ENOSPACE if the call
    // has more distinct keys than slots; the slots it had given to missing
    // keys are then emptied (nothing was copied into them).
    ds4g_status assign(const int64_t *keys, int n, int32_t *slot, uint8_t *miss) {
        ++call_;
        for (int i = 0; i < n; ++i) {
            slot[i] = -1;
            miss[i] = 0;
            const int64_t k = keys[i];
            if (k < 0) continue;
            auto it = where_.find(k);
            int s;
            if (it != where_.end()) {
                s = it->second;
            } else {
                s = order_.back();                      // least recently used
                if (stamp_[s] == call_) {   // every slot serves this call
                    for (int j = 0; j < i; ++j)
                        if (miss[j]) forget(slot[j]);
                    return DS4G_ENOSPACE;
                }
                if (key_[s] >= 0) where_.erase(key_[s]);
                key_[s] = k;
                where_[k] = s;
                miss[i] = 1;
            }
            if (stamp_[s] != call_) {
                stamp_[s] = call_;
                order_.splice(order_.begin(), order_, pos_[s]);   // most recent at the front
            }
            slot[i] = s;
        }
        return DS4G_OK;
    }

    // A slot whose copy could not be issued holds nothing valid.
    void forget(int s) {
        if (key_[s] >= 0) where_.erase(key_[s]);
        key_[s] = -1;
        stamp_[s] = 0;
        order_.splice(order_.end(), order_, pos_[s]);
    }

  private:
    std::vector<int64_t> key_;      // key held by each slot, -1 = empty
    std::vector<uint64_t> stamp_;   // last call that used the slot
    std::list<int> order_;          // slots, most recently used first
    std::vector<std::list<int>::iterator> pos_;
    std::unordered_map<int64_t, int> where_;
    uint64_t call_ = 0;
};

static bool stream_types_ok(int gut, int dt) {
    return (gut == DS4G_IQ2_XXS && dt == DS4G_Q2_K) || (gut == DS4G_Q4_K && dt == DS4G_Q4_K);
}

struct SlotGeometry {
    size_t gate, down, slot, table, total;   // bytes; table = offset of the pointer table
};
static SlotGeometry slot_geometry(int gut, int dt, int n_slots) {
    SlotGeometry g;
    g.gate = ds4g_packed_size((ds4g_qtype)gut, kF, kH);
    g.down = ds4g_packed_size((ds4g_qtype)dt, kH, kF);
    g.slot = align_up(2 * g.gate + g.down, 256);
    g.table = (size_t)n_slots * g.slot;
    g.total = g.table + align_up(3 * kE * sizeof(void *), 256);
    return g;
}

}  // namespace ds4g

using namespace ds4g;

struct ds4g_expert_cache {
    int gut, dt, n_slots, max_tokens;
    SlotGeometry geo;
    uint8_t *pool;           // dev: slots, then the pointer table [3][256]
    const void **table_h;    // pinned host copy of the pointer table
    int32_t *ids_h;          // pinned host copy of one call's ids [max_tokens][6]
    ExpertLru lru;
    std::vector<int64_t> keys;
    std::vector<int32_t> slot;
    std::vector<uint8_t> miss;
    uint64_t hits = 0, misses = 0, bytes = 0;
    explicit ds4g_expert_cache(int n) : lru(n) {}
};

extern "C" size_t ds4g_expert_cache_pool_bytes(ds4g_qtype gate_up_type, ds4g_qtype down_type, int n_slots) {
    if (!stream_types_ok(gate_up_type, down_type) || n_slots < 1) return 0;
    return slot_geometry(gate_up_type, down_type, n_slots).total;
}

extern "C" ds4g_status ds4g_expert_cache_create(ds4g_qtype gate_up_type, ds4g_qtype down_type, int n_slots,
                                                int max_tokens, void *pool, size_t pool_bytes,
                                                ds4g_expert_cache **cache) {
    if (!cache || !pool || n_slots < kK || max_tokens < 1 || max_tokens > (1 << 20)) return DS4G_EINVAL;
    *cache = nullptr;
    if (!stream_types_ok(gate_up_type, down_type)) return DS4G_EUNSUPPORTED;
    if ((uintptr_t)pool & 15) return DS4G_EALIGN;
    const SlotGeometry geo = slot_geometry(gate_up_type, down_type, n_slots);
    if (pool_bytes < geo.total) return DS4G_ENOSPACE;
    ds4g_expert_cache *c = new (std::nothrow) ds4g_expert_cache(n_slots);
    if (!c) return DS4G_ENOSPACE;
    c->gut = gate_up_type;
    c->dt = down_type;
    c->n_slots = n_slots;
    c->max_tokens = max_tokens;
    c->geo = geo;
    c->pool = (uint8_t *)pool;
    c->table_h = nullptr;
    c->ids_h = nullptr;
    if (cudaHostAlloc((void **)&c->table_h, 3 * kE * sizeof(void *), cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc((void **)&c->ids_h, (size_t)max_tokens * kK * sizeof(int32_t), cudaHostAllocDefault) !=
            cudaSuccess) {
        if (c->table_h) cudaFreeHost((void *)c->table_h);
        delete c;
        return DS4G_ECUDA;
    }
    c->keys.resize((size_t)max_tokens * kK);
    c->slot.resize((size_t)max_tokens * kK);
    c->miss.resize((size_t)max_tokens * kK);
    *cache = c;
    return DS4G_OK;
}

extern "C" ds4g_status ds4g_expert_cache_destroy(ds4g_expert_cache *cache) {
    if (!cache) return DS4G_EINVAL;
    const bool ok = cudaFreeHost((void *)cache->table_h) == cudaSuccess;
    const bool ok2 = cudaFreeHost(cache->ids_h) == cudaSuccess;
    delete cache;
    return ok && ok2 ? DS4G_OK : DS4G_ECUDA;
}

extern "C" ds4g_status ds4g_expert_cache_stats(const ds4g_expert_cache *cache, uint64_t *hits, uint64_t *misses,
                                               uint64_t *bytes_copied) {
    if (!cache || !hits || !misses || !bytes_copied) return DS4G_EINVAL;
    *hits = cache->hits;
    *misses = cache->misses;
    *bytes_copied = cache->bytes;
    return DS4G_OK;
}

extern "C" ds4g_status ds4g_expert_lru_simulate(int n_slots, int n_calls, const int32_t *call_sizes,
                                                const int64_t *keys, int32_t *slot_out, uint8_t *miss_out) {
    if (n_slots < 1 || n_calls < 0 || (n_calls && (!call_sizes || !keys || !slot_out || !miss_out)))
        return DS4G_EINVAL;
    ExpertLru lru(n_slots);
    size_t off = 0;
    for (int c = 0; c < n_calls; ++c) {
        if (call_sizes[c] < 0) return DS4G_EINVAL;
        const ds4g_status st = lru.assign(keys + off, call_sizes[c], slot_out + off, miss_out + off);
        if (st == DS4G_ENOSPACE) {
            for (int i = 0; i < call_sizes[c]; ++i) {   // the call is refused; the next one proceeds
                slot_out[off + i] = -2;
                miss_out[off + i] = 0;
            }
        } else if (st != DS4G_OK) {
            return st;
        }
        off += (size_t)call_sizes[c];
    }
    return DS4G_OK;
}

extern "C" ds4g_status ds4g_moe_forward_streamed(const float *hidden, int T, int layer_key,
                                                 const ds4g_host_experts *src, const uint16_t *sh_gate,
                                                 const uint16_t *sh_up, const uint16_t *sh_down,
                                                 const uint64_t *iq2_grid, const int32_t *ids, const float *w,
                                                 float *out, ds4g_expert_cache *c, void *workspace,
                                                 size_t ws_bytes, ds4g_stream_t s) {
    DS4G_TRACE();
    if (!c || !src || !src->gate || !src->up || !src->down || !ids || layer_key < 0) return DS4G_EINVAL;
    if (T < 1 || T > c->max_tokens) return DS4G_EINVAL;
    if (src->gate_up_type != c->gut || src->down_type != c->dt) return DS4G_EUNSUPPORTED;
    if ((uintptr_t)ids & 15) return DS4G_EALIGN;
    if (ws_bytes < ds4g_forward_workspace(T)) return DS4G_ENOSPACE;
    cudaStream_t st = (cudaStream_t)s;
    const int n = T * kK;
    // the ids decide what to copy: read them back; the synchronisation also
    // retires every earlier call's kernels on s, so any slot may be rewritten
    if (cudaMemcpyAsync(c->ids_h, ids, (size_t)n * sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return DS4G_ECUDA;
    for (int i = 0; i < n; ++i) {
        const int e = c->ids_h[i];
        c->keys[i] = (e >= 0 && e < kE) ? (int64_t)layer_key * kE + e : -1;   // bad ids: the kernels flag them
        if (c->keys[i] >= 0 && (!src->gate[e] || !src->up[e] || !src->down[e])) return DS4G_EINVAL;
    }
    ds4g_status rc = c->lru.assign(c->keys.data(), n, c->slot.data(), c->miss.data());
    if (rc != DS4G_OK) return rc;
    for (int i = 0; i < 3 * kE; ++i) c->table_h[i] = nullptr;
    const SlotGeometry &g = c->geo;
    for (int i = 0; i < n; ++i) {
        if (c->slot[i] < 0) continue;
        const int e = c->ids_h[i];
        uint8_t *dst = c->pool + (size_t)c->slot[i] * g.slot;
        if (c->miss[i]) {
            if (cudaMemcpyAsync(dst, src->gate[e], g.gate, cudaMemcpyHostToDevice, st) != cudaSuccess ||
                cudaMemcpyAsync(dst + g.gate, src->up[e], g.gate, cudaMemcpyHostToDevice, st) != cudaSuccess ||
                cudaMemcpyAsync(dst + 2 * g.gate, src->down[e], g.down, cudaMemcpyHostToDevice, st) !=
                    cudaSuccess) {
                for (int j = i; j < n; ++j)   // nothing valid was copied into these
                    if (c->miss[j]) c->lru.forget(c->slot[j]);
                return DS4G_ECUDA;
            }
            ++c->misses;
            c->bytes += 2 * g.gate + g.down;
        } else if (!c->table_h[e]) {
            ++c->hits;   // resident, first occurrence in this call
        }
        c->table_h[e] = dst;
        c->table_h[kE + e] = dst + g.gate;
        c->table_h[2 * kE + e] = dst + 2 * g.gate;
    }
    const void **table_d = (const void **)(c->pool + g.table);
    if (cudaMemcpyAsync(table_d, c->table_h, 3 * kE * sizeof(void *), cudaMemcpyHostToDevice, st) != cudaSuccess)
        return DS4G_ECUDA;
    ds4g_layer L;
    L.gate_up_type = (ds4g_qtype)c->gut;
    L.down_type = (ds4g_qtype)c->dt;
    L.gate = table_d;
    L.up = table_d + kE;
    L.down = table_d + 2 * kE;
    L.sh_gate = sh_gate;
    L.sh_up = sh_up;
    L.sh_down = sh_down;
    L.iq2_grid = iq2_grid;
    return ds4g_moe_forward(hidden, T, &L, ids, w, out, workspace, ws_bytes, s);
}
