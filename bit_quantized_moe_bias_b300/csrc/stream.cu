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

#include <errno.h>
#include <fcntl.h>
#include <stdio.h>
#include <string.h>
#include <unistd.h>

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
    size_t gate, down, slot, table, ready, total;   // bytes; table, ready: offsets of the pointer table, flags
};
constexpr int kReadyFlags = 64;   // per-slot ready flags of one overlapped call (6T <= 18)
static SlotGeometry slot_geometry(int gut, int dt, int n_slots) {
    SlotGeometry g;
    g.gate = ds4g_packed_size((ds4g_qtype)gut, kF, kH);
    g.down = ds4g_packed_size((ds4g_qtype)dt, kH, kF);
    g.slot = align_up(2 * g.gate + g.down, 256);
    g.table = (size_t)n_slots * g.slot;
    g.ready = g.table + align_up(3 * kE * sizeof(void *), 256);
    g.total = g.ready + align_up(kReadyFlags * sizeof(uint32_t), 256);
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
    uint32_t *flag_h;        // pinned: one call's initial ready flags [kReadyFlags], then the epoch word
    cudaStream_t cs;         // copy stream of the overlapped calls
    cudaEvent_t copied;      // the copies of the last overlapped call are done
    uint32_t epoch = 0;
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
    c->flag_h = nullptr;
    c->cs = nullptr;
    c->copied = nullptr;
    if (cudaHostAlloc((void **)&c->table_h, 3 * kE * sizeof(void *), cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc((void **)&c->ids_h, (size_t)max_tokens * kK * sizeof(int32_t), cudaHostAllocDefault) !=
            cudaSuccess ||
        cudaHostAlloc((void **)&c->flag_h, (kReadyFlags + 1) * sizeof(uint32_t), cudaHostAllocDefault) !=
            cudaSuccess ||
        cudaStreamCreateWithFlags(&c->cs, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->copied, cudaEventDisableTiming) != cudaSuccess) {
        if (c->table_h) cudaFreeHost((void *)c->table_h);
        if (c->ids_h) cudaFreeHost(c->ids_h);
        if (c->flag_h) cudaFreeHost(c->flag_h);
        if (c->cs) cudaStreamDestroy(c->cs);
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
    bool ok = cudaStreamSynchronize(cache->cs) == cudaSuccess;
    ok = (cudaEventDestroy(cache->copied) == cudaSuccess) && ok;
    ok = (cudaStreamDestroy(cache->cs) == cudaSuccess) && ok;
    ok = (cudaFreeHost((void *)cache->table_h) == cudaSuccess) && ok;
    ok = (cudaFreeHost(cache->ids_h) == cudaSuccess) && ok;
    ok = (cudaFreeHost(cache->flag_h) == cudaSuccess) && ok;
    delete cache;
    return ok ? DS4G_OK : DS4G_ECUDA;
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

// Where a streamed forward finds the routed experts that miss the cache.
struct ExpertSource {
    virtual ~ExpertSource() {}
    virtual bool has(int e) const = 0;
    // Copies expert e (gate, up, down) into the slot at dst on st.
    virtual ds4g_status copy(int e, uint8_t *dst, const SlotGeometry &g, cudaStream_t st) = 0;
};

// Experts in (pinned) host memory: three asynchronous copies each.
struct HostSource : ExpertSource {
    const ds4g_host_experts *src;
    explicit HostSource(const ds4g_host_experts *s) : src(s) {}
    bool has(int e) const override { return src->gate[e] && src->up[e] && src->down[e]; }
    ds4g_status copy(int e, uint8_t *dst, const SlotGeometry &g, cudaStream_t st) override {
        if (cudaMemcpyAsync(dst, src->gate[e], g.gate, cudaMemcpyHostToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(dst + g.gate, src->up[e], g.gate, cudaMemcpyHostToDevice, st) != cudaSuccess ||
            cudaMemcpyAsync(dst + 2 * g.gate, src->down[e], g.down, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return DS4G_ECUDA;
        return DS4G_OK;
    }
};

// The streamed forward, for any source: read the ids back, give each distinct
// selected expert its slot, copy the missing ones, point the layer's tables
// at the slots, run the ordinary forward.
static ds4g_status streamed_forward(const float *hidden, int T, int layer_key, int gut, int dt, ExpertSource &src,
                                    const uint16_t *sh_gate, const uint16_t *sh_up, const uint16_t *sh_down,
                                    const uint64_t *iq2_grid, const int32_t *ids, const float *w, float *out,
                                    ds4g_expert_cache *c, void *workspace, size_t ws_bytes, ds4g_stream_t s) {
    if (!c || !ids || layer_key < 0) return DS4G_EINVAL;
    if (T < 1 || T > c->max_tokens) return DS4G_EINVAL;
    if (gut != c->gut || dt != c->dt) return DS4G_EUNSUPPORTED;
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
        if (c->keys[i] >= 0 && !src.has(e)) return DS4G_EINVAL;
    }
    ds4g_status rc = c->lru.assign(c->keys.data(), n, c->slot.data(), c->miss.data());
    if (rc != DS4G_OK) return rc;
    for (int i = 0; i < 3 * kE; ++i) c->table_h[i] = nullptr;
    const SlotGeometry &g = c->geo;
    std::vector<int> todo;   // slots (first occurrences) whose expert must be copied
    for (int i = 0; i < n; ++i) {
        if (c->slot[i] < 0) continue;
        const int e = c->ids_h[i];
        uint8_t *dst = c->pool + (size_t)c->slot[i] * g.slot;
        if (c->miss[i]) todo.push_back(i);
        else if (!c->table_h[e]) ++c->hits;   // resident, first occurrence in this call
        c->table_h[e] = dst;
        c->table_h[kE + e] = dst + g.gate;
        c->table_h[2 * kE + e] = dst + 2 * g.gate;
    }
    const void **table_d = (const void **)(c->pool + g.table);
    if (cudaMemcpyAsync(table_d, c->table_h, 3 * kE * sizeof(void *), cudaMemcpyHostToDevice, st) != cudaSuccess) {
        for (int i : todo) c->lru.forget(c->slot[i]);
        return DS4G_ECUDA;
    }
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
    // Up to kDecodeMaxT tokens the copies run on the cache's copy stream while
    // the decode kernels already run the shared expert: slot i's routed work
    // waits for ready[i] == epoch, which the copy stream writes after that
    // slot's expert.  Larger T: the copies first, then the forward, on s.
    const bool overlap = T <= kDecodeMaxT && n <= kReadyFlags;
    cudaStream_t cst = overlap ? c->cs : st;
    uint32_t *ready_d = (uint32_t *)(c->pool + g.ready);
    uint32_t ep = 0;
    if (overlap) {
        ep = ++c->epoch;
        if (ep == 0) ep = ++c->epoch;
        for (int i = 0; i < n; ++i) {
            bool pending = false;
            for (int j : todo) pending = pending || c->ids_h[j] == c->ids_h[i];
            c->flag_h[i] = pending ? 0u : ep;
        }
        c->flag_h[kReadyFlags] = ep;
        if (cudaMemcpyAsync(ready_d, c->flag_h, (size_t)n * sizeof(uint32_t), cudaMemcpyHostToDevice, cst) !=
            cudaSuccess) {
            for (int i : todo) c->lru.forget(c->slot[i]);
            return DS4G_ECUDA;
        }
    }
    for (size_t q = 0; q < todo.size(); ++q) {
        const int i = todo[q], e = c->ids_h[i];
        uint8_t *dst = c->pool + (size_t)c->slot[i] * g.slot;
        rc = src.copy(e, dst, g, cst);
        for (int j = 0; rc == DS4G_OK && overlap && j < n; ++j)
            if (c->ids_h[j] == e &&
                cudaMemcpyAsync(ready_d + j, c->flag_h + kReadyFlags, sizeof(uint32_t), cudaMemcpyHostToDevice,
                                cst) != cudaSuccess)
                rc = DS4G_ECUDA;
        if (rc != DS4G_OK) {
            for (size_t r = q; r < todo.size(); ++r) c->lru.forget(c->slot[todo[r]]);   // nothing valid there
            if (overlap) cudaStreamSynchronize(cst);
            return rc;
        }
        ++c->misses;
        c->bytes += 2 * g.gate + g.down;
    }
    if (!overlap) return ds4g_moe_forward(hidden, T, &L, ids, w, out, workspace, ws_bytes, s);
    if (cudaEventRecord(c->copied, cst) != cudaSuccess) {
        cudaStreamSynchronize(cst);
        return DS4G_ECUDA;
    }
    rc = forward_streamed_decode(hidden, T, &L, ids, w, out, workspace, ws_bytes, st, ready_d, ep);
    // later work on s (the next call's slot rewrites included) follows the copies
    if (cudaStreamWaitEvent(st, c->copied, 0) != cudaSuccess) return DS4G_ECUDA;
    return rc;
}

extern "C" ds4g_status ds4g_moe_forward_streamed(const float *hidden, int T, int layer_key,
                                                 const ds4g_host_experts *src, const uint16_t *sh_gate,
                                                 const uint16_t *sh_up, const uint16_t *sh_down,
                                                 const uint64_t *iq2_grid, const int32_t *ids, const float *w,
                                                 float *out, ds4g_expert_cache *c, void *workspace,
                                                 size_t ws_bytes, ds4g_stream_t s) {
    DS4G_TRACE();
    if (!src || !src->gate || !src->up || !src->down) return DS4G_EINVAL;
    HostSource hs(src);
    return streamed_forward(hidden, T, layer_key, src->gate_up_type, src->down_type, hs, sh_gate, sh_up, sh_down,
                            iq2_grid, ids, w, out, c, workspace, ws_bytes, s);
}

// ---------------------------------------------------------------------------
// Expert files ([P1] §3.5, the DwarfStar page's "SSD Streaming": experts read
// from storage when they miss).  Layout, little-endian:
//   [0, 8)     magic "DS4GEXP1"
//   [8, 16)    uint32 gate_up_type, uint32 down_type
//   [16, 24)   uint32 n_experts (256), uint32 0
//   [24, 40)   uint64 bytes of one packed gate (= up) matrix, of one down matrix
//   [40, 48)   uint64 stride: bytes from one expert's record to the next
//   [48, 80)   presence bitmap, bit e of byte e / 8: expert e is stored
//   [80, 4096) zero
//   [4096 + e * stride, ...): expert e's packed gate, up, down (the layout of
//              ds4g_quantize_pack), back to back; stride = that size rounded
//              up to 4096 bytes
// ---------------------------------------------------------------------------
namespace ds4g {

constexpr size_t kFileHeader = 4096;
static const char kFileMagic[8] = {'D', 'S', '4', 'G', 'E', 'X', 'P', '1'};

struct FileHeader {
    char magic[8];
    uint32_t gut, dt, n, zero;
    uint64_t gate_bytes, down_bytes, stride;
    uint8_t present[kE / 8];
};
static_assert(sizeof(FileHeader) == 80, "expert file header");

static bool write_all(int fd, const void *p, size_t n, off_t off) {
    const uint8_t *b = (const uint8_t *)p;
    while (n) {
        const ssize_t w = pwrite(fd, b, n, off);
        if (w < 0 && errno == EINTR) continue;
        if (w <= 0) return false;
        b += w;
        n -= (size_t)w;
        off += w;
    }
    return true;
}
static bool read_all(int fd, void *p, size_t n, off_t off) {
    uint8_t *b = (uint8_t *)p;
    while (n) {
        const ssize_t r = pread(fd, b, n, off);
        if (r < 0 && errno == EINTR) continue;
        if (r <= 0) return false;
        b += r;
        n -= (size_t)r;
        off += r;
    }
    return true;
}

}  // namespace ds4g

struct ds4g_expert_file {
    int fd;
    ds4g::FileHeader h;
    uint8_t *stage[2];        // pinned staging buffers, one expert each
    cudaEvent_t done[2];      // copy out of stage[b] finished
    bool pending[2];
    int next;                 // staging buffer for the next expert
    ds4g_expert_file() : fd(-1), stage{nullptr, nullptr}, done{nullptr, nullptr}, pending{false, false}, next(0) {}
};

extern "C" ds4g_status ds4g_expert_file_write(const char *path, const ds4g_host_experts *src) {
    if (!path || !src || !src->gate || !src->up || !src->down) return DS4G_EINVAL;
    if (!stream_types_ok(src->gate_up_type, src->down_type)) return DS4G_EUNSUPPORTED;
    FileHeader h;
    memset(&h, 0, sizeof h);
    memcpy(h.magic, kFileMagic, 8);
    h.gut = (uint32_t)src->gate_up_type;
    h.dt = (uint32_t)src->down_type;
    h.n = kE;
    h.gate_bytes = ds4g_packed_size(src->gate_up_type, kF, kH);
    h.down_bytes = ds4g_packed_size(src->down_type, kH, kF);
    h.stride = align_up(2 * h.gate_bytes + h.down_bytes, 4096);
    for (int e = 0; e < kE; ++e) {
        const bool a = src->gate[e] != nullptr, b = src->up[e] != nullptr, d = src->down[e] != nullptr;
        if (a != b || a != d) return DS4G_EINVAL;   // an expert is stored whole or not at all
        if (a) h.present[e / 8] |= (uint8_t)(1u << (e % 8));
    }
    const int fd = open(path, O_WRONLY | O_CREAT | O_TRUNC, 0644);
    if (fd < 0) return DS4G_EINVAL;
    std::vector<uint8_t> head(kFileHeader, 0);
    memcpy(head.data(), &h, sizeof h);
    bool ok = write_all(fd, head.data(), kFileHeader, 0);
    for (int e = 0; ok && e < kE; ++e) {
        if (!src->gate[e]) continue;
        const off_t base = (off_t)(kFileHeader + (size_t)e * h.stride);
        ok = write_all(fd, src->gate[e], h.gate_bytes, base) &&
             write_all(fd, src->up[e], h.gate_bytes, base + (off_t)h.gate_bytes) &&
             write_all(fd, src->down[e], h.down_bytes, base + (off_t)(2 * h.gate_bytes));
    }
    // the file spans every record, stored or not
    ok = ok && ftruncate(fd, (off_t)(kFileHeader + (size_t)kE * h.stride)) == 0;
    ok = (close(fd) == 0) && ok;
    return ok ? DS4G_OK : DS4G_EINVAL;
}

extern "C" ds4g_status ds4g_expert_file_open(const char *path, ds4g_expert_file **file) {
    if (!path || !file) return DS4G_EINVAL;
    *file = nullptr;
    const int fd = open(path, O_RDONLY);
    if (fd < 0) return DS4G_EINVAL;
    FileHeader h;
    const off_t size = lseek(fd, 0, SEEK_END);
    bool ok = read_all(fd, &h, sizeof h, 0) && memcmp(h.magic, kFileMagic, 8) == 0 && h.n == (uint32_t)kE &&
              h.zero == 0;
    ok = ok && stream_types_ok((int)h.gut, (int)h.dt) &&
         h.gate_bytes == ds4g_packed_size((ds4g_qtype)h.gut, kF, kH) &&
         h.down_bytes == ds4g_packed_size((ds4g_qtype)h.dt, kH, kF) &&
         h.stride == align_up(2 * h.gate_bytes + h.down_bytes, 4096) &&
         size >= (off_t)(kFileHeader + (size_t)kE * h.stride);
    if (!ok) {
        close(fd);
        return DS4G_EINVAL;
    }
    ds4g_expert_file *f = new (std::nothrow) ds4g_expert_file();
    if (!f) {
        close(fd);
        return DS4G_ENOSPACE;
    }
    f->fd = fd;
    f->h = h;
    const size_t rec = 2 * h.gate_bytes + h.down_bytes;
    for (int b = 0; b < 2; ++b) {
        if (cudaHostAlloc((void **)&f->stage[b], rec, cudaHostAllocDefault) != cudaSuccess ||
            cudaEventCreateWithFlags(&f->done[b], cudaEventDisableTiming) != cudaSuccess) {
            ds4g_expert_file_close(f);
            return DS4G_ECUDA;
        }
    }
    *file = f;
    return DS4G_OK;
}

extern "C" ds4g_status ds4g_expert_file_close(ds4g_expert_file *f) {
    if (!f) return DS4G_EINVAL;
    bool ok = true;
    for (int b = 0; b < 2; ++b) {
        if (f->done[b]) ok = (cudaEventSynchronize(f->done[b]) == cudaSuccess) && ok;
        if (f->done[b]) ok = (cudaEventDestroy(f->done[b]) == cudaSuccess) && ok;
        if (f->stage[b]) ok = (cudaFreeHost(f->stage[b]) == cudaSuccess) && ok;
    }
    if (f->fd >= 0) close(f->fd);
    delete f;
    return ok ? DS4G_OK : DS4G_ECUDA;
}

namespace ds4g {

// Experts read from an expert file: each miss is read (pread) into one of two
// pinned staging buffers and copied from there; the read of the next expert
// overlaps the copy of the previous one, and a buffer is reused only after
// its copy has finished (an event).
struct FileSource : ExpertSource {
    ds4g_expert_file *f;
    explicit FileSource(ds4g_expert_file *file) : f(file) {}
    bool has(int e) const override { return (f->h.present[e / 8] >> (e % 8)) & 1u; }
    ds4g_status copy(int e, uint8_t *dst, const SlotGeometry &g, cudaStream_t st) override {
        const int b = f->next;
        f->next ^= 1;
        if (f->pending[b] && cudaEventSynchronize(f->done[b]) != cudaSuccess) return DS4G_ECUDA;
        f->pending[b] = false;
        const size_t rec = 2 * g.gate + g.down;
        if (!read_all(f->fd, f->stage[b], rec, (off_t)(kFileHeader + (size_t)e * f->h.stride))) return DS4G_EINVAL;
        if (cudaMemcpyAsync(dst, f->stage[b], rec, cudaMemcpyHostToDevice, st) != cudaSuccess ||
            cudaEventRecord(f->done[b], st) != cudaSuccess)
            return DS4G_ECUDA;
        f->pending[b] = true;
        return DS4G_OK;
    }
};

}  // namespace ds4g

extern "C" ds4g_status ds4g_moe_forward_streamed_file(const float *hidden, int T, int layer_key,
                                                      ds4g_expert_file *file, const uint16_t *sh_gate,
                                                      const uint16_t *sh_up, const uint16_t *sh_down,
                                                      const uint64_t *iq2_grid, const int32_t *ids, const float *w,
                                                      float *out, ds4g_expert_cache *c, void *workspace,
                                                      size_t ws_bytes, ds4g_stream_t s) {
    DS4G_TRACE();
    if (!file) return DS4G_EINVAL;
    FileSource fs(file);
    return streamed_forward(hidden, T, layer_key, (int)file->h.gut, (int)file->h.dt, fs, sh_gate, sh_up, sh_down,
                            iq2_grid, ids, w, out, c, workspace, ws_bytes, s);
}
