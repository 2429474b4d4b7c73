// paged.cu -- paged expert weights: a fixed GPU budget of expert slots shared
// by every paged layer of a model, arranged as N sets (indices) x M ways
// (expert-cache article, section 2.2: S = floor(available / expert size)
// slots, N = floor(S / M) sets, layer l uses set l mod N, least recently used
// expert replaced inside a set).  Each paged layer keeps its experts (in the
// stored, packed layout) in pinned host memory; a forward pass
//   1. copies the per-expert token counts to the host (the one host
//      synchronisation of the call), on the stream of the routing call that
//      wrote them, so that routing issued ahead on a side stream lets the
//      host look up and issue this layer's copies while earlier layers still
//      compute,
//   2. for each expert with tokens, in ascending id: looks it up in the set;
//      on a miss, picks a free or the least recently used way, makes the copy
//      stream wait until the compute that last read that slot has finished,
//      and copies the expert there page by page (page_bytes per copy) on the
//      copy stream (expert-cache article, section 3.2: weights move on a
//      stream of their own);
//   3. makes the compute stream wait for the expert's copy and runs the
//      expert's kernels, then records that the slot is in use until they end.
// So the copy of expert i+1 overlaps the compute of expert i (the expert
// prefetch of the HARMOEny write-up, part 3.2).  With cross-layer prefetch on
// (moe_pool_set_prefetch), a call then also copies, for layer_id + 1, the
// experts this call used most (up to the prefetch count), guessing that the
// next layer picks the same ones (expert-cache article, section 2.1); the
// copies queue on the copy stream behind this call's own.  The launch plan (token tiles,
// reduction splits) is the one a resident layer uses for the same T, so a paged
// layer's output is bit-identical to the resident layer's.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/moe_layer.h"
#include "common.cuh"
#include "kernels.cuh"
#include "layer_impl.h"

using namespace moe;

namespace {
constexpr size_t kLogCap = size_t(1) << 20;
size_t round256(size_t b) { return (b + 255) / 256 * 256; }
}  // namespace

struct moe_pool {
    int device = -1;
    size_t expert_bytes = 0, slot_bytes = 0, page_bytes = 0;
    int n_index = 0, ways = 0, n_slots = 0;
    uint8_t *slots = nullptr;
    cudaStream_t copy_stream = nullptr;
    struct Slot {
        int layer = -1, expert = -1;
        long long last_use = -1;
        bool fetched = false;         // filled by a prefetch and not used since
        cudaEvent_t ready = nullptr;  // copy into the slot finished
        cudaEvent_t busy = nullptr;   // last compute reading the slot finished
        bool busy_recorded = false;
    };
    std::vector<Slot> slot;
    std::vector<moe_layer *> layer_of;  // attached paged layers by layer id
    int prefetch = 0;                   // experts prefetched for the next layer per call
    long long fault_page = -1;          // MOE_FAULT_COPY_FAIL: index of the page copy to fail
    long long pages_issued = 0;
    long long clock = 0;
    std::vector<int32_t> log;  // (layer, expert, hit, slot) per query
    std::mutex mu;
    ~moe_pool();
};

moe_pool::~moe_pool() {
    if (device >= 0) cudaSetDevice(device);
    if (copy_stream) cudaStreamSynchronize(copy_stream);
    for (Slot &s : slot) {
        if (s.ready) cudaEventDestroy(s.ready);
        if (s.busy) cudaEventDestroy(s.busy);
    }
    if (slots) cudaFree(slots);
    if (copy_stream) cudaStreamDestroy(copy_stream);
}

extern "C" moe_status_t moe_pool_geometry(size_t budget_bytes, size_t expert_bytes, int ways,
                                          int *n_index, int *usable_slots) {
    if (!n_index || !usable_slots) return fail(MOE_ERR_INVALID_ARG, "NULL output pointer");
    if (expert_bytes == 0 || ways < 1) return fail(MOE_ERR_INVALID_ARG, "expert_bytes and ways must be positive");
    const size_t S = budget_bytes / expert_bytes;
    const size_t N = S / static_cast<size_t>(ways);
    if (N < 1) return fail(MOE_ERR_INVALID_ARG, "budget holds fewer than one set of %d ways", ways);
    if (N > (1u << 30)) return fail(MOE_ERR_INVALID_ARG, "too many sets");
    *n_index = static_cast<int>(N);
    *usable_slots = static_cast<int>(N) * ways;
    return MOE_OK;
}

extern "C" moe_status_t moe_pool_create(size_t budget_bytes, size_t expert_bytes, int ways,
                                        size_t page_bytes, moe_pool_t **out) {
    if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    int n_index = 0, usable = 0;
    moe_status_t st = moe_pool_geometry(budget_bytes, expert_bytes, ways, &n_index, &usable);
    if (st != MOE_OK) return st;
    if (page_bytes == 0) page_bytes = size_t(16) << 20;
    if (page_bytes % 256) return fail(MOE_ERR_INVALID_ARG, "page_bytes must be a multiple of 256");
    moe_pool *P = new (std::nothrow) moe_pool();
    if (!P) return fail(MOE_ERR_OOM, "host allocation failed");
    P->expert_bytes = expert_bytes;
    // a layer stores an expert as up to three 256-byte aligned parts
    P->slot_bytes = round256(expert_bytes) + 768;
    P->page_bytes = page_bytes;
    P->n_index = n_index;
    P->ways = ways;
    P->n_slots = usable;
    if (const char *f = std::getenv("MOE_FAULT_COPY_FAIL")) P->fault_page = std::atoll(f);
    cudaError_t e = cudaGetDevice(&P->device);
    if (e == cudaSuccess) e = cudaMalloc(&P->slots, P->slot_bytes * static_cast<size_t>(usable));
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&P->copy_stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) {
        P->slot.resize(static_cast<size_t>(usable));
        for (auto &s : P->slot) {
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.ready, cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.busy, cudaEventDisableTiming);
        }
    }
    if (e != cudaSuccess) {
        delete P;
        return cuda_fail(e, "moe_pool_create");
    }
    *out = P;
    return MOE_OK;
}

extern "C" moe_status_t moe_pool_destroy(moe_pool_t *pool) {
    delete pool;
    return MOE_OK;
}

extern "C" moe_status_t moe_pool_set_prefetch(moe_pool_t *pool, int max_experts) {
    if (!pool || max_experts < 0) return fail(MOE_ERR_INVALID_ARG, "pool is NULL or count negative");
    std::lock_guard<std::mutex> lock(pool->mu);
    pool->prefetch = max_experts;
    return MOE_OK;
}

extern "C" moe_status_t moe_pool_query_log(moe_pool_t *pool, int32_t *layer, int32_t *expert,
                                           int32_t *hit, int32_t *slot, int max, int *n_out) {
    if (!pool || !n_out || max < 0) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    std::lock_guard<std::mutex> lock(pool->mu);
    const int n = static_cast<int>(std::min<size_t>(pool->log.size() / 4, static_cast<size_t>(max)));
    for (int i = 0; i < n; ++i) {
        if (layer) layer[i] = pool->log[4 * i];
        if (expert) expert[i] = pool->log[4 * i + 1];
        if (hit) hit[i] = pool->log[4 * i + 2];
        if (slot) slot[i] = pool->log[4 * i + 3];
    }
    *n_out = n;
    return MOE_OK;
}

// ---- layer attach / detach -----------------------------------------------------------
moe_status_t paged_attach(moe_layer *L) {
    moe_pool *P = L->pool;
    if (L->expert_stride > P->slot_bytes)
        return fail(MOE_ERR_INVALID_ARG,
                    "pool slots hold %zu bytes but this layer stores %zu bytes per expert "
                    "(create the pool with moe_layer_info().expert_bytes)",
                    P->slot_bytes, L->expert_stride);
    if (P->device != L->device) return fail(MOE_ERR_INVALID_ARG, "pool and layer on different devices");
    {
        std::lock_guard<std::mutex> lock(P->mu);
        const size_t id = static_cast<size_t>(L->layer_id);
        if (id < P->layer_of.size() && P->layer_of[id])
            return fail(MOE_ERR_INVALID_ARG, "layer id %d is already attached to this pool", L->layer_id);
        if (id >= P->layer_of.size()) P->layer_of.resize(id + 1, nullptr);
        P->layer_of[id] = L;
    }
    const size_t bytes = L->expert_stride * static_cast<size_t>(L->cfg.E);
    void *host = nullptr;
    cudaError_t e = cudaHostAlloc(&host, bytes, cudaHostAllocDefault);
    if (e != cudaSuccess) return cuda_fail(e, "cudaHostAlloc(paged weights)");
    L->pinned_weights = static_cast<uint8_t *>(host);
    e = cudaMemcpy(L->pinned_weights, L->weights, bytes, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(paged weights)");
    // the device copy made during ingestion is no longer needed
    for (size_t i = 0; i < L->allocations.size(); ++i)
        if (L->allocations[i] == L->weights) {
            cudaFree(L->weights);
            L->allocations.erase(L->allocations.begin() + static_cast<long>(i));
            break;
        }
    L->weights = nullptr;
    return MOE_OK;
}

void paged_detach(moe_layer *L) {
    moe_pool *P = L->pool;
    if (!P) return;
    std::lock_guard<std::mutex> lock(P->mu);
    cudaStreamSynchronize(P->copy_stream);
    for (auto &s : P->slot)
        if (s.layer == L->layer_id) {
            s.layer = -1;
            s.expert = -1;
            s.last_use = -1;
            s.fetched = false;
        }
    const size_t id = static_cast<size_t>(L->layer_id);
    if (id < P->layer_of.size() && P->layer_of[id] == L) P->layer_of[id] = nullptr;
}

// ---- forward ---------------------------------------------------------------------------
namespace {

enum LogKind { kMiss = 0, kHit = 1, kPrefetch = 2, kPrefetchHit = 3 };

void pool_log(moe_pool *P, int layer, int expert, int kind, int slot) {
    if (P->log.size() + 4 <= 4 * kLogCap) {
        P->log.push_back(layer);
        P->log.push_back(expert);
        P->log.push_back(kind);
        P->log.push_back(slot);
    }
}

// Way of (layer, expert) in its set, or -1.
int pool_find(const moe_pool *P, int layer, int expert) {
    const int base = (layer % P->n_index) * P->ways;
    for (int w = 0; w < P->ways; ++w)
        if (P->slot[base + w].layer == layer && P->slot[base + w].expert == expert) return base + w;
    return -1;
}

// The way a new entry takes in the set of `layer`: the first empty way, else
// the least recently used.
int pool_victim(const moe_pool *P, int layer) {
    const int base = (layer % P->n_index) * P->ways;
    for (int w = 0; w < P->ways; ++w)
        if (P->slot[base + w].layer < 0) return base + w;
    int victim = base;
    for (int w = 1; w < P->ways; ++w)
        if (P->slot[base + w].last_use < P->slot[victim].last_use) victim = base + w;
    return victim;
}

// Demand lookup; on a miss the chosen way is re-tagged.  Returns the slot
// index and the log kind (miss, hit, or first use of a prefetched entry).
int pool_acquire(moe_pool *P, int layer, int expert, int *kind) {
    int si = pool_find(P, layer, expert);
    if (si < 0) {
        si = pool_victim(P, layer);
        P->slot[si].layer = layer;
        P->slot[si].expert = expert;
        P->slot[si].fetched = false;
        *kind = kMiss;
    } else {
        *kind = P->slot[si].fetched ? kPrefetchHit : kHit;
        P->slot[si].fetched = false;
    }
    P->slot[si].last_use = P->clock++;
    pool_log(P, layer, expert, *kind, si);
    return si;
}

// Copy expert `e` of layer N into slot si on the copy stream, page by page,
// after the last compute that read the slot; records the slot's ready event.
// Copy time is attributed to layer L (the caller).
moe_status_t pool_copy_in(moe_pool *P, moe_layer *L, moe_layer *N, int e, int si) {
    moe_pool::Slot &slot = P->slot[si];
    uint8_t *dst = P->slots + static_cast<size_t>(si) * P->slot_bytes;
    cudaError_t err = cudaSuccess;
    if (slot.busy_recorded) err = cudaStreamWaitEvent(P->copy_stream, slot.busy, 0);
    cudaEvent_t c0 = (err == cudaSuccess && L->timing) ? L->get_event() : nullptr;
    if (c0) err = cudaEventRecord(c0, P->copy_stream);
    const uint8_t *src = N->pinned_weights + N->expert_stride * static_cast<size_t>(e);
    for (size_t off = 0; err == cudaSuccess && off < N->expert_stride; off += P->page_bytes) {
        if (P->pages_issued++ == P->fault_page) {
            // injected failure: the slot holds a partial expert, so it must
            // not be found again; the caller sees the error
            slot.layer = -1;
            slot.expert = -1;
            slot.fetched = false;
            return fail(MOE_ERR_CUDA, "injected page-copy failure (MOE_FAULT_COPY_FAIL=%lld)", P->fault_page);
        }
        const size_t n = std::min(P->page_bytes, N->expert_stride - off);
        err = cudaMemcpyAsync(dst + off, src + off, n, cudaMemcpyHostToDevice, P->copy_stream);
    }
    if (err == cudaSuccess) err = cudaEventRecord(slot.ready, P->copy_stream);
    if (err == cudaSuccess && c0) {
        cudaEvent_t c1 = L->get_event();
        if (c1) {
            err = cudaEventRecord(c1, P->copy_stream);
            L->pending.push_back({MOE_PHASE_COPY, c0, c1});
        }
    }
    if (err != cudaSuccess) return cuda_fail(err, "expert page copy");
    L->stats.h2d_bytes += N->expert_stride;
    return MOE_OK;
}

// Cross-layer prefetch after layer L's demand lookups: up to P->prefetch of
// the experts with tokens (most tokens first, ties to the lower id) are
// brought in for layer L + 1 if it is attached and maps to another set.
moe_status_t pool_prefetch_next(moe_pool *P, moe_layer *L, const int32_t *counts, int E) {
    const int nl = L->layer_id + 1;
    if (P->prefetch <= 0 || nl >= static_cast<int>(P->layer_of.size()) || !P->layer_of[nl]) return MOE_OK;
    if (nl % P->n_index == L->layer_id % P->n_index) return MOE_OK;  // would evict this layer's experts
    moe_layer *N = P->layer_of[nl];
    if (N->cfg.E != E || N->expert_stride > P->slot_bytes) return MOE_OK;
    std::vector<int> order;
    for (int e = 0; e < E; ++e)
        if (counts[e] > 0) order.push_back(e);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return counts[a] > counts[b]; });
    if (static_cast<int>(order.size()) > P->prefetch) order.resize(static_cast<size_t>(P->prefetch));
    for (int e : order) {
        if (pool_find(P, nl, e) >= 0) continue;
        const int si = pool_victim(P, nl);
        moe_pool::Slot &slot = P->slot[si];
        slot.layer = nl;
        slot.expert = e;
        slot.fetched = true;
        slot.last_use = P->clock++;
        pool_log(P, nl, e, kPrefetch, si);
        moe_status_t st = pool_copy_in(P, L, N, e, si);
        if (st != MOE_OK) return st;
        L->stats.prefetch_copies += 1;
    }
    return MOE_OK;
}

}  // namespace

#define PG_TRY(expr)                                        \
    do {                                                    \
        cudaError_t e_ = (expr);                            \
        if (e_ != cudaSuccess) return cuda_fail(e_, #expr); \
    } while (0)

moe_status_t paged_forward(moe_layer *L, const void *x, const moe_routing_t *r, void *y,
                           cudaStream_t s) {
    moe_pool *P = L->pool;
    const moe_config_t &c = L->cfg;
    std::lock_guard<std::mutex> lock(P->mu);
    if (!L->counts_host) {
        PG_TRY(cudaHostAlloc(reinterpret_cast<void **>(&L->counts_host), sizeof(int32_t) * c.E,
                             cudaHostAllocDefault));
        PG_TRY(cudaEventCreate(&L->fwd_t0));
        PG_TRY(cudaEventCreate(&L->fwd_t1));
        PG_TRY(cudaEventCreateWithFlags(&L->counts_ready, cudaEventDisableTiming));
    }
    // 1. token counts to the host: the one synchronisation of a paged call
    if (L->fwd_pending) {  // the previous call's duration
        moe_status_t w = wait_event(L->fwd_t1, L->host_timeout_ms, "the previous paged call");
        if (w != MOE_OK) return w;
        float ms = 0.0f;
        PG_TRY(cudaEventElapsedTime(&ms, L->fwd_t0, L->fwd_t1));
        L->stats.forward_ms += ms;
        L->fwd_pending = false;
    }
    PG_TRY(cudaEventRecord(L->fwd_t0, s));
    // The counts are read on the stream of the routing call that wrote them
    // (when these tables come from this layer's last routing call), so a
    // caller that routes ahead on a side stream gets them without waiting for
    // the compute queued on `s`, and the copy stream is fed without a gap;
    // `s` then waits for that read before any expert reads the tables.
    cudaStream_t rs = (L->route_stream && L->route_counts == r->counts) ? L->route_stream : s;
    L->route_stream = nullptr;
    L->route_counts = nullptr;
    PG_TRY(cudaMemcpyAsync(L->counts_host, r->counts, sizeof(int32_t) * c.E, cudaMemcpyDeviceToHost, rs));
    PG_TRY(cudaEventRecord(L->counts_ready, rs));
    {
        moe_status_t w = wait_event(L->counts_ready, L->host_timeout_ms, "the token counts");
        if (w != MOE_OK) return w;  // no slot state changed yet
    }
    if (rs != s) PG_TRY(cudaStreamWaitEvent(s, L->counts_ready, 0));

    // the launch plan of a resident layer for the same T (bit-identical results)
    ExpertArgs a = make_expert_args(L, x, r);
    int splits = 1, nrows_cap = 0;
    bool part_bf16 = false;
    moe_status_t st = MOE_OK;
    bool first = true;
    for (int e = 0; e < c.E; ++e) {
        if (L->counts_host[e] <= 0) continue;
        int kind = kMiss;
        const int si = pool_acquire(P, L->layer_id, e, &kind);
        moe_pool::Slot &slot = P->slot[si];
        uint8_t *dst = P->slots + static_cast<size_t>(si) * P->slot_bytes;
        if (kind == kMiss) {
            // never overwrite weights a kernel may still be reading
            moe_status_t cs = pool_copy_in(P, L, L, e, si);
            if (cs != MOE_OK) return cs;
            L->stats.slot_misses += 1;
        } else {
            L->stats.slot_hits += 1;
            if (kind == kPrefetchHit) L->stats.prefetch_hits += 1;
        }
        PG_TRY(cudaStreamWaitEvent(s, slot.ready, 0));
        // this expert's stored matrices now live in the slot
        const size_t mp = static_cast<size_t>(c.m) * c.p;
        const bool gated = c.expert == MOE_EXPERT_SWIGLU;
        const bool i8 = c.weight_dtype == MOE_I8;
        const size_t wel = i8 ? 1 : 2;
        const size_t u_bytes = round256((gated ? 2 : 1) * mp * wel), d_bytes = round256(mp * wel);
        L->tab.w1[e] = dst;
        L->tab.w2[e] = dst + u_bytes;
        if (i8) {
            float *sc = reinterpret_cast<float *>(dst + u_bytes + d_bytes);
            L->tab.s1[e] = sc;
            L->tab.s3[e] = gated ? sc + c.p : nullptr;
            L->tab.s2[e] = sc + static_cast<size_t>(c.p) * (gated ? 2 : 1);
        }
        a.only[0] = e;
        a.n_only = 1;
        a.tab = &L->tab;
        int sp = 1;
        st = run_experts(L, a, L->regime, &sp, s);
        if (st != MOE_OK) return st;
        if (first) {
            splits = sp;
            nrows_cap = a.n_rows_cap;
            part_bf16 = a.ypart_bf16 != 0;
            first = false;
        }
        PG_TRY(cudaEventRecord(slot.busy, s));
        slot.busy_recorded = true;
    }
    if (!first) {
        st = run_combine(L, r, splits, nrows_cap, part_bf16, y, s);
        if (st != MOE_OK) return st;
    }
    st = pool_prefetch_next(P, L, L->counts_host, c.E);
    if (st != MOE_OK) return st;
    PG_TRY(cudaEventRecord(L->fwd_t1, s));
    L->last_stream = s;
    L->launched = true;
    L->fwd_pending = true;
    L->stats.forwards += 1;
    return MOE_OK;
}
