// moe_layer.cu -- host side of the C ABI declared in include/moe_layer.h:
// argument validation, weight ingestion, workspace ownership, regime choice
// and kernel orchestration on the caller's stream.
//
// The layer computes the forward pass the pages describe for one MoE FFN
// layer (HARMOEny write-up, parts 1 and 3.3; expert shape of part 3.2):
//   moe_route   : router GEMM + softmax + top-k, then histogram / scan /
//                 stable permute (the one-device form of the dispatch)
//   moe_forward : expert up-projection + activation, down-projection scaled by
//                 the routing weight, weighted un-permute and combine.
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <thread>
#include <vector>

#include <cudaTypedefs.h>

#include "../../include/moe_layer.h"
#include "common.cuh"
#include "kernels.cuh"
#include "layer_impl.h"
#include "packing.h"

using namespace moe;

// ---- error text ----------------------------------------------------------------
namespace {
thread_local std::string g_last_error;
}

namespace moe {

moe_status_t fail(moe_status_t st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

moe_status_t cuda_fail(cudaError_t e, const char *where) {
    cudaGetLastError();  // clear a non-sticky error
    if (e == cudaErrorMemoryAllocation)
        return fail(MOE_ERR_OOM, "%s: %s", where, cudaGetErrorString(e));
    return fail(MOE_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

moe_status_t wait_event(cudaEvent_t ev, int timeout_ms, const char *what) {
    const auto t0 = std::chrono::steady_clock::now();
    for (long long polls = 0;; ++polls) {
        const cudaError_t q = cudaEventQuery(ev);
        if (q == cudaSuccess) return MOE_OK;
        if (q != cudaErrorNotReady) return cuda_fail(q, what);
        const long long el =
            std::chrono::duration_cast<std::chrono::milliseconds>(std::chrono::steady_clock::now() - t0).count();
        if (timeout_ms >= 0 && el >= timeout_ms)
            return fail(MOE_ERR_TIMEOUT, "%s: not finished after %d ms", what, timeout_ms);
        if (polls < 1000)
            std::this_thread::yield();
        else
            std::this_thread::sleep_for(std::chrono::microseconds(20));
    }
}

}  // namespace moe

#define CUDA_TRY(expr)                                      \
    do {                                                    \
        cudaError_t e_ = (expr);                            \
        if (e_ != cudaSuccess) return cuda_fail(e_, #expr); \
    } while (0)

namespace {

constexpr int kDecodeMaxRows = 512;          // T*k handled with split-K partials
constexpr size_t kSmemBudgetB = 64 * 1024;   // staged token rows per CTA

size_t act_bytes(moe_dtype_t d) { return d == MOE_F32 ? 4 : 2; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

constexpr int kSplitUpMax = 4, kSplitDownMax = 16;
// Mean tokens per expert above which the tensor-core path runs (measured
// crossover, Mixtral shape: bf16 GEMV 446 us vs tensor cores 455 us at T = 16,
// 473 vs 457 at T = 20).  The int8 weight-streaming kernel widens each code
// once per pass and reuses it for every token tile, so it stays ahead of the
// tensor cores for longer (T = 48: 364 vs 487 us).  At T = 64 it is ahead
// only while no expert needs a second pass (456 vs 492 us; with one expert of
// 25 tokens 509 vs 495), which skewed routing makes common, while the tensor
// cores read each weight once for any count: the crossover stays at 12.  With
// two MMA-issuing warps on small tiles the int8 tensor cores take 371 us at
// T = 48 and 376 us at T = 64, so 12 is now about where the paths are even.
constexpr int kTcMinMeanTokens = 4;
constexpr int kTcMinMeanTokensI8 = 12;

// Smallest split of a K-long reduction whose staged token rows (8 * nt rows of
// K / splits bf16) fit the shared-memory budget.
int splits_for(int K, int nt, int min_splits) {
    int s = ceil_div(static_cast<long long>(8) * nt * 2 * K, static_cast<long long>(kSmemBudgetB));
    if (s < min_splits) s = min_splits;
    return s;
}

// Expected number of distinct experts that T tokens choose under uniform
// routing, E (1 - (1 - k/E)^T): exactly k for one token.
int expected_active(int T, int k, int E) {
    double miss = 1.0;
    for (int t = 0; t < T && miss > 1e-9; ++t) miss *= 1.0 - static_cast<double>(k) / E;
    int n = static_cast<int>(E * (1.0 - miss) + 0.5);
    return n < k ? k : (n > E ? E : n);
}

// Reduction split for a decode projection: at least what the staging budget
// needs, then the smallest count (up to max_s) whose units -- n_active
// experts x splits x ceil(rows / 128) -- fill the SMs in nearly whole waves.
int choose_splits(int K, int bk, int rows, int nt, int n_active, int num_sms, int max_s) {
    const int nkb = K / bk;
    const int rg8 = (rows / 16 + 7) / 8;
    int s0 = splits_for(K, nt, 1);
    if (s0 > max_s) s0 = max_s;
    int best = s0;
    double best_eff = -1.0;
    for (int S = s0; S <= max_s && S <= nkb; ++S) {
        const long long units = static_cast<long long>(n_active) * S * rg8;
        const long long waves = (units + num_sms - 1) / num_sms;
        const double eff = static_cast<double>(units) / static_cast<double>(waves * num_sms);
        if (eff >= 0.92) return S;
        if (eff > best_eff) {
            best_eff = eff;
            best = S;
        }
    }
    return best;
}

moe_status_t check_config(const moe_config_t *c) {
    if (!c) return fail(MOE_ERR_INVALID_ARG, "config is NULL");
    if (c->m <= 0 || c->p <= 0) return fail(MOE_ERR_INVALID_ARG, "m and p must be positive");
    if (c->E < 1 || c->E > kMaxExperts)
        return fail(MOE_ERR_INVALID_ARG, "E must be in [1, %d]", kMaxExperts);
    if (c->k < 1 || c->k > c->E || c->k > kMaxTopK)
        return fail(MOE_ERR_INVALID_ARG, "k must be in [1, min(E, %d)]", kMaxTopK);
    if (c->max_tokens < 1 || static_cast<long long>(c->max_tokens) * c->k > (1 << 30))
        return fail(MOE_ERR_INVALID_ARG, "max_tokens out of range");
    if (c->act_dtype != MOE_F32 && c->act_dtype != MOE_BF16)
        return fail(MOE_ERR_INVALID_ARG, "act_dtype must be F32 or BF16");
    if (c->expert != MOE_EXPERT_RELU2 && c->expert != MOE_EXPERT_SWIGLU)
        return fail(MOE_ERR_INVALID_ARG, "unknown expert form");
    if (c->act_dtype == MOE_F32) {
        if (c->weight_dtype != MOE_F32)
            return fail(MOE_ERR_UNSUPPORTED, "fp32 activations need fp32 weights");
        if (c->m % 4) return fail(MOE_ERR_UNSUPPORTED, "fp32 layers need m %% 4 == 0");
    } else {
        if (c->weight_dtype != MOE_BF16 && c->weight_dtype != MOE_I8)
            return fail(MOE_ERR_UNSUPPORTED, "bf16 activations need bf16 or int8 weights");
        if (c->m % 64 || c->p % 64)
            return fail(MOE_ERR_UNSUPPORTED, "bf16/int8 layers need m and p multiples of 64");
        if (c->weight_dtype == MOE_I8 && (c->m % 128 || c->p % 128))
            return fail(MOE_ERR_UNSUPPORTED, "int8 layers need m and p multiples of 128");
    }
    if (c->paged && c->weight_dtype == MOE_F32)
        return fail(MOE_ERR_UNSUPPORTED, "paged layers need bf16 or int8 weights");
    return MOE_OK;
}

moe_status_t check_routing(const moe_layer_t *L, const moe_routing_t *r) {
    if (!r) return fail(MOE_ERR_INVALID_ARG, "routing is NULL");
    if (!r->topk_ids || !r->topk_w || !r->counts || !r->offsets || !r->gather_index ||
        !r->scatter_index)
        return fail(MOE_ERR_INVALID_ARG, "a routing table pointer is NULL");
    (void)L;
    return MOE_OK;
}

}  // namespace

// ---- lifetime ---------------------------------------------------------------------
moe_layer::~moe_layer() {
    if (device >= 0) cudaSetDevice(device);
    for (void *p : allocations) cudaFree(p);
    if (pinned_weights) cudaFreeHost(pinned_weights);
    if (counts_host) cudaFreeHost(counts_host);
    if (fwd_t0) cudaEventDestroy(fwd_t0);
    if (fwd_t1) cudaEventDestroy(fwd_t1);
    if (counts_ready) cudaEventDestroy(counts_ready);
    for (cudaEvent_t ev : event_pool) cudaEventDestroy(ev);
    for (auto &pe : pending) {
        cudaEventDestroy(pe.a);
        cudaEventDestroy(pe.b);
    }
    if (done) cudaEventDestroy(done);
    if (ingest_stream) cudaStreamDestroy(ingest_stream);
}

cudaEvent_t moe_layer::get_event() {
    if (!event_pool.empty()) {
        cudaEvent_t ev = event_pool.back();
        event_pool.pop_back();
        return ev;
    }
    cudaEvent_t ev = nullptr;
    if (cudaEventCreate(&ev) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return ev;
}

void *moe_layer::dalloc(size_t bytes, cudaError_t *err) {
    void *p = nullptr;
    *err = cudaMalloc(&p, bytes ? bytes : 16);
    if (*err == cudaSuccess) allocations.push_back(p);
    return p;
}

static size_t round256(size_t b) { return (b + 255) / 256 * 256; }

static void free_one(moe_layer_t *L, void *p) {
    if (!p) return;
    for (size_t i = 0; i < L->allocations.size(); ++i)
        if (L->allocations[i] == p) {
            cudaFree(p);
            L->allocations.erase(L->allocations.begin() + static_cast<long>(i));
            return;
        }
}

static moe_status_t ingest_weights(moe_layer_t *L, const void *w_router, const float *b_router,
                                   const void *const *w1, const void *const *w2,
                                   const void *const *w3) {
    const moe_config_t &c = L->cfg;
    cudaError_t err;
    cudaStream_t s = L->ingest_stream;
    const bool bf16_act = c.act_dtype == MOE_BF16;
    const bool gated = c.expert == MOE_EXPERT_SWIGLU;
    const bool i8 = c.weight_dtype == MOE_I8;
    const size_t ab = act_bytes(c.act_dtype);
    const size_t src_elem = (c.weight_dtype == MOE_F32) ? 4 : 2;
    const size_t mp = static_cast<size_t>(c.m) * c.p;

    // router: [m x E] act type -> fp32 [E x m]
    void *stage_r = L->dalloc(static_cast<size_t>(c.m) * c.E * ab, &err);
    if (err) return cuda_fail(err, "cudaMalloc(router staging)");
    L->wrt = static_cast<float *>(L->dalloc(static_cast<size_t>(c.m) * c.E * 4, &err));
    if (err) return cuda_fail(err, "cudaMalloc(router)");
    CUDA_TRY(cudaMemcpyAsync(stage_r, w_router, static_cast<size_t>(c.m) * c.E * ab,
                             cudaMemcpyHostToDevice, s));
    CUDA_TRY(launch_router_prep(stage_r, bf16_act, c.m, c.E, L->wrt, s));
    // activation-typed copy [E_pad x m], zero rows past E (E_pad = 8, 16, 32 or 64)
    const int e_pad = c.E <= 8 ? 8 : c.E <= 16 ? 16 : c.E <= 32 ? 32 : 64;
    L->wra = L->dalloc(static_cast<size_t>(c.m) * e_pad * ab, &err);
    if (err) return cuda_fail(err, "cudaMalloc(router)");
    CUDA_TRY(cudaMemsetAsync(L->wra, 0, static_cast<size_t>(c.m) * e_pad * ab, s));
    CUDA_TRY(launch_transpose(stage_r, L->wra, c.m, c.E, static_cast<int>(ab), s));
    if (c.has_router_bias) {
        L->bias = static_cast<float *>(L->dalloc(static_cast<size_t>(c.E) * 4, &err));
        if (err) return cuda_fail(err, "cudaMalloc(bias)");
        CUDA_TRY(cudaMemcpyAsync(L->bias, b_router, static_cast<size_t>(c.E) * 4,
                                 cudaMemcpyHostToDevice, s));
    }

    // experts: one allocation holding every expert's stored matrices
    const int nmat = gated ? 3 : 2;
    const size_t wel = i8 ? 1 : src_elem;
    const int rows_u = gated ? 2 * c.p : c.p;
    size_t u_bytes, d_bytes, scale_bytes = 0;
    if (c.weight_dtype == MOE_F32) {  // W1^T, W2^T, W3^T row-major
        u_bytes = round256(mp * wel) * (gated ? 2 : 1);
        d_bytes = round256(mp * wel);
    } else {  // packed U and D
        u_bytes = round256(static_cast<size_t>(rows_u) * c.m * wel);
        d_bytes = round256(mp * wel);
        if (i8) scale_bytes = round256((static_cast<size_t>(c.p) * (nmat - 1) + c.m) * 4);
    }
    L->expert_stride = u_bytes + d_bytes + scale_bytes;
    L->expert_bytes = mp * wel * nmat + (i8 ? (static_cast<size_t>(c.p) * (nmat - 1) + c.m) * 4 : 0);
    L->weights = static_cast<uint8_t *>(L->dalloc(L->expert_stride * c.E, &err));
    if (err) return cuda_fail(err, "cudaMalloc(expert weights)");
    void *stage = L->dalloc(mp * src_elem, &err);
    if (err) return cuda_fail(err, "cudaMalloc(weight staging)");
    void *t1 = nullptr, *t3 = nullptr, *q1 = nullptr, *q3 = nullptr;
    if (c.weight_dtype != MOE_F32) {
        t1 = L->dalloc(mp * 2, &err);
        if (!err && gated) t3 = L->dalloc(mp * 2, &err);
        if (!err && i8) q1 = L->dalloc(mp, &err);
        if (!err && i8 && gated) q3 = L->dalloc(mp, &err);
        if (err) return cuda_fail(err, "cudaMalloc(weight staging)");
    }
    for (int e = 0; e < c.E; ++e) {
        uint8_t *base = L->weights + L->expert_stride * e;
        uint8_t *U = base, *D = base + u_bytes;
        float *sc = reinterpret_cast<float *>(base + u_bytes + d_bytes);
        float *s1 = i8 ? sc : nullptr;
        float *s3 = (i8 && gated) ? sc + c.p : nullptr;
        float *s2 = i8 ? sc + static_cast<size_t>(c.p) * (nmat - 1) : nullptr;
        // the staging buffers are reused: every step is ordered on stream s
        if (c.weight_dtype == MOE_F32) {
            uint8_t *W1t = U, *W3t = gated ? U + round256(mp * wel) : nullptr;
            CUDA_TRY(cudaMemcpyAsync(stage, w1[e], mp * 4, cudaMemcpyHostToDevice, s));
            CUDA_TRY(launch_transpose(stage, W1t, c.m, c.p, 4, s));
            if (gated) {
                CUDA_TRY(cudaMemcpyAsync(stage, w3[e], mp * 4, cudaMemcpyHostToDevice, s));
                CUDA_TRY(launch_transpose(stage, W3t, c.m, c.p, 4, s));
            }
            CUDA_TRY(cudaMemcpyAsync(stage, w2[e], mp * 4, cudaMemcpyHostToDevice, s));
            CUDA_TRY(launch_transpose(stage, D, c.p, c.m, 4, s));
            L->tab.w1[e] = W1t;
            L->tab.w3[e] = W3t;
            L->tab.w2[e] = D;
            continue;
        }
        // up: W1^T (and W3^T) [p x m] -> packed U (gate/up rows interleaved per 8)
        CUDA_TRY(cudaMemcpyAsync(stage, w1[e], mp * 2, cudaMemcpyHostToDevice, s));
        CUDA_TRY(launch_transpose(stage, t1, c.m, c.p, 2, s));
        if (gated) {
            CUDA_TRY(cudaMemcpyAsync(stage, w3[e], mp * 2, cudaMemcpyHostToDevice, s));
            CUDA_TRY(launch_transpose(stage, t3, c.m, c.p, 2, s));
        }
        if (i8) {
            CUDA_TRY(launch_quantize_rows(t1, c.p, c.m, static_cast<int8_t *>(q1), s1, s));
            if (gated) CUDA_TRY(launch_quantize_rows(t3, c.p, c.m, static_cast<int8_t *>(q3), s3, s));
            CUDA_TRY(launch_pack(q1, gated ? q3 : nullptr, rows_u, c.m, 1, U, s));
        } else {
            CUDA_TRY(launch_pack(t1, gated ? t3 : nullptr, rows_u, c.m, 2, U, s));
        }
        // down: W2^T [m x p] -> packed D
        CUDA_TRY(cudaMemcpyAsync(stage, w2[e], mp * 2, cudaMemcpyHostToDevice, s));
        CUDA_TRY(launch_transpose(stage, t1, c.p, c.m, 2, s));
        if (i8) {
            CUDA_TRY(launch_quantize_rows(t1, c.m, c.p, static_cast<int8_t *>(q1), s2, s));
            CUDA_TRY(launch_pack(q1, nullptr, c.m, c.p, 1, D, s));
        } else {
            CUDA_TRY(launch_pack(t1, nullptr, c.m, c.p, 2, D, s));
        }
        L->tab.w1[e] = U;
        L->tab.w2[e] = D;
        L->tab.w3[e] = nullptr;
        L->tab.s1[e] = s1;
        L->tab.s2[e] = s2;
        L->tab.s3[e] = s3;
    }
    CUDA_TRY(cudaStreamSynchronize(s));
    for (void *p : {stage_r, stage, t1, t3, q1, q3}) free_one(L, p);
    return MOE_OK;
}

namespace moe {

WorkspaceGeom workspace_geom(const moe_config_t &c) {
    WorkspaceGeom g;
    const size_t rows = static_cast<size_t>(c.max_tokens) * c.k;
    g.ypart_rows = rows;
    if (c.act_dtype == MOE_BF16) {
        g.split_up_max = kSplitUpMax;
        g.split_down_max = kSplitDownMax;
        g.decode_rows_cap = rows < static_cast<size_t>(kDecodeMaxRows) ? rows : kDecodeMaxRows;
        // decode: split_down_max partial rows per permuted row (T*k <= the cap);
        // batch: one fp32 row per permuted row
        const size_t need = static_cast<size_t>(g.split_down_max) * g.decode_rows_cap;
        g.ypart_rows = rows > need ? rows : need;
    }
    return g;
}

}  // namespace moe

static moe_status_t alloc_workspace(moe_layer_t *L) {
    const moe_config_t &c = L->cfg;
    cudaError_t err;
    const size_t rows = static_cast<size_t>(c.max_tokens) * c.k;
    const size_t ab = act_bytes(c.act_dtype);
    L->h = L->dalloc(rows * c.p * ab, &err);
    if (err) return cuda_fail(err, "cudaMalloc(h)");
    const WorkspaceGeom g = workspace_geom(c);
    const size_t ypart_rows = g.ypart_rows;
    L->split_up_max = g.split_up_max;
    L->split_down_max = g.split_down_max;
    L->decode_rows_cap = g.decode_rows_cap;
    if (c.act_dtype == MOE_BF16) {
        if (L->split_up_max > 1) {
            const size_t n = static_cast<size_t>(L->split_up_max) * g.decode_rows_cap * c.p;
            L->gate_part = static_cast<float *>(L->dalloc(n * 4, &err));
            if (err) return cuda_fail(err, "cudaMalloc(gate partials)");
            L->up_part = static_cast<float *>(L->dalloc(n * 4, &err));
            if (err) return cuda_fail(err, "cudaMalloc(up partials)");
            L->workspace_bytes += 2 * n * 4;
        }
    }
    if (c.act_dtype == MOE_BF16) {  // token rows in expert order for the tensor-core path
        L->x_perm = L->dalloc(rows * c.m * 2, &err);
        if (err) return cuda_fail(err, "cudaMalloc(x_perm)");
        L->workspace_bytes += rows * c.m * 2;
        if (c.weight_dtype == MOE_I8) {  // scales and split sums of its fp16 form
            const size_t n = rows * (1 + static_cast<size_t>(L->split_up_max));
            L->x_scale = static_cast<float *>(L->dalloc(n * 4, &err));
            if (err) return cuda_fail(err, "cudaMalloc(token row scales)");
            L->x_sum = L->x_scale + rows;
            L->workspace_bytes += n * 4;
        }
    }
    L->ypart_rows = ypart_rows;
    L->ypart = static_cast<float *>(L->dalloc(ypart_rows * c.m * 4, &err));
    if (err) return cuda_fail(err, "cudaMalloc(ypart)");
    {  // one row of expert counts per 16-token router CTA
        const size_t n = static_cast<size_t>((c.max_tokens + 15) / 16) * c.E;
        L->cta_count = static_cast<int32_t *>(L->dalloc(n * 4, &err));
        if (err) return cuda_fail(err, "cudaMalloc(router permute counts)");
        L->workspace_bytes += n * 4;
    }
    L->err_word = static_cast<uint32_t *>(L->dalloc(8, &err));
    if (err) return cuda_fail(err, "cudaMalloc(error word)");
    CUDA_TRY(cudaMemset(L->err_word, 0, 8));
    L->ticket = reinterpret_cast<unsigned *>(L->err_word + 1);
    L->workspace_bytes += rows * c.p * ab + ypart_rows * c.m * 4;
    return MOE_OK;
}

extern "C" moe_status_t moe_layer_create(const moe_config_t *cfg, const void *w_router,
                                         const float *b_router, const void *const *w1,
                                         const void *const *w2, const void *const *w3,
                                         moe_pool_t *pool, int layer_id, moe_layer_t **out) {
    if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (!w_router || !w1 || !w2) return fail(MOE_ERR_INVALID_ARG, "weight pointer is NULL");
    if (cfg->has_router_bias && !b_router) return fail(MOE_ERR_INVALID_ARG, "b_router is NULL");
    const bool gated = cfg->expert == MOE_EXPERT_SWIGLU;
    if (gated != (w3 != nullptr))
        return fail(MOE_ERR_INVALID_ARG, "w3 must be given exactly for the SwiGLU form");
    for (int e = 0; e < cfg->E; ++e)
        if (!w1[e] || !w2[e] || (gated && !w3[e]))
            return fail(MOE_ERR_INVALID_ARG, "expert %d weight pointer is NULL", e);
    if (cfg->paged && !pool) return fail(MOE_ERR_INVALID_ARG, "paged layer needs a pool");
    if (!cfg->paged && pool) return fail(MOE_ERR_INVALID_ARG, "pool given for a resident layer");
    if (layer_id < 0) return fail(MOE_ERR_INVALID_ARG, "layer_id must be >= 0");

    moe_layer_t *L = new (std::nothrow) moe_layer();
    if (!L) return fail(MOE_ERR_OOM, "host allocation failed");
    L->cfg = *cfg;
    L->layer_id = layer_id;
    L->pool = pool;
    cudaError_t err = cudaGetDevice(&L->device);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device);
    if (err == cudaSuccess) err = cudaStreamCreateWithFlags(&L->ingest_stream, cudaStreamNonBlocking);
    if (err == cudaSuccess) err = cudaEventCreateWithFlags(&L->done, cudaEventDisableTiming);
    if (err != cudaSuccess) {
        delete L;
        return cuda_fail(err, "device setup");
    }
    std::memset(&L->tab, 0, sizeof L->tab);
    st = ingest_weights(L, w_router, b_router, w1, w2, w3);
    if (st == MOE_OK) st = alloc_workspace(L);
    if (st == MOE_OK && cfg->paged) st = paged_attach(L);
    if (st != MOE_OK) {
        std::string keep = g_last_error;
        delete L;
        g_last_error = keep;
        return st;
    }
    *out = L;
    return MOE_OK;
}

extern "C" moe_status_t moe_destroy(moe_layer_t *L) {
    if (!L) return MOE_OK;
    cudaSetDevice(L->device);
    cudaDeviceSynchronize();
    if (L->pool) paged_detach(L);
    delete L;
    return MOE_OK;
}

// ---- routing ---------------------------------------------------------------------------
static moe_status_t run_permute(moe_layer_t *L, int T, moe_routing_t *r, cudaStream_t s) {
    PermuteArgs pa{r->topk_ids, T, L->cfg.k, L->cfg.E, r->counts, r->offsets, r->gather_index,
                   r->scatter_index, nullptr};
    moe_status_t st = launch_phase(L, MOE_PHASE_PERMUTE, s, "permute", [&] { return launch_permute(pa, s); });
    if (st != MOE_OK) return st;
    L->last_stream = s;
    L->route_stream = s;
    L->route_counts = r->counts;
    L->launched = true;
    r->T = T;
    return MOE_OK;
}

static moe_status_t check_T(const moe_layer_t *L, int T) {
    if (T < 0 || T > L->cfg.max_tokens)
        return fail(MOE_ERR_INVALID_ARG, "T = %d outside [0, max_tokens = %d]", T, L->cfg.max_tokens);
    return MOE_OK;
}

extern "C" moe_status_t moe_route(moe_layer_t *L, const void *x, int T, moe_routing_t *r,
                                  void *stream) {
    NvtxRange range("moe_route");
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    moe_status_t st = check_T(L, T);
    if (st == MOE_OK) st = check_routing(L, r);
    if (st != MOE_OK) return st;
    if (T > 0 && (!x || !aligned16(x))) return fail(MOE_ERR_INVALID_ARG, "x is NULL or not 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) return run_permute(L, T, r, s);
    RouterArgs ra{x, L->wrt, L->wra, L->bias, T, L->cfg.m, L->cfg.E, L->cfg.k, r->topk_ids,
                  r->topk_w, r->logits, L->ticket, L->err_word};
    PermuteArgs pa{r->topk_ids, T, L->cfg.k, L->cfg.E, r->counts, r->offsets, r->gather_index,
                   r->scatter_index, L->cta_count};
    st = launch_phase(L, MOE_PHASE_ROUTER, s, "router_topk_permute",
                      [&] { return launch_router_topk(ra, pa, L->cfg.act_dtype == MOE_BF16, s); });
    if (st != MOE_OK) return st;
    L->last_stream = s;
    L->route_stream = s;
    L->route_counts = r->counts;
    L->launched = true;
    r->T = T;
    return MOE_OK;
}

extern "C" moe_status_t moe_route_from_logits(moe_layer_t *L, const float *logits, int T,
                                              moe_routing_t *r, void *stream) {
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    moe_status_t st = check_T(L, T);
    if (st == MOE_OK) st = check_routing(L, r);
    if (st != MOE_OK) return st;
    if (T > 0 && !logits) return fail(MOE_ERR_INVALID_ARG, "logits is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T > 0) {
        st = launch_phase(L, MOE_PHASE_ROUTER, s, "topk_from_logits", [&] {
            return launch_topk_from_logits(logits, T, L->cfg.E, L->cfg.k, r->topk_ids, r->topk_w, s);
        });
        if (st != MOE_OK) return st;
    }
    return run_permute(L, T, r, s);
}

extern "C" moe_status_t moe_route_from_topk(moe_layer_t *L, const int32_t *ids, const float *w,
                                            int T, moe_routing_t *r, void *stream) {
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    moe_status_t st = check_T(L, T);
    if (st == MOE_OK) st = check_routing(L, r);
    if (st != MOE_OK) return st;
    if (T > 0 && (!ids || !w)) return fail(MOE_ERR_INVALID_ARG, "ids or w is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T > 0) {
        st = launch_phase(L, MOE_PHASE_ROUTER, s, "topk_copy_validate", [&] {
            return launch_topk_copy_validate(ids, w, T, L->cfg.E, L->cfg.k, r->topk_ids, r->topk_w,
                                             L->err_word, s);
        });
        if (st != MOE_OK) return st;
    }
    return run_permute(L, T, r, s);
}

// ---- forward ---------------------------------------------------------------------------
namespace moe {

ExpertArgs make_expert_args(moe_layer_t *L, const void *x, const moe_routing_t *r) {
    ExpertArgs a;
    std::memset(&a, 0, sizeof a);
    a.tab = &L->tab;
    a.x = x;
    a.gather = r->gather_index;
    a.offsets = r->offsets;
    a.topk_w = r->topk_w;
    a.T = r->T;
    a.k = L->cfg.k;
    a.E = L->cfg.E;
    a.m = L->cfg.m;
    a.p = L->cfg.p;
    a.h = L->h;
    a.ypart = L->ypart;
    a.gate_part = L->gate_part;
    a.up_part = L->up_part;
    a.err = L->err_word;
    a.n_only = 0;
    return a;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library does not link the driver library itself).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// 2D bf16 map over a [rows x K] row-major buffer, N x 64 boxes, 128-byte swizzle.
static moe_status_t make_row_map(CUtensorMap *map, void *base, int K, size_t rows, int N) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(N)};
    const cuuint32_t es[2] = {1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
    return MOE_OK;
}

// The resident weight buffer as rows of 128 bytes, 128-row boxes (16 KB): one
// box is one 128-row block of a packed matrix at one reduction block.
static moe_status_t weight_map(moe_layer_t *L, const CUtensorMap **out) {
    if (!L->tmap_w_ok) {
        PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
        if (!enc) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
        const size_t bytes = L->expert_stride * static_cast<size_t>(L->cfg.E);
        const cuuint64_t dims[2] = {64u, static_cast<cuuint64_t>(bytes / 128)};
        const cuuint64_t strides[1] = {128u};
        const cuuint32_t box[2] = {64u, 128u};
        const cuuint32_t es[2] = {1u, 1u};
        const CUresult r = enc(&L->tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, L->weights, dims, strides, box, es,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled(weights) failed (%d)", int(r));
        L->tmap_w_ok = true;
    }
    *out = &L->tmap_w;
    return MOE_OK;
}

static int tc_tile_n(int mean_q) {
    if (mean_q <= 12) return 16;
    if (mean_q <= 24) return 32;
    if (mean_q <= 48) return 64;
    if (mean_q <= 96) return 128;
    return 256;
}

// Token-row maps (x_perm and h) whose boxes are N rows: one pair per width.
static moe_status_t tc_maps(moe_layer_t *L, int N, const CUtensorMap **xm, const CUtensorMap **hm) {
    int idx;
    switch (N) {
    case 16: idx = 0; break;
    case 32: idx = 1; break;
    case 64: idx = 2; break;
    case 128: idx = 3; break;
    case 256: idx = 4; break;
    case 192: idx = 5; break;  // int8 tensor-core tiles
    default: return fail(MOE_ERR_INTERNAL, "no token-row map of width %d", N);
    }
    if (!L->tmap_ok[idx]) {
        const size_t rows = static_cast<size_t>(L->cfg.max_tokens) * L->cfg.k;
        moe_status_t st = make_row_map(&L->tmap_x[idx], L->x_perm, L->cfg.m, rows, N);
        if (st == MOE_OK) st = make_row_map(&L->tmap_h[idx], L->h, L->cfg.p, rows, N);
        if (st != MOE_OK) return st;
        L->tmap_ok[idx] = true;
    }
    *xm = &L->tmap_x[idx];
    *hm = &L->tmap_h[idx];
    return MOE_OK;
}

// Splits of the reduction for tensor-core launches: the smallest count (up to
// max_s and the K-block count) whose tiles fill the SMs in near-whole waves.
static int tc_splits(int nkb, int rows, int N, int mean_q, int n_active, int num_sms, int max_s) {
    const long long ntt = (mean_q + N - 1) / N;
    int best = 1;
    double best_eff = -1.0;
    for (int S = 1; S <= max_s && S <= nkb; ++S) {
        const long long tiles = static_cast<long long>(n_active) * S * (rows / 128) * ntt;
        const long long waves = (tiles + num_sms - 1) / num_sms;
        const double eff = static_cast<double>(tiles) / static_cast<double>(waves * num_sms);
        if (eff >= 0.92) return S;
        if (eff > best_eff) {
            best_eff = eff;
            best = S;
        }
    }
    return best;
}

// The launch plan of the expert MLPs for T tokens (moe_plan_forward states the
// rules): regime, token tiles or passes, reduction splits, CTA pairs.
moe_status_t plan_forward(const moe_config_t &c, const WorkspaceGeom &w, int num_sms, int T, int regime,
                          bool pair_tiles, moe_plan_t *out) {
    moe_plan_t p{};
    p.splits_up = p.splits_down = 1;
    const int rows = T * c.k;
    p.mean_tokens = (rows + c.E - 1) / c.E;
    if (T == 0) {
        p.path = MOE_PATH_NONE;
    } else if (c.act_dtype == MOE_F32) {
        p.path = MOE_PATH_SIMT;
    } else {
        // regime: the weight-streaming GEMV while experts see few tokens, the
        // tensor-core grouped GEMM beyond (rows in 128-row blocks; int8 weights
        // also need K in 128-element blocks, which int8 layers have)
        const bool gated = c.expert == MOE_EXPERT_SWIGLU;
        const bool i8 = c.weight_dtype == MOE_I8;
        const int mean_q = p.mean_tokens;
        const int rows_up = gated ? 2 * c.p : c.p;
        const int bk = i8 ? 128 : 64;  // reduction elements per pipeline stage
        const bool tc_shape = rows_up % 128 == 0 && c.m % 128 == 0 && (!i8 || c.p % 128 == 0);
        const bool fits_decode = static_cast<size_t>(rows) <= w.decode_rows_cap;
        bool use_tc = false;
        if (regime == 2) {
            if (!tc_shape) return fail(MOE_ERR_UNSUPPORTED, "batch kernels need 128-row blocks");
            use_tc = true;
        } else if (regime == 0) {
            const int min_q = i8 ? kTcMinMeanTokensI8 : kTcMinMeanTokens;
            use_tc = tc_shape && (mean_q > min_q || !fits_decode);
        }
        if (use_tc) {
            int N = tc_tile_n(mean_q);
            if (i8 && N > kTcI8MaxN) N = kTcI8MaxN;
            if (fits_decode) {
                const int n_act = expected_active(T, c.k, c.E);
                p.splits_up = tc_splits(c.m / bk, rows_up, N, mean_q, n_act, num_sms, w.split_up_max);
                p.splits_down = tc_splits(c.p / bk, c.m, N, mean_q, n_act, num_sms, w.split_down_max);
            } else if (w.ypart_rows >= 2 * static_cast<size_t>(rows)) {
                // batch: the down projection's tiles (128 output rows x a token
                // tile, the whole reduction of p) can be too few to fill the SMs
                // evenly; it splits the reduction in two where that evens out the
                // waves and the partial-sum workspace has room (measured, Mixtral
                // shape T = 2048: 418 -> 393 us; four splits at T = 512 measured
                // slower than none)
                p.splits_down = tc_splits(c.p / bk, c.m, N, mean_q, c.E, num_sms, 2);
            }
            // The up projection's 256-token tiles run on CTA pairs (less
            // shared-memory traffic per SM; measured faster) for resident
            // weights in 256-row pair blocks with nothing split; the down
            // projection stays on one CTA per tile, which measured faster for it.
            p.pair_up = (!i8 && pair_tiles && !c.paged && N == 256 && p.splits_up == 1 && rows_up % 256 == 0);
            // The down projection streams its weights while experts see a few
            // hundred tokens (HBM-bound): 128-token tiles halve each stage's
            // token fill, so more weight stages fit in flight (Mixtral shape,
            // Zipf 1.2, T = 512: down 256.5 -> 244.5 us).
            p.tile_up = N;
            p.tile_down = (!i8 && N == 256 && mean_q <= 192) ? 128 : N;
            p.path = MOE_PATH_TENSOR;
        } else {
            if (!fits_decode) return fail(MOE_ERR_UNSUPPORTED, "decode kernels take T*k <= %d", kDecodeMaxRows);
            const int nt = decode_token_tiles(T, c.k, c.E);
            const int n_act = expected_active(T, c.k, c.E);
            p.splits_up = choose_splits(c.m, bk, rows_up, nt, n_act, num_sms, w.split_up_max);
            p.splits_down = choose_splits(c.p, bk, c.m, nt, n_act, num_sms, w.split_down_max);
            if (p.splits_up > w.split_up_max || p.splits_down > w.split_down_max)
                return fail(MOE_ERR_INTERNAL, "split count exceeds workspace");
            p.tile_up = p.tile_down = 8 * nt;
            p.path = MOE_PATH_GEMV;
        }
    }
    *out = p;
    return MOE_OK;
}

WorkspaceGeom layer_geom(const moe_layer_t *L) {
    WorkspaceGeom w;
    w.split_up_max = L->split_up_max;
    w.split_down_max = L->split_down_max;
    w.decode_rows_cap = L->decode_rows_cap;
    w.ypart_rows = L->ypart_rows;
    return w;
}

// Tensor-core path: gather the token rows into expert order, then the grouped
// GEMMs (up with the activation fused, down with the routing weight fused).
static moe_status_t run_experts_tc(moe_layer_t *L, ExpertArgs &a, const moe_plan_t &plan, int *splits_out,
                                   cudaStream_t s) {
    const moe_config_t &c = L->cfg;
    const bool gated = c.expert == MOE_EXPERT_SWIGLU;
    const int rows = a.T * a.k;
    const bool i8 = c.weight_dtype == MOE_I8;
    const int N = plan.tile_up, N_down = plan.tile_down;
    const int s_up = plan.splits_up, s_down = plan.splits_down;
    const bool pair_up = plan.pair_up != 0;
    a.n_rows_cap = static_cast<size_t>(rows) <= L->decode_rows_cap ? static_cast<int>(L->decode_rows_cap) : rows;
    // batch regime (more rows than the decode cap): the down projection's
    // output rows go to the combine rounded to bf16, halving their write and
    // read; decode-sized calls keep fp32 partial sums
    a.ypart_bf16 = (c.act_dtype == MOE_BF16 && static_cast<size_t>(rows) > L->decode_rows_cap) ? 1 : 0;
    const CUtensorMap *xm = nullptr, *hm = nullptr, *xm_half = nullptr, *hm_half = nullptr;
    moe_status_t st = tc_maps(L, N, &xm, &hm);
    if (st == MOE_OK && pair_up) st = tc_maps(L, N / 2, &xm_half, &hm_half);
    if (st != MOE_OK) return st;
    if (i8) {  // fp16 token rows, their scales and split sums (the up projection's MMAs run in fp16)
        a.x_scale = L->x_scale;
        a.x_sum = L->x_sum;
        a.xsum_stride = static_cast<int>(static_cast<size_t>(c.max_tokens) * c.k);
        st = launch_phase(L, MOE_PHASE_GATHER, s, "gather_rows_f16", [&] {
            return launch_gather_rows_f16(a.x, a.gather, rows, a.k, c.m, s_up, L->x_perm, L->x_scale, L->x_sum,
                                          a.xsum_stride, L->err_word, s);
        });
    } else {
        st = launch_phase(L, MOE_PHASE_GATHER, s, "gather_rows", [&] {
            return launch_gather_rows(a.x, a.gather, rows, a.k, c.m, L->x_perm, L->err_word, s);
        });
    }
    if (pair_up) {
        const CUtensorMap *wm = nullptr;
        if (st == MOE_OK) st = weight_map(L, &wm);
        a.wbase = L->weights;
        if (st == MOE_OK)
            st = launch_phase(L, MOE_PHASE_UP, s, "tc2_up",
                              [&] { return launch_tc2_up(a, gated, *wm, *xm_half, L->num_sms, s); });
    } else if (st == MOE_OK) {
        st = launch_phase(L, MOE_PHASE_UP, s, "tc_up", [&] {
            return i8 ? launch_tc_i8_up(a, gated, s_up, N, *xm, L->num_sms, s)
                      : launch_tc_up(a, gated, s_up, N, *xm, L->num_sms, s);
        });
    }
    if (st == MOE_OK && s_up > 1)
        st = launch_phase(L, MOE_PHASE_UP_FINISH, s, "up_finish",
                          [&] { return launch_decode_up_finish(a, gated, s_up, s); });
    const CUtensorMap *hm_down = hm;
    if (st == MOE_OK && N_down != N) {
        const CUtensorMap *unused = nullptr;
        st = tc_maps(L, N_down, &unused, &hm_down);
    }
    if (st == MOE_OK)
        st = launch_phase(L, MOE_PHASE_DOWN, s, "tc_down", [&] {
            return i8 ? launch_tc_i8_down(a, s_down, N_down, *hm_down, L->num_sms, s)
                      : launch_tc_down(a, s_down, N_down, *hm_down, L->num_sms, s);
        });
    *splits_out = s_down;
    return st;
}

// Expert MLPs for the experts of `a` (all with tokens, or a.only) into ypart;
// returns the number of ypart splits written.
moe_status_t run_experts(moe_layer_t *L, ExpertArgs &a, int regime, int *splits_out,
                         cudaStream_t s) {
    const moe_config_t &c = L->cfg;
    const bool gated = c.expert == MOE_EXPERT_SWIGLU;
    moe_plan_t plan;
    moe_status_t plan_st = plan_forward(c, layer_geom(L), L->num_sms, a.T, regime, L->pair_tiles, &plan);
    if (plan_st != MOE_OK) return plan_st;
    *splits_out = 1;
    if (plan.path == MOE_PATH_NONE) return MOE_OK;
    if (plan.path == MOE_PATH_SIMT) {
        a.n_rows_cap = a.T * a.k;
        moe_status_t st = launch_phase(L, MOE_PHASE_UP, s, "simt_up", [&] { return launch_simt_up(a, gated, s); });
        if (st == MOE_OK)
            st = launch_phase(L, MOE_PHASE_DOWN, s, "simt_down", [&] { return launch_simt_down(a, s); });
        return st;
    }
    if (plan.path == MOE_PATH_TENSOR) {
        L->stats.tc_runs += 1;
        return run_experts_tc(L, a, plan, splits_out, s);
    }
    L->stats.gemv_runs += 1;
    const WeightType wt = (c.weight_dtype == MOE_I8) ? WeightType::kI8 : WeightType::kBF16;
    const int s_up = plan.splits_up, s_down = plan.splits_down;
    a.n_rows_cap = static_cast<int>(L->decode_rows_cap);
    moe_status_t st = launch_phase(L, MOE_PHASE_UP, s, "decode_up",
                                   [&] { return launch_decode_up(a, wt, gated, s_up, L->num_sms, s); });
    if (st == MOE_OK && s_up > 1)
        st = launch_phase(L, MOE_PHASE_UP_FINISH, s, "decode_up_finish",
                          [&] { return launch_decode_up_finish(a, gated, s_up, s); });
    if (st == MOE_OK)
        st = launch_phase(L, MOE_PHASE_DOWN, s, "decode_down",
                          [&] { return launch_decode_down(a, wt, s_down, L->num_sms, s); });
    *splits_out = s_down;
    return st;
}

moe_status_t run_combine(moe_layer_t *L, const moe_routing_t *r, int splits, int n_rows_cap,
                         bool part_bf16, void *y, cudaStream_t s) {
    CombineArgs ca{L->ypart, splits, static_cast<size_t>(n_rows_cap) * L->cfg.m, r->scatter_index,
                   r->T, L->cfg.k, L->cfg.m, y, L->err_word, part_bf16};
    return launch_phase(L, MOE_PHASE_COMBINE, s, "combine",
                        [&] { return launch_combine(ca, L->cfg.act_dtype == MOE_BF16, s); });
}

}  // namespace moe

extern "C" moe_status_t moe_forward(moe_layer_t *L, const void *x, const moe_routing_t *r,
                                    void *y, void *stream) {
    NvtxRange range("moe_forward");
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    moe_status_t st = check_routing(L, r);
    if (st != MOE_OK) return st;
    st = check_T(L, r->T);
    if (st != MOE_OK) return st;
    if (r->T == 0) return MOE_OK;
    if (!x || !y || !aligned16(x) || !aligned16(y))
        return fail(MOE_ERR_INVALID_ARG, "x or y is NULL or not 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (L->pool) return paged_forward(L, x, r, y, s);
    ExpertArgs a = make_expert_args(L, x, r);
    int splits = 1;
    st = run_experts(L, a, L->regime, &splits, s);
    if (st != MOE_OK) return st;
    st = run_combine(L, r, splits, a.n_rows_cap, a.ypart_bf16 != 0, y, s);
    if (st != MOE_OK) return st;
    L->last_stream = s;
    L->launched = true;
    return MOE_OK;
}

extern "C" moe_status_t moe_plan_forward(const moe_config_t *cfg, int T, int num_sms, int regime,
                                         int pair_tiles, moe_plan_t *out) {
    if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
    moe_status_t st = check_config(cfg);
    if (st != MOE_OK) return st;
    if (T < 0 || T > cfg->max_tokens)
        return fail(MOE_ERR_INVALID_ARG, "T = %d outside [0, max_tokens = %d]", T, cfg->max_tokens);
    if (num_sms < 1) return fail(MOE_ERR_INVALID_ARG, "num_sms must be >= 1");
    if (regime < 0 || regime > 2) return fail(MOE_ERR_INVALID_ARG, "regime must be 0, 1 or 2");
    if (pair_tiles != 0 && pair_tiles != 1) return fail(MOE_ERR_INVALID_ARG, "pair_tiles must be 0 or 1");
    return plan_forward(*cfg, workspace_geom(*cfg), num_sms, T, regime, pair_tiles != 0, out);
}

// ---- options, info, stats, checks ----------------------------------------------------
extern "C" moe_status_t moe_layer_set_option(moe_layer_t *L, moe_option_t opt, int value) {
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    if (opt == MOE_OPT_REGIME) {
        if (value < 0 || value > 2) return fail(MOE_ERR_INVALID_ARG, "regime must be 0, 1 or 2");
        L->regime = value;
        return MOE_OK;
    }
    if (opt == MOE_OPT_TIMING) {
        if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "timing must be 0 or 1");
        L->timing = value != 0;
        return MOE_OK;
    }
    if (opt == MOE_OPT_PAIR_TILES) {
        if (value != 0 && value != 1) return fail(MOE_ERR_INVALID_ARG, "pair tiles must be 0 or 1");
        L->pair_tiles = value != 0;
        return MOE_OK;
    }
    if (opt == MOE_OPT_HOST_TIMEOUT_MS) {
        if (value < -1) return fail(MOE_ERR_INVALID_ARG, "host timeout must be >= 0 ms, or -1");
        L->host_timeout_ms = value;
        return MOE_OK;
    }
    return fail(MOE_ERR_INVALID_ARG, "unknown option %d", int(opt));
}

extern "C" moe_status_t moe_layer_timings(moe_layer_t *L, moe_timings_t *out, int reset) {
    if (!L || !out) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    cudaSetDevice(L->device);
    for (auto &pe : L->pending) {
        CUDA_TRY(cudaEventSynchronize(pe.b));
        float ms = 0.0f;
        CUDA_TRY(cudaEventElapsedTime(&ms, pe.a, pe.b));
        L->phase_ms[pe.phase] += ms;
        L->phase_launches[pe.phase] += 1;
        if (pe.phase == MOE_PHASE_COPY) L->stats.h2d_ms += ms;
        L->event_pool.push_back(pe.a);
        L->event_pool.push_back(pe.b);
    }
    L->pending.clear();
    for (int i = 0; i < MOE_NUM_PHASES; ++i) {
        out->ms[i] = L->phase_ms[i];
        out->launches[i] = L->phase_launches[i];
        if (reset) {
            L->phase_ms[i] = 0.0;
            L->phase_launches[i] = 0;
        }
    }
    return MOE_OK;
}

extern "C" moe_status_t moe_layer_info(const moe_layer_t *L, moe_layer_info_t *out) {
    if (!L || !out) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    std::memset(out, 0, sizeof *out);
    out->expert_bytes = L->expert_bytes;
    out->weight_bytes = L->expert_bytes * L->cfg.E;
    out->workspace_bytes = L->workspace_bytes;
    out->decode_splits_up = L->split_up_max;
    out->decode_splits_down = L->split_down_max;
    out->num_sms = L->num_sms;
    return MOE_OK;
}

extern "C" moe_status_t moe_layer_stats(moe_layer_t *L, moe_stats_t *out) {
    if (!L || !out) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    if (L->fwd_pending) {  // duration of the last paged forward
        cudaSetDevice(L->device);
        const moe_status_t w = wait_event(L->fwd_t1, L->host_timeout_ms, "the last paged call");
        if (w != MOE_OK) return w;
        float ms = 0.0f;
        CUDA_TRY(cudaEventElapsedTime(&ms, L->fwd_t0, L->fwd_t1));
        L->stats.forward_ms += ms;
        L->fwd_pending = false;
    }
    *out = L->stats;
    return MOE_OK;
}

extern "C" moe_status_t moe_layer_sync_check(moe_layer_t *L, int timeout_ms, uint32_t *flags) {
    if (!L) return fail(MOE_ERR_INVALID_ARG, "layer is NULL");
    if (flags) *flags = 0;
    cudaSetDevice(L->device);
    if (L->launched) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        CUDA_TRY(cudaStreamIsCapturing(L->last_stream, &cs));
        if (cs != cudaStreamCaptureStatusNone)
            return fail(MOE_ERR_INVALID_ARG, "the layer's last stream is being captured into a graph");
        CUDA_TRY(cudaEventRecord(L->done, L->last_stream));
    }
    const moe_status_t w = wait_event(L->done, timeout_ms, "layer work");
    if (w != MOE_OK) return w;
    uint32_t word = 0;
    CUDA_TRY(cudaMemcpy(&word, L->err_word, 4, cudaMemcpyDeviceToHost));
    if (word) {
        CUDA_TRY(cudaMemset(L->err_word, 0, 4));
        if (flags) *flags = word;
        if (word & MOE_FLAG_WAIT_TIMEOUT)
            return fail(MOE_ERR_TIMEOUT, "a bounded device wait gave up (bits 0x%x)", word);
        return fail(MOE_ERR_INVALID_ARG, "device flagged bad routing data (bits 0x%x)", word);
    }
    return MOE_OK;
}

extern "C" moe_status_t moe_layer_read_expert(const moe_layer_t *L, int expert, int which,
                                              void *values, float *scales) {
    if (!L || !values) return fail(MOE_ERR_INVALID_ARG, "NULL argument");
    const moe_config_t &c = L->cfg;
    if (expert < 0 || expert >= c.E) return fail(MOE_ERR_INVALID_ARG, "expert out of range");
    const bool gated = c.expert == MOE_EXPERT_SWIGLU;
    if (which < 1 || which > 3 || (which == 3 && !gated))
        return fail(MOE_ERR_INVALID_ARG, "which must be 1, 2 or (SwiGLU) 3");
    if (c.weight_dtype == MOE_I8 && !scales) return fail(MOE_ERR_INVALID_ARG, "scales is NULL");
    if (L->pool) return fail(MOE_ERR_UNSUPPORTED, "read_expert on a paged layer");
    cudaSetDevice(L->device);
    CUDA_TRY(cudaDeviceSynchronize());
    // user orientation: W1/W3 are m x p (out = columns = p), W2 is p x m
    const int out_n = (which == 2) ? c.m : c.p, red = (which == 2) ? c.p : c.m;
    uint8_t *dst = static_cast<uint8_t *>(values);
    if (c.weight_dtype == MOE_F32) {
        const void *src = which == 1 ? L->tab.w1[expert] : which == 2 ? L->tab.w2[expert] : L->tab.w3[expert];
        std::vector<float> buf(static_cast<size_t>(out_n) * red);
        CUDA_TRY(cudaMemcpy(buf.data(), src, buf.size() * 4, cudaMemcpyDeviceToHost));
        float *o = reinterpret_cast<float *>(dst);
        for (int n = 0; n < out_n; ++n)
            for (int i = 0; i < red; ++i) o[static_cast<size_t>(i) * out_n + n] = buf[static_cast<size_t>(n) * red + i];
        return MOE_OK;
    }
    const int el = (c.weight_dtype == MOE_I8) ? 1 : 2;
    const int rows = (which == 2) ? c.m : (gated ? 2 * c.p : c.p);
    const void *src = (which == 2) ? L->tab.w2[expert] : L->tab.w1[expert];
    std::vector<uint8_t> buf(static_cast<size_t>(rows) * red * el);
    CUDA_TRY(cudaMemcpy(buf.data(), src, buf.size(), cudaMemcpyDeviceToHost));
    for (int n = 0; n < out_n; ++n) {
        const int row = (which == 2) ? n : (!gated ? n : (which == 1 ? up_row_gate(n) : up_row_up(n)));
        for (int i = 0; i < red; ++i)
            std::memcpy(dst + (static_cast<size_t>(i) * out_n + n) * el,
                        buf.data() + packed_offset(row, i, rows, el), el);
    }
    if (c.weight_dtype == MOE_I8) {
        const float *ssrc = which == 1 ? L->tab.s1[expert] : which == 2 ? L->tab.s2[expert] : L->tab.s3[expert];
        CUDA_TRY(cudaMemcpy(scales, ssrc, static_cast<size_t>(out_n) * 4, cudaMemcpyDeviceToHost));
    }
    return MOE_OK;
}

extern "C" const char *moe_status_string(moe_status_t s) {
    switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_OOM: return "out of memory";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "timeout";
    case MOE_ERR_INTERNAL: return "internal error";
    }
    return "unknown status";
}

extern "C" const char *moe_last_error(void) { return g_last_error.c_str(); }

extern "C" int moe_version(void) { return 100; }
