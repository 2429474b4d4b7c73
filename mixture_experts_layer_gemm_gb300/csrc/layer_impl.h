// layer_impl.h -- the layer object behind the opaque moe_layer_t handle.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <vector>

#include "../../include/moe_layer.h"
#include "kernels.cuh"

struct moe_layer {
    moe_config_t cfg{};
    int layer_id = 0;
    int device = -1;
    int num_sms = 0;
    int regime = 0;  // MOE_OPT_REGIME
    bool pair_tiles = true;  // MOE_OPT_PAIR_TILES
    int host_timeout_ms = 120000;  // MOE_OPT_HOST_TIMEOUT_MS (-1: no limit)
    size_t ypart_rows = 0;  // fp32 partial rows the down projection's workspace holds
    int32_t *cta_count = nullptr;  // router permute: per-CTA expert counts

    // weights (resident copy, or unused for paged layers)
    float *wrt = nullptr;      // router [E x m] fp32
    void *wra = nullptr;       // router [E x m] in the activation type
    float *bias = nullptr;     // [E] fp32
    uint8_t *weights = nullptr;
    size_t expert_stride = 0;  // bytes between experts inside `weights`
    size_t expert_bytes = 0;   // bytes of one expert's stored weights (no padding)
    moe::ExpertTables tab{};

    // workspace
    void *h = nullptr;
    void *x_perm = nullptr;  // [max_tokens*k x m] bf16: token rows in expert order (tensor-core path)
    // tensor maps over x_perm and h for token tiles N = 16, 32, 64, 128, 256
    bool tmap_ok[6] = {};
    CUtensorMap tmap_x[6], tmap_h[6];  // token-row maps, boxes of 16, 32, 64, 128, 256, 192 rows
    bool tmap_w_ok = false;  // the resident weights as 128-byte rows (CTA-pair kernels)
    CUtensorMap tmap_w;
    float *ypart = nullptr;
    float *gate_part = nullptr, *up_part = nullptr;
    // int8 layers: per permuted row, the fp16 token rows' power-of-two scale and
    // their sums per up-projection reduction split ([split_up_max x rows])
    float *x_scale = nullptr, *x_sum = nullptr;
    size_t decode_rows_cap = 0;
    int split_up_max = 1, split_down_max = 1;
    size_t workspace_bytes = 0;
    uint32_t *err_word = nullptr;
    unsigned *ticket = nullptr;  // fused-permute completion counter (0 between launches)

    // paged weights
    moe_pool_t *pool = nullptr;
    uint8_t *pinned_weights = nullptr;  // E experts x expert_stride, pinned host
    int32_t *counts_host = nullptr;     // pinned copy of the routing counts
    cudaEvent_t fwd_t0 = nullptr, fwd_t1 = nullptr;  // bracket a paged forward
    cudaEvent_t counts_ready = nullptr;              // paged forward: token counts on the host
    bool fwd_pending = false;

    moe_stats_t stats{};
    // per-launch event timing (MOE_OPT_TIMING)
    struct Pending {
        int phase;
        cudaEvent_t a, b;
    };
    bool timing = false;
    std::vector<cudaEvent_t> event_pool;
    std::vector<Pending> pending;
    double phase_ms[MOE_NUM_PHASES] = {};
    uint64_t phase_launches[MOE_NUM_PHASES] = {};
    cudaEvent_t get_event();

    cudaEvent_t done = nullptr;
    // Stream of the last route or forward call.  No event is recorded per call:
    // an event between two launches would end the programmatic-launch overlap
    // of the last kernel of one call with the first of the next.
    // moe_layer_sync_check records `done` on this stream when it is called.
    cudaStream_t last_stream = nullptr;
    // The stream and the counts of the last routing call, until a forward call
    // consumes them: a paged forward reads the token counts on the routing
    // call's stream, so a caller that routes ahead on a side stream does not
    // make that read wait for the compute queued on the forward's stream.
    cudaStream_t route_stream = nullptr;
    const int32_t *route_counts = nullptr;
    bool launched = false;
    cudaStream_t ingest_stream = nullptr;
    std::vector<void *> allocations;

    ~moe_layer();
    void *dalloc(size_t bytes, cudaError_t *err);
};

namespace moe {
moe_status_t fail(moe_status_t st, const char *fmt, ...);
moe_status_t cuda_fail(cudaError_t e, const char *where);
// Host wait for an event with a deadline: polls the event (yielding, then
// sleeping 20 us between polls), so that device work that does not finish
// becomes MOE_ERR_TIMEOUT instead of a caller blocked for good.
// timeout_ms < 0: no limit.
moe_status_t wait_event(cudaEvent_t ev, int timeout_ms, const char *what);

ExpertArgs make_expert_args(moe_layer *L, const void *x, const moe_routing_t *r);
moe_status_t run_experts(moe_layer *L, ExpertArgs &a, int regime, int *splits_out, cudaStream_t s);
moe_status_t run_combine(moe_layer *L, const moe_routing_t *r, int splits, int n_rows_cap, bool part_bf16, void *y,
                         cudaStream_t s);

// Workspace a layer of configuration c allocates at create time, and to which
// its launch plans are cut.
struct WorkspaceGeom {
    int split_up_max = 1, split_down_max = 1;  // reduction splits the partial-sum buffers hold
    size_t decode_rows_cap = 0;                // largest T*k of the split (decode-sized) forms
    size_t ypart_rows = 0;                     // fp32 rows of the down projection's output
};
WorkspaceGeom workspace_geom(const moe_config_t &c);
WorkspaceGeom layer_geom(const moe_layer *L);  // the workspace this layer allocated
// The launch plan of the expert MLPs for T tokens (the rules moe_plan_forward
// states); MOE_ERR_UNSUPPORTED where a forced regime cannot run.
moe_status_t plan_forward(const moe_config_t &c, const WorkspaceGeom &w, int num_sms, int T, int regime,
                          bool pair_tiles, moe_plan_t *out);

// Launch one kernel (f returns its cudaError_t) as phase `phase`: counts the
// launch and, with timing on, brackets it with events on stream s.
// A named range on the host timeline of profilers (NVTX; no cost without one).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

template <typename F>
moe_status_t launch_phase(moe_layer *L, int phase, cudaStream_t s, const char *what, F &&f) {
    NvtxRange range(what);
    cudaEvent_t a = nullptr;
    if (L->timing) {
        a = L->get_event();
        if (a) cudaEventRecord(a, s);
    }
    const cudaError_t e = f();
    if (e != cudaSuccess) {
        if (a) L->event_pool.push_back(a);
        return cuda_fail(e, what);
    }
    if (a) {
        cudaEvent_t b = L->get_event();
        if (b) {
            cudaEventRecord(b, s);
            L->pending.push_back({phase, a, b});
        } else {
            L->event_pool.push_back(a);
        }
    }
    L->stats.kernel_launches += 1;
    return MOE_OK;
}
}  // namespace moe

// paged.cu
moe_status_t paged_attach(moe_layer *L);
void paged_detach(moe_layer *L);
moe_status_t paged_forward(moe_layer *L, const void *x, const moe_routing_t *r, void *y,
                           cudaStream_t s);
