// noalloc.cu -- moe_forward_static_scratch: the decode-regime forward pass
// with its scratch memory in a fixed array compiled into this library, for
// callers that must not allocate device memory while they run.
//
// Who needs it: a serving engine that hands all free device memory to its own
// allocator (so a cudaMalloc could fail or fragment that pool), a latency-
// critical loop that cannot afford cudaMalloc's implicit device
// synchronisation, or code that runs where allocation is not permitted.  Such
// a caller creates the layer once, up front, and then runs every forward pass
// through this entry point, which calls no cudaMalloc, cudaFree or other
// allocating routine.
//
// The scratch (the expert hidden activations and the split-reduction
// partial sums of the down projection, plus those of the up projection when it
// is split) lives in g_static_scratch below: kStaticScratchBytes per GPU that
// loads the library, held until the process exits.  A request that needs more
// is rejected with MOE_ERR_INVALID_ARG and a message giving both sizes.
//
// The kernels are the same ones moe_forward runs in the decode regime, with
// the same launch plan, so the results are the same.  Every scratch element a
// call reads is written earlier in that call, so nothing needs clearing.
//
// All calls on one device share the one array: two calls whose work overlaps
// on the GPU (different streams, or different host threads) race on it.
// Serialise them, e.g. by issuing them on one stream.
//
// Set-up: the first call on each device looks up the device address of the
// array (cudaGetSymbolAddress) with that device current; later calls reuse
// it.  Make that first call before any stream capture begins.  A call must be
// made with the layer's device current (else MOE_ERR_INVALID_ARG).  The
// cached address belongs to the device's primary context: after a context
// reset (cudaDeviceReset) the library must be unloaded and loaded again.
#include <mutex>

#include "../../include/moe_layer.h"
#include "common.cuh"
#include "kernels.cuh"
#include "layer_impl.h"

using namespace moe;

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// Device address of the scratch array on the layer's device (set-up once per
// device).  The symbol lookup answers for the current device, so a call made
// with another device current is refused rather than handed an address of the
// wrong GPU's copy.
moe_status_t scratch_address(int layer_device, void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != layer_device)
        return fail(MOE_ERR_INVALID_ARG, "current device %d is not the layer's device %d", dev,
                    layer_device);
    if (dev < 0 || dev >= kMaxDevices) return fail(MOE_ERR_UNSUPPORTED, "device index %d", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_forward_static_scratch(moe_layer_t *L, const void *x,
                                                   const moe_routing_t *r, void *y, void *stream) {
    if (!L || !r) return fail(MOE_ERR_INVALID_ARG, "layer or routing is NULL");
    const moe_config_t &c = L->cfg;
    if (c.act_dtype != MOE_BF16 || c.paged)
        return fail(MOE_ERR_UNSUPPORTED, "static-scratch forward needs a resident bf16/int8 layer");
    if (r->T < 0 || r->T > c.max_tokens)
        return fail(MOE_ERR_INVALID_ARG, "T = %d outside [0, max_tokens = %d]", r->T, c.max_tokens);
    if (!r->topk_w || !r->offsets || !r->gather_index || !r->scatter_index)
        return fail(MOE_ERR_INVALID_ARG, "a routing table pointer is NULL");
    if (r->T == 0) return MOE_OK;
    if (!x || !y || (reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(y) & 15u))
        return fail(MOE_ERR_INVALID_ARG, "x or y is NULL or not 16-byte aligned");
    const int rows = r->T * c.k;
    if (static_cast<size_t>(rows) > L->decode_rows_cap)
        return fail(MOE_ERR_INVALID_ARG, "T*k = %d exceeds the decode limit %zu", rows,
                    L->decode_rows_cap);

    // the decode regime's plan, as moe_forward would take it
    moe_plan_t plan;
    moe_status_t st = plan_forward(c, layer_geom(L), L->num_sms, r->T, 1, false, &plan);
    if (st != MOE_OK) return st;
    const int s_up = plan.splits_up, s_down = plan.splits_down;
    const size_t h_bytes = round256(static_cast<size_t>(rows) * c.p * 2);
    const size_t y_bytes = round256(static_cast<size_t>(s_down) * rows * c.m * 4);
    const size_t part_bytes = (s_up > 1) ? round256(static_cast<size_t>(s_up) * rows * c.p * 4) : 0;
    const size_t need = h_bytes + y_bytes + 2 * part_bytes;
    if (need > kStaticScratchBytes)
        return fail(MOE_ERR_INVALID_ARG,
                    "T = %d needs %zu bytes of scratch; the static scratch holds %zu bytes",
                    r->T, need, kStaticScratchBytes);

    void *base = nullptr;
    st = scratch_address(L->device, &base);
    if (st != MOE_OK) return st;
    uint8_t *b = static_cast<uint8_t *>(base);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ExpertArgs a = make_expert_args(L, x, r);
    a.h = b;
    a.ypart = reinterpret_cast<float *>(b + h_bytes);
    a.gate_part = s_up > 1 ? reinterpret_cast<float *>(b + h_bytes + y_bytes) : nullptr;
    a.up_part = s_up > 1 ? reinterpret_cast<float *>(b + h_bytes + y_bytes + part_bytes) : nullptr;
    a.n_rows_cap = rows;
    const bool gated = c.expert == MOE_EXPERT_SWIGLU;
    const WeightType wt = (c.weight_dtype == MOE_I8) ? WeightType::kI8 : WeightType::kBF16;
    L->stats.gemv_runs += 1;
    st = launch_phase(L, MOE_PHASE_UP, s, "decode_up",
                      [&] { return launch_decode_up(a, wt, gated, s_up, L->num_sms, s); });
    if (st == MOE_OK && s_up > 1)
        st = launch_phase(L, MOE_PHASE_UP_FINISH, s, "decode_up_finish",
                          [&] { return launch_decode_up_finish(a, gated, s_up, s); });
    if (st == MOE_OK)
        st = launch_phase(L, MOE_PHASE_DOWN, s, "decode_down",
                          [&] { return launch_decode_down(a, wt, s_down, L->num_sms, s); });
    if (st != MOE_OK) return st;
    CombineArgs ca{a.ypart, s_down, static_cast<size_t>(rows) * c.m, r->scatter_index, r->T, c.k, c.m,
                   y, L->err_word, false};
    st = launch_phase(L, MOE_PHASE_COMBINE, s, "combine",
                      [&] { return launch_combine(ca, true, s); });
    if (st != MOE_OK) return st;
    L->last_stream = s;
    L->launched = true;
    return MOE_OK;
}
