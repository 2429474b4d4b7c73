// paged.cu -- paged expert weights: a fixed GPU budget of expert slots,
// arranged as N sets (indices) x M ways, shared by every layer of a model
// (expert-cache article, section 2.2: S = floor(available / expert size)
// slots, N = floor(S / M) sets, layer l uses set l mod N, LRU inside a set).
#include <cstring>

#include "../../include/moe_layer.h"
#include "kernels.cuh"
#include "layer_impl.h"

using namespace moe;

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
    (void)budget_bytes;
    (void)expert_bytes;
    (void)ways;
    (void)page_bytes;
    if (out) *out = nullptr;
    return fail(MOE_ERR_UNSUPPORTED, "paged pools are not built yet");
}

extern "C" moe_status_t moe_pool_destroy(moe_pool_t *pool) {
    (void)pool;
    return MOE_OK;
}

moe_status_t paged_attach(moe_layer *L) {
    (void)L;
    return fail(MOE_ERR_UNSUPPORTED, "paged layers are not built yet");
}

void paged_detach(moe_layer *L) { (void)L; }

moe_status_t paged_forward(moe_layer *L, const void *x, const moe_routing_t *r, void *y,
                           cudaStream_t s) {
    (void)L;
    (void)x;
    (void)r;
    (void)y;
    (void)s;
    return fail(MOE_ERR_UNSUPPORTED, "paged layers are not built yet");
}
