// selftest.cu -- the device-side wait limit, exercised without a fault.
//
// Every wait in the library's kernels polls an mbarrier a bounded number of
// times; if the phase has not completed by then, the kernel sets the
// wait-timeout bit of its error word, lets go of what it holds and returns, so
// that a lost signal (a bug) ends as a status the host reads while the CUDA
// context stays usable.  This kernel waits, with the same polling primitive,
// on a phase that nothing completes, so its wait always runs out.
#include <cstdint>

#include "../../include/moe_layer.h"
#include "common.cuh"
#include "layer_impl.h"

static_assert(moe::kErrExpertId == MOE_FLAG_EXPERT_ID && moe::kErrDuplicateId == MOE_FLAG_DUPLICATE_ID &&
                  moe::kErrGatherIndex == MOE_FLAG_GATHER_INDEX && moe::kErrOffsets == MOE_FLAG_OFFSETS &&
                  moe::kErrWaitTimeout == MOE_FLAG_WAIT_TIMEOUT && moe::kErrTmemAlloc == MOE_FLAG_TMEM_ALLOC,
              "device error bits and the public flags must agree");

namespace {

__global__ void wait_never_kernel(uint32_t polls, uint32_t *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        moe::mbar_init(&bar, 1);  // one arrival expected; none comes
        moe::fence_barrier_init();
    }
    __syncthreads();
    bool done = false;
    for (uint32_t i = 0; i < polls && !done; ++i) done = moe::mbar_try_wait(&bar, 0);
    if (!__all_sync(0xffffffffu, done) && (threadIdx.x & 31) == 0) moe::flag_error(err, moe::kErrWaitTimeout);
}

}  // namespace

extern "C" moe_status_t moe_selftest_bounded_wait(uint32_t polls, uint32_t *flags, void *stream) {
    if (flags) *flags = 0;
    if (polls < 1 || polls > (1u << 24)) return moe::fail(MOE_ERR_INVALID_ARG, "polls must be in [1, 2^24]");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t *err = nullptr;
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void **>(&err), sizeof(uint32_t), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(uint32_t), s);
    if (e == cudaSuccess) {
        wait_never_kernel<<<1, 64, 0, s>>>(polls, err);
        e = cudaGetLastError();
    }
    uint32_t word = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&word, err, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
    if (err) {
        const cudaError_t f = cudaFreeAsync(err, s);
        if (e == cudaSuccess) e = f;
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return moe::cuda_fail(e, "moe_selftest_bounded_wait");
    if (flags) *flags = word;
    if (word & MOE_FLAG_WAIT_TIMEOUT) return moe::fail(MOE_ERR_TIMEOUT, "the bounded wait gave up after %u polls", polls);
    return moe::fail(MOE_ERR_INTERNAL, "the wait completed although nothing arrived");
}
