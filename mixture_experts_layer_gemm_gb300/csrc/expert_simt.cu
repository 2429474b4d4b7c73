// expert_simt.cu -- fp32 expert MLP on CUDA cores (fp32 weights and
// activations; no TF32).  One warp computes one output: lanes take strided
// slices of the reduction and a warp-shuffle tree adds them (the register-level
// reduction of SBI-GeMM, DeepSpeed-Inference article, part 3.2).  Used for the
// fp32 layers, whose sizes are small; correctness, not speed, is its purpose.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

// Expert owning permuted position pos (offsets are monotone), or -1.
__device__ __forceinline__ int expert_of(const int32_t *offsets, int E, int pos) {
    for (int e = 0; e < E; ++e)
        if (pos >= offsets[e] && pos < offsets[e + 1]) return e;
    return -1;
}

template <bool GATED>
__global__ void __launch_bounds__(256) simt_up_kernel(const ExpertTables tab, const ExpertArgs a) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const long long wid = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
    const int rows = a.T * a.k;
    if (wid >= static_cast<long long>(rows) * a.p) return;
    const int pos = static_cast<int>(wid / a.p), n = static_cast<int>(wid % a.p);
    const int e = expert_of(a.offsets, a.E, pos);
    const int fi = a.gather[pos];
    if (e < 0 || fi < 0 || fi >= rows) {
        if (lane == 0) flag_error(a.err, e < 0 ? kErrOffsets : kErrGatherIndex);
        return;
    }
    const float *x = static_cast<const float *>(a.x) + static_cast<size_t>(fi / a.k) * a.m;
    const float *w1 = static_cast<const float *>(tab.w1[e]) + static_cast<size_t>(n) * a.m;
    const float *w3 = GATED ? static_cast<const float *>(tab.w3[e]) + static_cast<size_t>(n) * a.m
                            : nullptr;
    float g = 0.0f, u = 0.0f;
    for (int c = lane; c < a.m; c += 32) {
        const float xv = x[c];
        g = fmaf(xv, w1[c], g);
        if (GATED) u = fmaf(xv, w3[c], u);
    }
    g = warp_sum(g);
    if (GATED) u = warp_sum(u);
    if (lane == 0) {
        const float hv = GATED ? silu(g) * u : fmaxf(g, 0.0f);
        static_cast<float *>(a.h)[static_cast<size_t>(pos) * a.p + n] = hv;
    }
}

__global__ void __launch_bounds__(256) simt_down_kernel(const ExpertTables tab, const ExpertArgs a) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const long long wid = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
    const int rows = a.T * a.k;
    if (wid >= static_cast<long long>(rows) * a.m) return;
    const int pos = static_cast<int>(wid / a.m), r = static_cast<int>(wid % a.m);
    const int e = expert_of(a.offsets, a.E, pos);
    const int fi = a.gather[pos];
    if (e < 0 || fi < 0 || fi >= rows) {
        if (lane == 0) flag_error(a.err, e < 0 ? kErrOffsets : kErrGatherIndex);
        return;
    }
    const float *h = static_cast<const float *>(a.h) + static_cast<size_t>(pos) * a.p;
    const float *w2 = static_cast<const float *>(tab.w2[e]) + static_cast<size_t>(r) * a.p;
    float v = 0.0f;
    for (int c = lane; c < a.p; c += 32) v = fmaf(h[c], w2[c], v);
    v = warp_sum(v);
    if (lane == 0) a.ypart[static_cast<size_t>(pos) * a.m + r] = a.topk_w[fi] * v;
}

}  // namespace

cudaError_t launch_simt_up(const ExpertArgs &a, bool gated, cudaStream_t s) {
    const long long warps = static_cast<long long>(a.T) * a.k * a.p;
    if (warps == 0) return cudaSuccess;
    const long long blocks = (warps * 32 + 255) / 256;
    if (gated)
        return launch_pdl(simt_up_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, *a.tab, a);
    else
        return launch_pdl(simt_up_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, *a.tab, a);
}

cudaError_t launch_simt_down(const ExpertArgs &a, cudaStream_t s) {
    const long long warps = static_cast<long long>(a.T) * a.k * a.m;
    if (warps == 0) return cudaSuccess;
    const long long blocks = (warps * 32 + 255) / 256;
    return launch_pdl(simt_down_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, *a.tab, a);
}

}  // namespace moe
