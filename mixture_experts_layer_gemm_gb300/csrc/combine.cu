// combine.cu -- weighted un-permute and combine: every token collects its k
// expert outputs from their permuted positions and adds them in slot order
// (HARMOEny write-up, part 2 and part 3.3 step 6: finished tokens return to
// their owner).  The routing weight was applied in the down-projection
// epilogue; a split-K down projection leaves `splits` partial rows, added
// here first (in a fixed order over the splits), then the k slots (in
// ascending j), in fp32,
// rounded once to the activation type.  Deterministic: no atomics.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

template <bool BF16>
__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
    pdl_wait();
    pdl_trigger();
    const int vec = a.m / 4;  // 4 fp32 per thread
    const long long n = static_cast<long long>(a.T) * vec;
    const int rows = a.T * a.k;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / vec), c = static_cast<int>(i % vec) * 4;
        float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < a.k; ++j) {
            const int pos = a.scatter[static_cast<size_t>(t) * a.k + j];
            if (pos < 0 || pos >= rows) {
                flag_error(a.err, kErrGatherIndex);
                continue;
            }
            // partial rows of the split reduction, four loads in flight at a
            // time, added in a fixed order: ((p0 + p1) + (p2 + p3)) per group,
            // groups in split order
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            const float *base = a.ypart + static_cast<size_t>(pos) * a.m + c;
            int s = 0;
            for (; s + 4 <= a.splits; s += 4) {
                const float4 p0 = __ldcg(reinterpret_cast<const float4 *>(base + (s + 0) * a.split_stride));
                const float4 p1 = __ldcg(reinterpret_cast<const float4 *>(base + (s + 1) * a.split_stride));
                const float4 p2 = __ldcg(reinterpret_cast<const float4 *>(base + (s + 2) * a.split_stride));
                const float4 p3 = __ldcg(reinterpret_cast<const float4 *>(base + (s + 3) * a.split_stride));
                v.x += (p0.x + p1.x) + (p2.x + p3.x);
                v.y += (p0.y + p1.y) + (p2.y + p3.y);
                v.z += (p0.z + p1.z) + (p2.z + p3.z);
                v.w += (p0.w + p1.w) + (p2.w + p3.w);
            }
            for (; s < a.splits; ++s) {
                const float4 p = __ldcg(reinterpret_cast<const float4 *>(base + s * a.split_stride));
                v.x += p.x;
                v.y += p.y;
                v.z += p.z;
                v.w += p.w;
            }
            y.x += v.x;
            y.y += v.y;
            y.z += v.z;
            y.w += v.w;
        }
        if (BF16) {
            uint2 o;
            o.x = pack_bf16x2(y.x, y.y);
            o.y = pack_bf16x2(y.z, y.w);
            *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(a.y) +
                                       static_cast<size_t>(t) * a.m + c) = o;
        } else {
            *reinterpret_cast<float4 *>(static_cast<float *>(a.y) + static_cast<size_t>(t) * a.m +
                                        c) = y;
        }
    }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs &a, bool act_bf16, cudaStream_t s) {
    const long long n = static_cast<long long>(a.T) * (a.m / 4);
    if (n == 0) return cudaSuccess;
    long long blocks = (n + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (act_bf16)
        return launch_pdl(combine_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, a);
    else
        return launch_pdl(combine_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s, a);
}

}  // namespace moe
