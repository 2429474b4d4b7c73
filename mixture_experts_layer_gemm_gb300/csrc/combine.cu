// combine.cu -- weighted un-permute and combine: every token collects its k
// expert outputs from their permuted positions and adds them in slot order
// (HARMOEny write-up, part 2 and part 3.3 step 6: finished tokens return to
// their owner).  The routing weight was applied in the down-projection
// epilogue; a split-K down projection leaves `splits` partial rows, added
// here first (in split order), then the k slots (in ascending j), in fp32,
// rounded once to the activation type.  Deterministic: no atomics.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

template <bool BF16>
__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
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
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s = 0; s < a.splits; ++s) {
                const float4 p = *reinterpret_cast<const float4 *>(
                    a.ypart + s * a.split_stride + static_cast<size_t>(pos) * a.m + c);
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
        combine_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
    else
        combine_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
