// combine.cu -- weighted un-permute and combine: every token collects its k
// expert outputs from their permuted positions and adds them in slot order
// (HARMOEny write-up, part 2 and part 3.3 step 6: finished tokens return to
// their owner).  The routing weight was applied in the down-projection
// epilogue; a split-K down projection leaves `splits` partial rows, added
// here first (in a fixed order over the splits), then the k slots (in
// ascending j), in fp32, rounded once to the activation type.  In the batch
// regime the partial rows arrive rounded to bf16 (half the bytes to write and
// read; one more rounding, which the tolerance of bf16 layers covers).
// Deterministic: no atomics.
//
// The kernel is bound by HBM (the partial rows are read once): each thread
// reads all k of its token's permuted positions first and then issues every
// partial-row load of the token before adding any of them, so that the loads
// of all slots are in flight together instead of one slot's address waiting
// on the previous slot's data.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

// W consecutive values of one partial row -- fp32, or bf16 (PB) where the batch
// regime's down projection rounded its rows -- widened to fp32, loaded with
// vector loads that bypass L1 (each partial row is read once).  `base` is the
// partial buffer, `off` the element offset of the first value.
template <int W, bool PB>
struct Vec {
    float v[W];
    __device__ __forceinline__ void load(const void *base, size_t off) {
        if constexpr (PB) {
            const uint16_t *p = static_cast<const uint16_t *>(base) + off;
            if constexpr (W >= 8) {
#pragma unroll
                for (int h = 0; h < W / 8; ++h) {
                    const uint4 q = __ldcg(reinterpret_cast<const uint4 *>(p + 8 * h));
                    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        v[8 * h + 2 * i] = bf16lo(w[i]);
                        v[8 * h + 2 * i + 1] = bf16hi(w[i]);
                    }
                }
            } else {
                const uint2 q = __ldcg(reinterpret_cast<const uint2 *>(p));
                v[0] = bf16lo(q.x);
                v[1] = bf16hi(q.x);
                v[2] = bf16lo(q.y);
                v[3] = bf16hi(q.y);
            }
        } else {
            const float *p = static_cast<const float *>(base) + off;
#pragma unroll
            for (int i = 0; i < W; i += 4) {
                const float4 q = __ldcg(reinterpret_cast<const float4 *>(p + i));
                v[i] = q.x;
                v[i + 1] = q.y;
                v[i + 2] = q.z;
                v[i + 3] = q.w;
            }
        }
    }
};

// One output chunk: token t, features c .. c + W - 1, from the token's
// permuted positions pos[j] (-1 for a slot past k or a bad position): the sum
// over slots j, ascending, of the partial rows (the reduction splits added
// first, in groups of four in split order), rounded once to the activation type.
template <bool BF16, int KMAX, int W, bool PB>
__device__ __forceinline__ void combine_item(const CombineArgs &a, int t, int c, const int (&pos)[KMAX]) {
    float y[W];
#pragma unroll
    for (int e = 0; e < W; ++e) y[e] = 0.0f;
    if (a.splits == 1) {
        Vec<W, PB> q[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
#pragma unroll
            for (int e = 0; e < W; ++e) q[j].v[e] = 0.0f;
            if (pos[j] >= 0) q[j].load(a.ypart, static_cast<size_t>(pos[j]) * a.m + c);
        }
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
            if (pos[j] >= 0)
#pragma unroll
                for (int e = 0; e < W; ++e) y[e] += 0.0f + q[j].v[e];
    } else {
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            if (pos[j] < 0) continue;
            // partial rows of the split reduction, added in a fixed order
            const size_t base = static_cast<size_t>(pos[j]) * a.m + c;
            float v[W];
#pragma unroll
            for (int e = 0; e < W; ++e) v[e] = 0.0f;
            // groups of up to four splits, each group's loads issued
            // together (a short last group too: one round trip instead of
            // one per split); a full group adds ((p0 + p1) + (p2 + p3)),
            // a short one its splits one at a time in split order
            for (int s = 0; s < a.splits; s += 4) {
                const int n = a.splits - s < 4 ? a.splits - s : 4;
                Vec<W, PB> p0, p1, p2, p3;
                p0.load(a.ypart, base + (s + 0) * a.split_stride);
                if (n > 1) p1.load(a.ypart, base + (s + 1) * a.split_stride);
                if (n > 2) p2.load(a.ypart, base + (s + 2) * a.split_stride);
                if (n > 3) p3.load(a.ypart, base + (s + 3) * a.split_stride);
                if (n == 4) {
#pragma unroll
                    for (int e = 0; e < W; ++e) v[e] += (p0.v[e] + p1.v[e]) + (p2.v[e] + p3.v[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < W; ++e) {
                        v[e] += p0.v[e];
                        if (n > 1) v[e] += p1.v[e];
                        if (n > 2) v[e] += p2.v[e];
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < W; ++e) y[e] += v[e];
        }
    }
    if (BF16) {
        uint32_t o[W / 2];
#pragma unroll
        for (int e = 0; e < W / 2; ++e) o[e] = pack_bf16x2(y[2 * e], y[2 * e + 1]);
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.y) + static_cast<size_t>(t) * a.m + c;
        if constexpr (W >= 8) {
#pragma unroll
            for (int h = 0; h < W / 8; ++h)
                *reinterpret_cast<uint4 *>(dst + 8 * h) =
                    make_uint4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3]);
        } else {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(o[0], o[1]);
        }
    } else {
        float *dst = static_cast<float *>(a.y) + static_cast<size_t>(t) * a.m + c;
#pragma unroll
        for (int e = 0; e < W; e += 4)
            *reinterpret_cast<float4 *>(dst + e) = make_float4(y[e], y[e + 1], y[e + 2], y[e + 3]);
    }
}

// W outputs per thread (4 or 8 consecutive features of one token); KMAX >= k.
template <bool BF16, int KMAX, int W, bool PB>
__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
    if (threadIdx.x == 0)
        touch_params(a.ypart, a.splits, a.split_stride, a.scatter, a.T, a.k, a.m, a.y, a.err);
    pdl_wait();
    pdl_trigger();
    const int vec = a.m / W;
    const long long n = static_cast<long long>(a.T) * vec;
    const int rows = a.T * a.k;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / vec), c = static_cast<int>(i % vec) * W;
        int pos[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            pos[j] = -1;
            if (j < a.k) {
                const int p = a.scatter[static_cast<size_t>(t) * a.k + j];
                if (p < 0 || p >= rows)
                    flag_error(a.err, kErrGatherIndex);
                else
                    pos[j] = p;
            }
        }
        combine_item<BF16, KMAX, W, PB>(a, t, c, pos);
    }
}

// Batch-sized calls with bf16 partial rows: one warp per token.  The token's k
// permuted positions are read once (lanes 0 .. k - 1) and shared by shuffle,
// then the warp walks the token's features in chunks of 32 W (W per lane): no
// dependent position load per chunk, so a lane's partial-row loads of
// successive chunks are the only round trips.  Same arithmetic and order as
// combine_kernel.
template <bool BF16, int KMAX, int W, bool PB>
__global__ void __launch_bounds__(256) combine_tokens_kernel(const CombineArgs a) {
    if (threadIdx.x == 0)
        touch_params(a.ypart, a.splits, a.split_stride, a.scatter, a.T, a.k, a.m, a.y, a.err);
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const long long warp0 = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const int rows = a.T * a.k;
    for (long long tt = warp0; tt < a.T; tt += nwarps) {
        const int t = static_cast<int>(tt);
        int mine = -1;
        if (lane < a.k) {
            const int p = a.scatter[static_cast<size_t>(t) * a.k + lane];
            if (p < 0 || p >= rows)
                flag_error(a.err, kErrGatherIndex);
            else
                mine = p;
        }
        int pos[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) pos[j] = __shfl_sync(0xffffffffu, mine, j);
#pragma unroll 2
        for (int c = lane * W; c < a.m; c += 32 * W) combine_item<BF16, KMAX, W, PB>(a, t, c, pos);
    }
}

template <bool BF16, int KMAX, bool PB>
cudaError_t launch_w(const CombineArgs &a, cudaStream_t s) {
    constexpr long long kGridThreads = 152LL * 16 * 256;
    if constexpr (PB) {
        // bf16 partial rows of a large batch (batch regime): a warp per token,
        // 16 features per lane, so a lane has as many bytes in flight as with
        // fp32 rows and 8 features, and no position load per chunk (Mixtral
        // shape, T = 8192: 71 us with the per-chunk kernel and 8 features of
        // bf16 rows, 30% of HBM; 56 us now).  Smaller batches give too few
        // warps for it (T = 512: 16 us against 11 with the per-chunk kernel),
        // so it takes batches of at least two blocks of warps per SM.
        if (a.m % 16 == 0 && a.T >= 2 * 152 * 8) {
            long long blocks = (static_cast<long long>(a.T) + 7) / 8;  // 8 warps per block
            if (blocks * 256 > kGridThreads) blocks = kGridThreads / 256;
            return launch_pdl(combine_tokens_kernel<BF16, KMAX, 16, PB>, dim3(static_cast<unsigned>(blocks)),
                              dim3(256), 0, s, a);
        }
    }
    const int w = (a.m % 8 == 0) ? 8 : 4;
    const long long n = static_cast<long long>(a.T) * (a.m / w);
    long long blocks = (n + 255) / 256;
    if (blocks * 256 > kGridThreads) blocks = kGridThreads / 256;
    const dim3 grid(static_cast<unsigned>(blocks));
    return w == 8 ? launch_pdl(combine_kernel<BF16, KMAX, 8, PB>, grid, dim3(256), 0, s, a)
                  : launch_pdl(combine_kernel<BF16, KMAX, 4, PB>, grid, dim3(256), 0, s, a);
}

template <bool BF16>
cudaError_t launch_k(const CombineArgs &a, cudaStream_t s) {
    if (a.part_bf16)
        return a.k <= 2 ? launch_w<BF16, 2, true>(a, s) : launch_w<BF16, kMaxTopK, true>(a, s);
    return a.k <= 2 ? launch_w<BF16, 2, false>(a, s) : launch_w<BF16, kMaxTopK, false>(a, s);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs &a, bool act_bf16, cudaStream_t s) {
    if (static_cast<long long>(a.T) * a.m == 0) return cudaSuccess;
    return act_bf16 ? launch_k<true>(a, s) : launch_k<false>(a, s);
}

}  // namespace moe
