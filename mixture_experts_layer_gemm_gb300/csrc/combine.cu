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

// Batch regime, bf16 partial rows, bf16 output: the partial rows staged in
// shared memory by bulk copies.  A warp takes (token, chunk of staged_chunk(R)
// features) items in turn; lanes 0 .. k*splits-1 each copy one partial row's
// chunk (the token's k positions read once per item and shared by shuffle)
// into the warp's buffer, completing on its mbarrier, while the warp sums the
// previous item from the other buffer.  The bytes in flight no longer cost
// registers: the register-staged kernels above stay latency-bound on these
// rows (a warp per token: 58% of HBM at T = 8192).  Same arithmetic and order
// as combine_item.  Every wait is bounded; a warp that gives up flags the
// error word and waits (bounded) for its own copies before leaving.
constexpr int kStagedMaxRows = 8;    // k x splits partial rows per item
constexpr int kStagedMaxWarps = 8;

// Features of one staged chunk for R partial rows an item: R chunks fill at
// most 8 KB, so a warp's double buffer is at most 16 KB and at least six warps
// fit in 96 KB for any R; chunks are whole multiples of a warp's 256-feature
// pass.
__host__ __device__ constexpr int staged_chunk(int R) {
    return (4096 / R) / 256 * 256 < 256 ? 256 : (4096 / R) / 256 * 256;
}

template <int KMAX>
__global__ void __launch_bounds__(kStagedMaxWarps * 32) combine_staged_kernel(const CombineArgs a) {
    extern __shared__ __align__(128) uint8_t smem_cs[];
    __shared__ uint64_t bar[kStagedMaxWarps][2];
    if (threadIdx.x == 0)
        touch_params(a.ypart, a.splits, a.split_stride, a.scatter, a.T, a.k, a.m, a.y, a.err);
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int R = a.k * a.splits;  // partial rows per item, <= kStagedMaxRows
    const int CW = staged_chunk(R);
    const size_t buf_bytes = static_cast<size_t>(R) * CW * 2;
    uint8_t *bufs = smem_cs + static_cast<size_t>(wib) * 2 * buf_bytes;
    if (lane == 0) {
        mbar_init(&bar[wib][0], 1);
        mbar_init(&bar[wib][1], 1);
        fence_barrier_init();
    }
    __syncwarp();
    const int nch = (a.m + CW - 1) / CW;
    const long long items = static_cast<long long>(a.T) * nch;
    const long long step = static_cast<long long>(gridDim.x) * nw;
    const int rows_total = a.T * a.k;
    const uint16_t *part = static_cast<const uint16_t *>(a.ypart);
    int pos[2][KMAX];
    uint32_t phase[2] = {0u, 0u};
    bool pending[2] = {false, false};
    // copies of item `it` into buffer b (positions into pos[b])
    auto issue = [&](long long it, int b) {
        const int t = static_cast<int>(it / nch), c0 = static_cast<int>(it % nch) * CW;
        const int cw = min(CW, a.m - c0);
        int mine = -1;
        if (lane < a.k) {
            const int p = a.scatter[static_cast<size_t>(t) * a.k + lane];
            if (p < 0 || p >= rows_total)
                flag_error(a.err, kErrGatherIndex);
            else
                mine = p;
        }
        int valid = 0;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            pos[b][j] = __shfl_sync(0xffffffffu, mine, j);
            valid += (j < a.k && pos[b][j] >= 0) ? 1 : 0;
        }
        uint8_t *dst = bufs + static_cast<size_t>(b) * buf_bytes;
        if (lane == 0) mbar_arrive_expect_tx(&bar[wib][b], static_cast<uint32_t>(valid * a.splits * cw * 2));
        __syncwarp();
        if (lane < R) {
            const int j = lane / a.splits, sp = lane - j * a.splits;
            int pj = -1;
#pragma unroll
            for (int jj = 0; jj < KMAX; ++jj)
                if (jj == j) pj = pos[b][jj];
            if (pj >= 0)
                bulk_g2s_once(dst + static_cast<size_t>(lane) * CW * 2,
                              part + static_cast<size_t>(sp) * a.split_stride + static_cast<size_t>(pj) * a.m + c0,
                              static_cast<uint32_t>(cw * 2), &bar[wib][b]);
        }
        pending[b] = true;
    };
    long long it = static_cast<long long>(blockIdx.x) * nw + wib;
    int b = 0;
    if (it < items) issue(it, 0);
    bool ok = true;
    for (; it < items; it += step, b ^= 1) {
        const long long nxt = it + step;
        if (nxt < items) {
            // buffer b ^ 1 was read by every lane in the last iteration
            fence_proxy_async_smem();
            __syncwarp();
            issue(nxt, b ^ 1);
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&bar[wib][b], phase[b]))) {
            if (lane == 0) flag_error(a.err, kErrWaitTimeout);
            ok = false;
            break;
        }
        phase[b] ^= 1u;
        pending[b] = false;
        const int t = static_cast<int>(it / nch), c0 = static_cast<int>(it % nch) * CW;
        const int cw = min(CW, a.m - c0);
        const uint8_t *src = bufs + static_cast<size_t>(b) * buf_bytes;
        for (int f = lane * 8; f < cw; f += 256) {
            float y[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = 0.0f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (j >= a.k || pos[b][j] < 0) continue;
                const uint8_t *row0 = src + static_cast<size_t>(j * a.splits) * CW * 2 + f * 2;
                if (a.splits == 1) {
                    const uint4 q = *reinterpret_cast<const uint4 *>(row0);
                    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        y[2 * i] += 0.0f + bf16lo(w[i]);
                        y[2 * i + 1] += 0.0f + bf16hi(w[i]);
                    }
                } else {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = 0.0f;
                    for (int s0 = 0; s0 < a.splits; s0 += 4) {
                        const int n = a.splits - s0 < 4 ? a.splits - s0 : 4;
                        float pv[4][8];
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            if (g < n) {
                                const uint4 q = *reinterpret_cast<const uint4 *>(
                                    row0 + static_cast<size_t>(s0 + g) * CW * 2);
                                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    pv[g][2 * i] = bf16lo(w[i]);
                                    pv[g][2 * i + 1] = bf16hi(w[i]);
                                }
                            }
                        }
                        if (n == 4) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) v[e] += (pv[0][e] + pv[1][e]) + (pv[2][e] + pv[3][e]);
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                v[e] += pv[0][e];
                                if (n > 1) v[e] += pv[1][e];
                                if (n > 2) v[e] += pv[2][e];
                            }
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) y[e] += v[e];
                }
            }
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = pack_bf16x2(y[2 * e], y[2 * e + 1]);
            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.y) + static_cast<size_t>(t) * a.m + c0 + f) =
                make_uint4(o[0], o[1], o[2], o[3]);
        }
        __syncwarp();  // every lane is past its reads of buffer b before it is refilled
    }
    if (!ok) {
        // copies this warp issued may still be landing in its buffers
        for (int bb = 0; bb < 2; ++bb)
            if (pending[bb] && lane == 0) mbar_wait(&bar[wib][bb], phase[bb]);
        __syncwarp();
    }
}

template <bool BF16, int KMAX, bool PB>
cudaError_t launch_w(const CombineArgs &a, cudaStream_t s) {
    constexpr long long kGridThreads = 152LL * 16 * 256;
    if constexpr (PB && BF16) {
        // bf16 partial rows staged in shared memory by bulk copies (96 KB a
        // block, two blocks an SM), for an unsplit down projection (Mixtral
        // shape, Zipf 1.2: combine T = 512 11.8 -> 10.0 us, T = 8192 55.9 ->
        // 40.9 us).  With two splits (T = 2048: four rows an item in
        // 1024-feature chunks, six warps a block) it measured the same as the
        // per-chunk kernel (26.6 us), which stays there.
        const int R = a.k * a.splits;
        if (a.m % 8 == 0 && a.splits == 1 && R <= kStagedMaxRows) {
            const int CW = staged_chunk(R);
            const size_t per_warp = 2 * static_cast<size_t>(R) * CW * 2;
            int nw = static_cast<int>((96 * 1024) / per_warp);
            nw = nw < 1 ? 1 : (nw > kStagedMaxWarps ? kStagedMaxWarps : nw);
            const size_t smem = per_warp * nw;
            auto kern = combine_staged_kernel<KMAX>;
            static int configured = 0;
            if (static_cast<int>(smem) > configured) {
                const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                             static_cast<int>(smem));
                if (err != cudaSuccess) return err;
                configured = static_cast<int>(smem);
            }
            const long long items = static_cast<long long>(a.T) * ((a.m + CW - 1) / CW);
            long long blocks = (items + nw - 1) / nw;
            if (blocks > 2 * 152) blocks = 2 * 152;
            return launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(32 * nw), smem, s, a);
        }
    }
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
