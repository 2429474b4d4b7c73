// route.cu -- routing kernels: router GEMM fused with softmax + top-k, and the
// histogram / scan / stable permute that puts the T*k (token, slot) pairs in
// expert-contiguous order.
//
// Router and gating: HARMOEny write-up, part 1 "What is MoE" (a router picks
// experts per token) and part 3.3 step 1; the gating network runs on the GPU
// in the expert-cache article, section 3.1.  The fusion of GEMM, softmax and
// selection into one kernel follows the Deep-Fusion rule of the
// DeepSpeed-Inference article, part 2: tile along the token dimension, which
// carries no cross-tile dependency, and keep the reduction (over m, then over
// E) inside the tile.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

// Top-k over the logits held (identically) by every lane: larger logit first,
// ties to the lower expert id; weights are exp(l_j - l_0) / sum_j' exp(l_j' - l_0).
template <int EMAX>
__device__ __forceinline__ void select_topk(const float (&l)[EMAX], int E, int k, int (&ids)[kMaxTopK],
                                            float (&w)[kMaxTopK]) {
    uint64_t taken = 0;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
        if (j < k) {
            int best = -1;
            float bv = 0.0f;
#pragma unroll
            for (int e = 0; e < EMAX; ++e) {
                if (e < E && !((taken >> e) & 1ull)) {
                    if (best < 0 || l[e] > bv) {
                        best = e;
                        bv = l[e];
                    }
                }
            }
            ids[j] = best;
            w[j] = bv;  // logit for now
            taken |= 1ull << best;
        }
    }
    const float l0 = w[0];
    float denom = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
        if (j < k) {
            w[j] = expf(w[j] - l0);
            denom += w[j];
        }
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
        if (j < k) w[j] = w[j] / denom;
}

// One CTA per group of 8 tokens.  The 256 threads split the hidden dimension
// into 16-byte chunks (chunk c goes to thread c mod 256), so even a single
// token spreads its m x E router products over the whole CTA.  For each token
// every thread adds its products in sequence, a warp-shuffle tree adds the 32
// lane sums, and one thread per (token, expert) adds the 8 warp sums in warp
// order: a fixed, deterministic order.  Then warp w selects the top-k of
// token w.  x: [T x m] (fp32 or bf16); wrt: router weights transposed to
// [E x m] fp32 (an exact copy of the given values).
constexpr int kRouterTokens = 8;

template <typename ActT, int EMAX>
__global__ void __launch_bounds__(256) router_topk_kernel(RouterArgs a) {
    __shared__ float s_part[kRouterTokens][8][EMAX];
    __shared__ float s_logit[kRouterTokens][EMAX];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * kRouterTokens;
    const int ntok = min(kRouterTokens, a.T - t0);
    constexpr int kVec = 16 / sizeof(ActT);  // elements per 16-byte chunk
    const int nchunks = a.m / kVec;

    for (int tk = 0; tk < ntok; ++tk) {
        const ActT *xr = static_cast<const ActT *>(a.x) + static_cast<size_t>(t0 + tk) * a.m;
        float acc[EMAX];
#pragma unroll
        for (int e = 0; e < EMAX; ++e) acc[e] = 0.0f;
        for (int ch = tid; ch < nchunks; ch += 256) {
            const int c = ch * kVec;
            const uint4 raw = ld_nc_v4(xr + c);
            float xv[kVec];
            if constexpr (sizeof(ActT) == 2) {
                const uint32_t u[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    xv[2 * i] = bf16lo(u[i]);
                    xv[2 * i + 1] = bf16hi(u[i]);
                }
            } else {
                xv[0] = __uint_as_float(raw.x);
                xv[1] = __uint_as_float(raw.y);
                xv[2] = __uint_as_float(raw.z);
                xv[3] = __uint_as_float(raw.w);
            }
#pragma unroll
            for (int e = 0; e < EMAX; ++e) {
                if (e < a.E) {
                    const float *wr = a.wrt + static_cast<size_t>(e) * a.m + c;
#pragma unroll
                    for (int i = 0; i < kVec; i += 4) {
                        const float4 wv = __ldg(reinterpret_cast<const float4 *>(wr + i));
                        acc[e] = fmaf(xv[i], wv.x, acc[e]);
                        acc[e] = fmaf(xv[i + 1], wv.y, acc[e]);
                        acc[e] = fmaf(xv[i + 2], wv.z, acc[e]);
                        acc[e] = fmaf(xv[i + 3], wv.w, acc[e]);
                    }
                }
            }
        }
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
            const float v = warp_sum(acc[e]);
            if (lane == 0 && e < a.E) s_part[tk][warp][e] = v;
        }
    }
    __syncthreads();
    for (int i = tid; i < ntok * a.E; i += 256) {
        const int tk = i / a.E, e = i % a.E;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) v += s_part[tk][w][e];
        if (a.bias) v += a.bias[e];
        s_logit[tk][e] = v;
        if (a.logits) a.logits[static_cast<size_t>(t0 + tk) * a.E + e] = v;
    }
    __syncthreads();
    if (warp < ntok) {
        const int t = t0 + warp;
        float l[EMAX];
#pragma unroll
        for (int e = 0; e < EMAX; ++e) l[e] = (e < a.E) ? s_logit[warp][e] : 0.0f;
        int ids[kMaxTopK];
        float w[kMaxTopK];
        select_topk<EMAX>(l, a.E, a.k, ids, w);
#pragma unroll
        for (int j = 0; j < kMaxTopK; ++j)
            if (j < a.k && lane == j) {
                a.ids[static_cast<size_t>(t) * a.k + j] = ids[j];
                a.w[static_cast<size_t>(t) * a.k + j] = w[j];
            }
    }
}

// One thread per token: top-k from given fp32 logits.
template <int EMAX>
__global__ void __launch_bounds__(128) topk_from_logits_kernel(const float *logits, int T, int E,
                                                               int k, int32_t *ids_out,
                                                               float *w_out) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    float l[EMAX];
#pragma unroll
    for (int e = 0; e < EMAX; ++e) l[e] = (e < E) ? logits[static_cast<size_t>(t) * E + e] : 0.0f;
    int ids[kMaxTopK];
    float w[kMaxTopK];
    select_topk<EMAX>(l, E, k, ids, w);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
        if (j < k) {
            ids_out[static_cast<size_t>(t) * k + j] = ids[j];
            w_out[static_cast<size_t>(t) * k + j] = w[j];
        }
}

// One thread per token: copy a caller-given top-k choice, sending ids outside
// [0, E) to expert 0 and flagging them, and flagging repeated ids.
__global__ void topk_copy_validate_kernel(const int32_t *ids_in, const float *w_in, int T, int E,
                                          int k, int32_t *ids_out, float *w_out, uint32_t *err) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    uint32_t bits = 0;
    int seen[kMaxTopK];
    for (int j = 0; j < k; ++j) {
        int id = ids_in[static_cast<size_t>(t) * k + j];
        if (id < 0 || id >= E) {
            bits |= kErrExpertId;
            id = 0;
        }
        for (int jj = 0; jj < j; ++jj)
            if (seen[jj] == id) bits |= kErrDuplicateId;
        seen[j] = id;
        ids_out[static_cast<size_t>(t) * k + j] = id;
        w_out[static_cast<size_t>(t) * k + j] = w_in[static_cast<size_t>(t) * k + j];
    }
    if (bits) flag_error(err, bits);
}

// Histogram, exclusive scan and stable scatter in one CTA of 1024 threads.
//   pass 1: counts[e] by shared-memory integer atomics (order-free);
//   scan:   offsets by one warp;
//   pass 2: chunks of 1024 flat indices in index order; inside a warp the
//           rank of an index among equal ids is the popcount of the match
//           mask below its lane; per-warp counts are scanned across warps per
//           expert, so positions follow flat-index order exactly.
__global__ void __launch_bounds__(1024) permute_kernel(PermuteArgs a) {
    __shared__ int s_count[kMaxExperts];
    __shared__ int s_base[kMaxExperts];
    __shared__ int s_warp[32][kMaxExperts];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = a.T * a.k;
    if (tid < kMaxExperts) s_count[tid] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += blockDim.x) {
        int id = a.ids[i];
        if (id < 0 || id >= a.E) id = 0;  // flagged by whoever produced ids
        atomicAdd(&s_count[id], 1);
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive scan over E <= 64 counts, two per lane
        const int c0 = (2 * lane < a.E) ? s_count[2 * lane] : 0;
        const int c1 = (2 * lane + 1 < a.E) ? s_count[2 * lane + 1] : 0;
        int incl = c0 + c1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const int excl = incl - c0 - c1;
        if (2 * lane < a.E) {
            s_base[2 * lane] = excl;
            a.counts[2 * lane] = c0;
            a.offsets[2 * lane] = excl;
        }
        if (2 * lane + 1 < a.E) {
            s_base[2 * lane + 1] = excl + c0;
            a.counts[2 * lane + 1] = c1;
            a.offsets[2 * lane + 1] = excl + c0;
        }
        if (lane == 31) a.offsets[a.E] = incl;
    }
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int c0 = 0; c0 < n; c0 += blockDim.x) {
        const int i = c0 + tid;
        const bool valid = i < n;
        int id = valid ? a.ids[i] : -1;
        if (valid && (id < 0 || id >= a.E)) id = 0;
        for (int e = lane; e < a.E; e += 32) s_warp[warp][e] = 0;
        __syncwarp();
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        const int rank = __popc(peers & lt_mask);
        if (valid && lane == __ffs(peers) - 1) s_warp[warp][id] = __popc(peers);
        __syncthreads();
        if (tid < a.E) {
            int run = s_base[tid];
            for (int w = 0; w < 32; ++w) {
                const int c = s_warp[w][tid];
                s_warp[w][tid] = run;
                run += c;
            }
            s_base[tid] = run;
        }
        __syncthreads();
        if (valid) {
            const int pos = s_warp[warp][id] + rank;
            a.gather[pos] = i;
            a.scatter[i] = pos;
        }
        __syncthreads();
    }
}

// ---- launchers ----------------------------------------------------------------
template <typename ActT>
static cudaError_t launch_router_t(const RouterArgs &a, cudaStream_t s) {
    dim3 grid((a.T + kRouterTokens - 1) / kRouterTokens), block(256);
    if (a.E <= 8)
        router_topk_kernel<ActT, 8><<<grid, block, 0, s>>>(a);
    else if (a.E <= 16)
        router_topk_kernel<ActT, 16><<<grid, block, 0, s>>>(a);
    else if (a.E <= 32)
        router_topk_kernel<ActT, 32><<<grid, block, 0, s>>>(a);
    else
        router_topk_kernel<ActT, 64><<<grid, block, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_router_topk(const RouterArgs &a, bool act_bf16, cudaStream_t s) {
    if (a.T <= 0) return cudaSuccess;
    return act_bf16 ? launch_router_t<__nv_bfloat16>(a, s) : launch_router_t<float>(a, s);
}

cudaError_t launch_topk_from_logits(const float *logits, int T, int E, int k, int32_t *ids,
                                    float *w, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    dim3 grid((T + 127) / 128), block(128);
    if (E <= 8)
        topk_from_logits_kernel<8><<<grid, block, 0, s>>>(logits, T, E, k, ids, w);
    else if (E <= 16)
        topk_from_logits_kernel<16><<<grid, block, 0, s>>>(logits, T, E, k, ids, w);
    else if (E <= 32)
        topk_from_logits_kernel<32><<<grid, block, 0, s>>>(logits, T, E, k, ids, w);
    else
        topk_from_logits_kernel<64><<<grid, block, 0, s>>>(logits, T, E, k, ids, w);
    return cudaGetLastError();
}

cudaError_t launch_topk_copy_validate(const int32_t *ids_in, const float *w_in, int T, int E,
                                      int k, int32_t *ids_out, float *w_out, uint32_t *err,
                                      cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    topk_copy_validate_kernel<<<(T + 127) / 128, 128, 0, s>>>(ids_in, w_in, T, E, k, ids_out, w_out,
                                                              err);
    return cudaGetLastError();
}

cudaError_t launch_permute(const PermuteArgs &a, cudaStream_t s) {
    permute_kernel<<<1, 1024, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
