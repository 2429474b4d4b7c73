// route.cu -- routing kernels: router GEMM fused with softmax + top-k, and the
// histogram / scan / stable permute that puts the T*k (token, slot) pairs in
// expert-contiguous order.
//
// Router and gating: HARMOEny write-up, part 1 "What is MoE" (a router picks
// experts per token) and part 3.3 step 1; the gating network runs on the GPU
// in the expert-cache article, section 3.1.  The fusion of GEMM, softmax and
// selection (and the permute) into one kernel follows the Deep-Fusion rule of
// the DeepSpeed-Inference article, part 2: tile along the token dimension,
// which carries no cross-tile dependency, and keep the reduction (over m, then
// over E) inside the tile.
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

// The same selection by one warp, for a token whose logits sit in shared
// memory: lane l holds experts l and (EMAX = 64) l + 32, and each of the k
// rounds is a warp reduction instead of a scan over all experts.  The choice
// equals select_topk's scan in expert order: the largest logit left, the lower
// id among equal ones; a NaN is chosen only when it is the first candidate
// left (the scan starts from that candidate and no comparison replaces a NaN;
// a NaN met later never replaces a number).  The weights are select_topk's
// arithmetic on the same logits: exp(l_j - l_0) summed in round order, then
// divided.  Lane j < k receives slot j: *id and *wt.
template <int EMAX>
__device__ __forceinline__ void select_topk_warp(const float *lg, int E, int k, int lane, int *id, float *wt) {
    const float v0 = (lane < EMAX && lane < E) ? lg[lane] : 0.0f;
    const float v1 = (EMAX > 32 && lane + 32 < E) ? lg[lane + 32] : 0.0f;
    bool left0 = lane < EMAX && lane < E, left1 = EMAX > 32 && lane + 32 < E;  // untaken candidates
    float l0 = 0.0f, denom = 0.0f, mine = 0.0f;
    int my_id = -1;
#pragma unroll 1
    for (int j = 0; j < k; ++j) {
        const unsigned m0 = __ballot_sync(0xffffffffu, left0), m1 = __ballot_sync(0xffffffffu, left1);
        const int first = m0 ? __ffs(m0) - 1 : 32 + __ffs(m1) - 1;
        const float fv = __shfl_sync(0xffffffffu, first < 32 ? v0 : v1, first & 31);
        int bi = first;
        float bv = fv;
        if (fv == fv) {
            // this lane's best number left: (v0, lane) before (v1, lane + 32) on a tie
            const bool h0 = left0 && v0 == v0, h1 = left1 && v1 == v1;
            const bool pick0 = h0 && (!h1 || v0 >= v1);
            bool has = h0 || h1;
            float cv = pick0 ? v0 : v1;
            int ci = pick0 ? lane : lane + 32;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, cv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, ci, o);
                const bool oh = __shfl_xor_sync(0xffffffffu, has, o);
                if (oh && (!has || ov > cv || (ov == cv && oi < ci))) {
                    cv = ov;
                    ci = oi;
                    has = true;
                }
            }
            bi = ci;
            bv = cv;
        }
        if (bi == lane) left0 = false;
        if (bi == lane + 32) left1 = false;
        if (j == 0) l0 = bv;
        const float ej = expf(bv - l0);
        denom += ej;
        if (lane == j) {
            my_id = bi;
            mine = ej;
        }
    }
    *id = my_id;
    *wt = mine / denom;
}

// Histogram, exclusive scan and stable scatter of the n = T*k flat indices by
// expert, done by one CTA (any multiple of 32 threads up to 1024):
//   pass 1: counts[e] by shared-memory integer atomics (order-free);
//   scan:   offsets by one warp;
//   pass 2: chunks of blockDim flat indices in index order; inside a warp the
//           rank of an index among equal ids is the popcount of the match
//           mask below its lane; per-warp counts are scanned across warps per
//           expert, so positions follow flat-index order exactly.
// The ids are read through L2 (they may have been written by other CTAs of the
// same launch).
struct PermuteSmem {
    int count[kMaxExperts];
    int base[kMaxExperts];
    int warp_cnt[32][kMaxExperts];
};

// The same stable counting sort for at most 32 (token, slot) pairs, by one
// warp and without block barriers (decode batches): lane i holds pair i; the
// lanes with equal expert ids find each other with a match, a pair's rank
// among them is the number of lower lanes with its id (stable by i); lanes e
// and e + 32 count expert e and e + 32 and scan the counts.
constexpr int kPermuteWarpMax = 32;
__device__ void permute_warp(const PermuteArgs &a, int lane) {
    const int n = a.T * a.k;  // <= kPermuteWarpMax
    int id = -1;
    if (lane < n) {
        id = __ldcg(a.ids + lane);
        if (id < 0 || id >= a.E) id = 0;
    }
    const unsigned peers = __match_any_sync(0xffffffffu, id);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    int c0 = 0, c1 = 0;  // pairs choosing expert lane, lane + 32
    for (int j = 0; j < n; ++j) {
        const int idj = __shfl_sync(0xffffffffu, id, j);
        c0 += idj == lane;
        c1 += idj == lane + 32;
    }
    int s0 = c0, s1 = c1;  // inclusive scans over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v0 = __shfl_up_sync(0xffffffffu, s0, o);
        const int v1 = __shfl_up_sync(0xffffffffu, s1, o);
        if (lane >= o) {
            s0 += v0;
            s1 += v1;
        }
    }
    const int total0 = __shfl_sync(0xffffffffu, s0, 31);
    const int excl0 = s0 - c0, excl1 = total0 + s1 - c1;
    if (lane < a.E) {
        a.counts[lane] = c0;
        a.offsets[lane] = excl0;
    }
    if (lane + 32 < a.E) {
        a.counts[lane + 32] = c1;
        a.offsets[lane + 32] = excl1;
    }
    if (lane == 0) a.offsets[a.E] = n;
    const int b0 = __shfl_sync(0xffffffffu, excl0, id & 31);
    const int b1 = __shfl_sync(0xffffffffu, excl1, id & 31);
    if (lane < n) {
        const int pos = (id < 32 ? b0 : b1) + rank;
        a.gather[pos] = lane;
        a.scatter[lane] = pos;
    }
}

__device__ void permute_block(const PermuteArgs &a, PermuteSmem &sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x;
    const int n = a.T * a.k;
    if (tid < kMaxExperts) sm.count[tid] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += nthreads) {
        int id = __ldcg(a.ids + i);
        if (id < 0 || id >= a.E) id = 0;  // flagged by whoever produced ids
        atomicAdd(&sm.count[id], 1);
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive scan over E <= 64 counts, two per lane
        const int c0 = (2 * lane < a.E) ? sm.count[2 * lane] : 0;
        const int c1 = (2 * lane + 1 < a.E) ? sm.count[2 * lane + 1] : 0;
        int incl = c0 + c1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const int excl = incl - c0 - c1;
        if (2 * lane < a.E) {
            sm.base[2 * lane] = excl;
            a.counts[2 * lane] = c0;
            a.offsets[2 * lane] = excl;
        }
        if (2 * lane + 1 < a.E) {
            sm.base[2 * lane + 1] = excl + c0;
            a.counts[2 * lane + 1] = c1;
            a.offsets[2 * lane + 1] = excl + c0;
        }
        if (lane == 31) a.offsets[a.E] = incl;
    }
    __syncthreads();
    const unsigned lt_mask = (1u << lane) - 1u;
    const int nwarps = nthreads >> 5;
    for (int c0 = 0; c0 < n; c0 += nthreads) {
        const int i = c0 + tid;
        const bool valid = i < n;
        int id = valid ? __ldcg(a.ids + i) : -1;
        if (valid && (id < 0 || id >= a.E)) id = 0;
        for (int e = lane; e < a.E; e += 32) sm.warp_cnt[warp][e] = 0;
        __syncwarp();
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        const int rank = __popc(peers & lt_mask);
        if (valid && lane == __ffs(peers) - 1) sm.warp_cnt[warp][id] = __popc(peers);
        __syncthreads();
        if (tid < a.E) {
            int run = sm.base[tid];
            for (int w = 0; w < nwarps; ++w) {
                const int c = sm.warp_cnt[w][tid];
                sm.warp_cnt[w][tid] = run;
                run += c;
            }
            sm.base[tid] = run;
        }
        __syncthreads();
        if (valid) {
            const int pos = sm.warp_cnt[warp][id] + rank;
            a.gather[pos] = i;
            a.scatter[i] = pos;
        }
        __syncthreads();
    }
}

// The permute of a multi-CTA router launch, in two parts, so that no single
// CTA walks the whole batch with block barriers.  Each CTA first ranks its own
// (token, slot) pairs [i0, i0 + n): a pair's rank is the number of earlier
// pairs of the CTA with the same expert (stable by flat index).  Warp 0 only;
// the rank goes to scatter[i] for now and the CTA's per-expert counts to
// cta_count[cta][e].  s_cnt: kMaxExperts ints of shared memory.
__device__ void permute_rank_local(const PermuteArgs &a, int i0, int n, int cta, int *s_cnt, int lane) {
    for (int e = lane; e < a.E; e += 32) s_cnt[e] = 0;
    __syncwarp();
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int c0 = 0; c0 < n; c0 += 32) {
        const bool valid = c0 + lane < n;
        int id = valid ? __ldcg(a.ids + i0 + c0 + lane) : -1;
        if (valid && (id < 0 || id >= a.E)) id = 0;  // flagged by whoever produced ids
        const unsigned peers = __match_any_sync(0xffffffffu, id);
        const int base = valid ? s_cnt[id] : 0;
        __syncwarp();
        if (valid) {
            a.scatter[i0 + c0 + lane] = base + __popc(peers & lt_mask);
            if (lane == __ffs(peers) - 1) s_cnt[id] = base + __popc(peers);
        }
        __syncwarp();
    }
    for (int e = lane; e < a.E; e += 32) a.cta_count[static_cast<size_t>(cta) * a.E + e] = s_cnt[e];
}

// The launch's last CTA, once every CTA ranked its pairs: per expert, the
// exclusive prefix of the counts over CTAs (one warp per expert, in place);
// the expert totals, counts and offsets; then every pair in parallel at
// offsets[e] + prefix[cta][e] + rank.  The result is the stable counting sort
// of permute_block.
__device__ void permute_finish(const PermuteArgs &a, int ncta, int per_cta, PermuteSmem &sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    // loads are issued in batches of kB, so that a batch costs one round trip
    // to L2 instead of one per element
    constexpr int kB = 8;
    for (int e = warp; e < a.E; e += nwarps) {
        int carry = 0;
        for (int c0 = 0; c0 < ncta; c0 += 32 * kB) {
            int v[kB];
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const int c = c0 + 32 * b + lane;
                v[b] = c < ncta ? __ldcg(a.cta_count + static_cast<size_t>(c) * a.E + e) : 0;
            }
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                const int c = c0 + 32 * b + lane;
                int incl = v[b];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int x = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += x;
                }
                if (c < ncta) a.cta_count[static_cast<size_t>(c) * a.E + e] = carry + incl - v[b];
                carry += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
        if (lane == 0) sm.count[e] = carry;
    }
    __syncthreads();
    if (warp == 0) {  // exclusive scan over E <= 64 totals, two per lane
        const int c0 = (2 * lane < a.E) ? sm.count[2 * lane] : 0;
        const int c1 = (2 * lane + 1 < a.E) ? sm.count[2 * lane + 1] : 0;
        int incl = c0 + c1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const int excl = incl - c0 - c1;
        if (2 * lane < a.E) {
            sm.base[2 * lane] = excl;
            a.counts[2 * lane] = c0;
            a.offsets[2 * lane] = excl;
        }
        if (2 * lane + 1 < a.E) {
            sm.base[2 * lane + 1] = excl + c0;
            a.counts[2 * lane + 1] = c1;
            a.offsets[2 * lane + 1] = excl + c0;
        }
        if (lane == 31) a.offsets[a.E] = incl;
    }
    __syncthreads();
    const int n = a.T * a.k;
    const int nthreads = blockDim.x;
    for (int i0 = 0; i0 < n; i0 += nthreads * kB) {
        int id[kB], rank[kB], pre[kB];
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int i = i0 + b * nthreads + tid;
            id[b] = i < n ? __ldcg(a.ids + i) : 0;
            rank[b] = i < n ? __ldcg(a.scatter + i) : 0;
            if (id[b] < 0 || id[b] >= a.E) id[b] = 0;
        }
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int i = i0 + b * nthreads + tid;
            pre[b] = i < n ? __ldcg(a.cta_count + static_cast<size_t>(i / per_cta) * a.E + id[b]) : 0;
        }
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int i = i0 + b * nthreads + tid;
            if (i < n) {
                const int pos = sm.base[id[b]] + pre[b] + rank[b];
                a.gather[pos] = i;
                a.scatter[i] = pos;
            }
        }
    }
}

// Router GEMM + softmax + top-k, with the permute fused in.
// One CTA per group of TOK tokens (TOK * EMAX <= 64).  The 256 threads split
// the hidden dimension into 16-byte chunks (chunk c goes to thread c mod 256);
// a thread loads the router weights of its chunk once and applies them to all
// TOK tokens, keeping TOK x E partial sums.  Every thread adds its products in
// sequence, a warp-shuffle tree adds the 32 lane sums and one thread per
// (token, expert) adds the 8 warp sums in warp order: a fixed, deterministic
// order.  Warp w then selects the top-k of token w.  The last CTA to finish
// (a fenced ticket on a counter it resets) runs the permute for the whole batch.
// With SMEM_W the whole transposed router matrix (E x m, activation type) is
// first brought into shared memory by bulk copies, so that each thread's
// products wait on shared-memory reads instead of a chain of L2 round trips.
template <typename ActT, int EMAX, bool SMEM_W>
__global__ void __launch_bounds__(256) router_topk_kernel(RouterArgs a, PermuteArgs pa) {
    pdl_wait();
    pdl_trigger();
    constexpr int TOK = (64 / EMAX) < 1 ? 1 : (64 / EMAX);
    extern __shared__ __align__(16) uint8_t s_w[];
    __shared__ float s_part[8][TOK][EMAX];
    __shared__ float s_logit[TOK][EMAX];
    __shared__ PermuteSmem psm;
    __shared__ int s_last;
    __shared__ uint64_t s_wbar;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * TOK;
    const int ntok = min(TOK, a.T - t0);
    constexpr int kVec = 16 / sizeof(ActT);  // elements per 16-byte chunk
    const int nchunks = a.m / kVec;
    if constexpr (SMEM_W) {
        const uint32_t bytes = static_cast<uint32_t>(a.E) * a.m * sizeof(ActT);
        if (tid == 0) {
            mbar_init(&s_wbar, 1);
            fence_barrier_init();
            mbar_arrive_expect_tx(&s_wbar, bytes);
            for (uint32_t off = 0; off < bytes; off += 32768u) {
                const uint32_t n = bytes - off < 32768u ? bytes - off : 32768u;
                bulk_g2s(s_w + off, static_cast<const uint8_t *>(a.wra) + off, n, &s_wbar);
            }
        }
        __syncthreads();
        if (!mbar_wait(&s_wbar, 0) && tid == 0) flag_error(a.err, kErrWaitTimeout);
    }

    float acc[TOK][EMAX];
#pragma unroll
    for (int tk = 0; tk < TOK; ++tk)
#pragma unroll
        for (int e = 0; e < EMAX; ++e) acc[tk][e] = 0.0f;
    for (int ch = tid; ch < nchunks; ch += 256) {
        const int c = ch * kVec;
        uint4 xraw[TOK];  // this chunk of every token of the group, packed
#pragma unroll
        for (int tk = 0; tk < TOK; ++tk)
            xraw[tk] = (tk < ntok) ? ld_nc_v4(static_cast<const ActT *>(a.x) +
                                              static_cast<size_t>(t0 + tk) * a.m + c)
                                   : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
            if (e < a.E) {
                float wv[kVec];
                if constexpr (SMEM_W) {
                    const uint4 wr = *reinterpret_cast<const uint4 *>(
                        s_w + (static_cast<size_t>(e) * a.m + c) * sizeof(ActT));
                    const uint32_t wu[4] = {wr.x, wr.y, wr.z, wr.w};
                    if constexpr (sizeof(ActT) == 2) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            wv[2 * i] = bf16lo(wu[i]);
                            wv[2 * i + 1] = bf16hi(wu[i]);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) wv[i] = __uint_as_float(wu[i]);
                    }
                } else {
                    const float *wr = a.wrt + static_cast<size_t>(e) * a.m + c;
#pragma unroll
                    for (int i = 0; i < kVec; i += 4) {
                        const float4 w4 = __ldg(reinterpret_cast<const float4 *>(wr + i));
                        wv[i] = w4.x;
                        wv[i + 1] = w4.y;
                        wv[i + 2] = w4.z;
                        wv[i + 3] = w4.w;
                    }
                }
#pragma unroll
                for (int tk = 0; tk < TOK; ++tk) {
                    const uint32_t u[4] = {xraw[tk].x, xraw[tk].y, xraw[tk].z, xraw[tk].w};
                    if constexpr (sizeof(ActT) == 2) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            acc[tk][e] = fmaf(bf16lo(u[i]), wv[2 * i], acc[tk][e]);
                            acc[tk][e] = fmaf(bf16hi(u[i]), wv[2 * i + 1], acc[tk][e]);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[tk][e] = fmaf(__uint_as_float(u[i]), wv[i], acc[tk][e]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int tk = 0; tk < TOK; ++tk)
#pragma unroll
        for (int e = 0; e < EMAX; ++e) {
            const float v = warp_sum(acc[tk][e]);
            if (lane == 0) s_part[warp][tk][e] = v;
        }
    __syncthreads();
    for (int i = tid; i < ntok * a.E; i += 256) {
        const int tk = i / a.E, e = i % a.E;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) v += s_part[w][tk][e];
        if (a.bias) v += a.bias[e];
        s_logit[tk][e] = v;
        if (a.logits) a.logits[static_cast<size_t>(t0 + tk) * a.E + e] = v;
    }
    __syncthreads();
    for (int tk = warp; tk < ntok; tk += 8) {
        const int t = t0 + tk;
        float l[EMAX];
#pragma unroll
        for (int e = 0; e < EMAX; ++e) l[e] = (e < a.E) ? s_logit[tk][e] : 0.0f;
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
    // ---- the last CTA to finish permutes the whole batch
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned ticket = atomicAdd(a.ticket, 1u);
        s_last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        permute_block(pa, psm);
        if (tid == 0) *a.ticket = 0;  // ready for the next launch
    }
}

// bf16 router on the warp-level tensor cores: logits[16 tokens x E] per CTA
// as an m16n8k16 GEMM with the tokens on M and the experts on N (8 per MMA).
// The warps of the CTA (32 for E <= 16) split the hidden dimension in
// 32-element steps (4 per warp for m = 4096, loads issued together: the kernel
// is a latency chain at decode sizes, so many warps with few steps each); lane (g, t) reads the
// 16-byte run t of token rows g and g + 8 and of expert row g of the router
// matrix (stored [EMAX x m], zero rows past E), which feed two MMAs under one
// shared permutation of the reduction index.  The warp partials are added
// in warp order (a fixed order), then each warp selects the top-k of its
// tokens, and the launch's last CTA runs the permute.
// Warps per CTA: 32 while the per-thread expert state is small; fewer for
// wide routers (E > 16) so that 64 K registers cover the top-k state.
template <int EMAX>
constexpr int router_warps() { return EMAX <= 16 ? 32 : (EMAX == 32 ? 16 : 8); }

template <int EMAX>
__global__ void __launch_bounds__(router_warps<EMAX>() * 32) router_mma_kernel(RouterArgs a, PermuteArgs pa) {
    // Before the wait: the parameters, and the router matrix (read by every
    // CTA; [EMAX x m] in the activation type) on its way into L2 -- neither is
    // written by the predecessor.
    if (threadIdx.x == 0) {
        touch_params(a.x, a.wra, a.bias, a.T, a.m, a.E, a.k, a.ids, a.w, a.logits, a.ticket, a.err);
        touch_params(pa.ids, pa.T, pa.k, pa.E, pa.counts, pa.offsets, pa.gather, pa.scatter, pa.cta_count);
        if (blockIdx.x == 0) bulk_prefetch_l2(a.wra, static_cast<size_t>(EMAX) * a.m * 2);
    }
    pdl_wait();
    pdl_trigger();
    constexpr int kRouterWarps = router_warps<EMAX>();
    constexpr int NT = EMAX / 8;
    constexpr int TOK = 16;
    extern __shared__ __align__(16) float s_red[];  // [kRouterWarps][TOK][EMAX]
    __shared__ float s_logit[TOK][EMAX];
    __shared__ PermuteSmem psm;
    __shared__ int s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int t0 = blockIdx.x * TOK;
    const int ntok = min(TOK, a.T - t0);
    const int nsteps = a.m / 32;
    const int s0 = (nsteps * warp) / kRouterWarps, s1 = (nsteps * (warp + 1)) / kRouterWarps;
    const uint16_t *x = static_cast<const uint16_t *>(a.x);
    const uint16_t *w = static_cast<const uint16_t *>(a.wra);
    const bool ra = g < ntok, rb = g + 8 < ntok;
    const uint16_t *xa = x + static_cast<size_t>(t0 + (ra ? g : 0)) * a.m + 8 * t;
    const uint16_t *xb = x + static_cast<size_t>(t0 + (rb ? g + 8 : 0)) * a.m + 8 * t;
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
#pragma unroll 4
    for (int st = s0; st < s1; ++st) {
        const int kb = st * 32;
        const uint4 va = ra ? ld_nc_v4(xa + kb) : make_uint4(0, 0, 0, 0);
        const uint4 vb = rb ? ld_nc_v4(xb + kb) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint4 wv = ld_nc_v4(w + static_cast<size_t>(nt * 8 + g) * a.m + kb + 8 * t);
            mma_bf16_16816(acc[nt], va.x, vb.x, va.y, vb.y, wv.x, wv.y);
            mma_bf16_16816(acc[nt], va.z, vb.z, va.w, vb.w, wv.z, wv.w);
        }
    }
    // D fragment: acc[nt][0..1] = (token g, experts nt*8+2t, +1), [2..3] = token g + 8
    float *red = s_red + static_cast<size_t>(warp) * TOK * EMAX;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int e = nt * 8 + 2 * t;
        red[g * EMAX + e] = acc[nt][0];
        red[g * EMAX + e + 1] = acc[nt][1];
        red[(g + 8) * EMAX + e] = acc[nt][2];
        red[(g + 8) * EMAX + e + 1] = acc[nt][3];
    }
    __syncthreads();
    for (int i = tid; i < ntok * a.E; i += kRouterWarps * 32) {
        const int tk = i / a.E, e = i % a.E;
        float v = 0.0f;
        for (int ww = 0; ww < kRouterWarps; ++ww) v += s_red[(ww * TOK + tk) * EMAX + e];
        if (a.bias) v += a.bias[e];
        s_logit[tk][e] = v;
        if (a.logits) a.logits[static_cast<size_t>(t0 + tk) * a.E + e] = v;
    }
    __syncthreads();
    for (int tk = warp; tk < ntok; tk += kRouterWarps) {
        const int tok = t0 + tk;
        int id;
        float wt;
        select_topk_warp<EMAX>(s_logit[tk], a.E, a.k, lane, &id, &wt);
        if (lane < a.k) {
            a.ids[static_cast<size_t>(tok) * a.k + lane] = id;
            a.w[static_cast<size_t>(tok) * a.k + lane] = wt;
        }
    }
    if (gridDim.x == 1) {
        // the whole batch is in this CTA: no ticket; one warp permutes small batches
        __syncthreads();
        if (pa.T * pa.k <= kPermuteWarpMax) {
            if (warp == 0) permute_warp(pa, lane);
        } else {
            permute_block(pa, psm);
        }
        return;
    }
    if (pa.cta_count) {  // this CTA ranks its own pairs first
        __syncthreads();
        if (warp == 0) permute_rank_local(pa, t0 * a.k, ntok * a.k, blockIdx.x, psm.count, lane);
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned ticket = atomicAdd(a.ticket, 1u);
        s_last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        if (pa.cta_count)
            permute_finish(pa, gridDim.x, TOK * a.k, psm);
        else
            permute_block(pa, psm);
        if (tid == 0) *a.ticket = 0;  // ready for the next launch
    }
}

// One thread per token: top-k from given fp32 logits.
template <int EMAX>
__global__ void __launch_bounds__(128) topk_from_logits_kernel(const float *logits, int T, int E,
                                                               int k, int32_t *ids_out,
                                                               float *w_out) {
    pdl_wait();
    pdl_trigger();
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
    pdl_wait();
    pdl_trigger();
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

// Standalone permute (after top-k from logits or from a given choice).
__global__ void __launch_bounds__(1024) permute_kernel(PermuteArgs a) {
    pdl_wait();
    pdl_trigger();
    __shared__ PermuteSmem psm;
    if (a.T * a.k <= kPermuteWarpMax) {
        if (threadIdx.x < 32) permute_warp(a, threadIdx.x);
        return;
    }
    permute_block(a, psm);
}

// ---- launchers ----------------------------------------------------------------
constexpr size_t kRouterSmemMax = 96 * 1024;

template <typename ActT, int EMAX>
static cudaError_t launch_router_e(const RouterArgs &a, const PermuteArgs &pa, cudaStream_t s) {
    constexpr int TOK = (64 / EMAX) < 1 ? 1 : (64 / EMAX);
    const unsigned grid = (a.T + TOK - 1) / TOK;
    const size_t wbytes = static_cast<size_t>(a.E) * a.m * sizeof(ActT);
    if (a.wra && wbytes <= kRouterSmemMax) {
        auto kern = router_topk_kernel<ActT, EMAX, true>;
        static size_t configured = 0;
        if (wbytes > configured) {
            const cudaError_t e = cudaFuncSetAttribute(
                kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kRouterSmemMax));
            if (e != cudaSuccess) return e;
            configured = kRouterSmemMax;
        }
        return launch_pdl(kern, dim3(grid), dim3(256), wbytes, s, a, pa);
    } else {
        return launch_pdl(router_topk_kernel<ActT, EMAX, false>, dim3(grid), dim3(256), 0, s, a, pa);
    }
}

template <int EMAX>
static cudaError_t launch_router_mma(const RouterArgs &a, const PermuteArgs &pa, cudaStream_t s) {
    constexpr int kRouterWarps = router_warps<EMAX>();
    const size_t smem = static_cast<size_t>(kRouterWarps) * 16 * EMAX * sizeof(float);
    auto kern = router_mma_kernel<EMAX>;
    static bool configured = false;
    if (!configured) {
        const cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch_pdl(kern, dim3((a.T + 15) / 16), dim3(kRouterWarps * 32), smem, s, a, pa);
}

template <typename ActT>
static cudaError_t launch_router_t(const RouterArgs &a, const PermuteArgs &pa, cudaStream_t s) {
    if (sizeof(ActT) == 2 && a.wra && a.m % 32 == 0) {
        if (a.E <= 8) return launch_router_mma<8>(a, pa, s);
        if (a.E <= 16) return launch_router_mma<16>(a, pa, s);
        if (a.E <= 32) return launch_router_mma<32>(a, pa, s);
        return launch_router_mma<64>(a, pa, s);
    }
    if (a.E <= 8) return launch_router_e<ActT, 8>(a, pa, s);
    if (a.E <= 16) return launch_router_e<ActT, 16>(a, pa, s);
    if (a.E <= 32) return launch_router_e<ActT, 32>(a, pa, s);
    return launch_router_e<ActT, 64>(a, pa, s);
}

cudaError_t launch_router_topk(const RouterArgs &a, const PermuteArgs &pa, bool act_bf16,
                               cudaStream_t s) {
    if (a.T <= 0) return cudaSuccess;
    return act_bf16 ? launch_router_t<__nv_bfloat16>(a, pa, s) : launch_router_t<float>(a, pa, s);
}

cudaError_t launch_topk_from_logits(const float *logits, int T, int E, int k, int32_t *ids,
                                    float *w, cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    dim3 grid((T + 127) / 128), block(128);
    if (E <= 8)
        return launch_pdl(topk_from_logits_kernel<8>, grid, block, 0, s, logits, T, E, k, ids, w);
    else if (E <= 16)
        return launch_pdl(topk_from_logits_kernel<16>, grid, block, 0, s, logits, T, E, k, ids, w);
    else if (E <= 32)
        return launch_pdl(topk_from_logits_kernel<32>, grid, block, 0, s, logits, T, E, k, ids, w);
    else
        return launch_pdl(topk_from_logits_kernel<64>, grid, block, 0, s, logits, T, E, k, ids, w);
}

cudaError_t launch_topk_copy_validate(const int32_t *ids_in, const float *w_in, int T, int E,
                                      int k, int32_t *ids_out, float *w_out, uint32_t *err,
                                      cudaStream_t s) {
    if (T <= 0) return cudaSuccess;
    return launch_pdl(topk_copy_validate_kernel, dim3((T + 127) / 128), dim3(128), 0, s, ids_in,
                      w_in, T, E, k, ids_out, w_out, err);
}

cudaError_t launch_permute(const PermuteArgs &a, cudaStream_t s) {
    return launch_pdl(permute_kernel, dim3(1), dim3(1024), 0, s, a);
}

}  // namespace moe
