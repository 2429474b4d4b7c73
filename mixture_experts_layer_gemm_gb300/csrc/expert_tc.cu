// expert_tc.cu -- grouped expert GEMM on the 5th-generation tensor cores
// (tcgen05 + tensor memory), for the batch regime and for decode batches
// with many tokens per expert.
//
// Where the time goes: with hundreds of tokens per expert the expert matmuls
// are compute-bound (DeepSpeed-Inference article, part 1: batch inference is
// limited by compute; MoE-Lightning note, Hierarchical Roofline Model: the
// FFN's intensity grows with the batch).  The pages hand this regime to a
// vendor GEMM left unfused (DeepSpeed-Inference article, part 4); here it is a
// grouped GEMM over the experts' ragged token segments with the activation
// (SiLU(gate) * up) and the routing-weight scale fused into the epilogue.
//
// Orientation (weights on the M side): D[weight row, token] = sum_k W[row, k] x[token, k].
//   A = 128 stored weight rows x 64 reduction elements: one contiguous 16 KB
//       run of the packed layout (packing.h), already in the 64-byte-swizzled
//       K-major form, fetched with one bulk copy;
//   B = N tokens x 64 elements of the permuted activations (x_perm for the
//       up projection, h for the down projection), fetched by a tensor-map
//       copy with the 128-byte swizzle; rows past an expert's segment belong
//       to the next expert or are zero-filled past the buffer, and are masked
//       in the epilogue;
//   D = 128 TMEM lanes x N fp32 columns, two buffers so that the epilogue of
//       one tile overlaps the main loop of the next.
// Tiles: (expert, reduction split, 128-row block, token tile), token tile
// fastest so that concurrent CTAs share the weight block through L2.
// Warp roles (192 threads, one persistent CTA per SM): warp 0 = producer (one
// thread issues the copies), warp 1 = tensor-memory owner and MMA issuer (one
// thread), warps 2-5 = epilogue (one TMEM lane per thread).
// The SwiGLU up-projection's stored rows interleave 8 gate and 8 up rows, so a
// thread holding a gate row finds the matching up row 8 lanes away.
// Every wait is bounded; a wait that gives up sets kErrWaitTimeout in the
// layer's error word and the CTA drains its copies and MMAs and returns.
#include "common.cuh"
#include "kernels.cuh"
#include "packing.h"
#include "tc.cuh"
#include "tc_tiles.cuh"
#include "tile_trace.cuh"

namespace moe {

namespace {

constexpr int kTcThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kATileBytes = 16384;  // 128 rows x 64 bf16
constexpr int kMaxTcStages = 8;
constexpr int kTcSmemBudget = 200 * 1024;

enum Phase { kUp = 0, kDown = 1 };

template <int PHASE, bool GATED>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_kernel(const ExpertTables tab, const ExpertArgs a, const TcGeom geo,
              const __grid_constant__ CUtensorMap bmap) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full_bar[kMaxTcStages], empty_bar[kMaxTcStages];
    __shared__ uint64_t tfull_bar[2], tempty_bar[2], done_bar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_act[kMaxExperts], s_off[kMaxExperts], s_q[kMaxExperts];
    __shared__ long long s_prefix[kMaxExperts + 1];
    __shared__ int s_nact;
    __shared__ volatile int s_abort;
    __shared__ float s_w[kEpiWarps][kTcMaxTileTokens];  // down: routing weights of the tile

    // 1024-byte aligned operand area (swizzle atoms are address-based)
    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    uint8_t *a_slots = smem;
    uint8_t *b_slots = smem + geo.stages * kATileBytes;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    MOE_TRACE_ENTRY(PHASE);
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // the whole warp lists the tiles (one round trip for the offsets)
        const int n_listed = tc_list_tiles(a, geo, s_act, s_off, s_q, s_prefix, lane);
        if (lane == 0) {
            s_nact = n_listed;
            s_abort = 0;
            for (int i = 0; i < geo.stages; ++i) {
                mbar_init(&full_bar[i], 1);
                mbar_init(&empty_bar[i], 1);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(&tfull_bar[i], 1);
                mbar_init(&tempty_bar[i], kEpiWarps);
            }
            mbar_init(&done_bar, 1);
            fence_barrier_init();
        }
    }
    if (warp == 1) tmem_alloc(&s_tmem, geo.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s_tmem;
    const int nact = s_nact;
    const long long total = nact ? s_prefix[nact] : 0;

    uint32_t last_parity[kMaxTcStages];
    bool used[kMaxTcStages];
    for (int i = 0; i < kMaxTcStages; ++i) used[i] = false;
    if (warp == 0) {
        // ======================= producer =======================================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int cur = 0;  // expert of the last tile (a role's tiles come in order)
            for (long long u = blockIdx.x; u < total && !s_abort; u += gridDim.x) {
                const TcTile t = tc_tile(u, s_prefix, s_act, s_off, s_q, nact, geo, cur);
                const uint8_t *w = static_cast<const uint8_t *>(PHASE == kUp ? tab.w1[t.e] : tab.w2[t.e]);
                const int brow = t.off + t.tt * geo.N;
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1u)) {
                        flag_error(a.err, kErrWaitTimeout);
                        s_abort = 1;
                        break;
                    }
                    mbar_arrive_expect_tx(&full_bar[stage], kATileBytes + geo.b_bytes);
                    const size_t blk = static_cast<size_t>(kb) * geo.rg + 8 * t.rb;
                    bulk_g2s(a_slots + stage * kATileBytes, w + blk * kBlockBytes, kATileBytes,
                             &full_bar[stage]);
                    tma_load_2d(b_slots + stage * geo.b_bytes, &bmap, kb * 64, brow, &full_bar[stage]);
                    used[stage] = true;
                    last_parity[stage] = phase;
                    if (++stage == geo.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ======================= MMA issuer =====================================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int ntile = 0;
            int cur = 0;  // expert of the last tile (a role's tiles come in order)
            for (long long u = blockIdx.x; u < total && !s_abort; u += gridDim.x, ++ntile) {
                const TcTile t = tc_tile(u, s_prefix, s_act, s_off, s_q, nact, geo, cur);
                const int buf = ntile & 1;
                const uint32_t use_parity = (ntile >> 1) & 1;
                if (!mbar_wait_spin(&tempty_bar[buf], use_parity ^ 1u)) {
                    flag_error(a.err, kErrWaitTimeout);
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(buf * geo.N);
                // the last token tile of an expert may be partly empty: issue the
                // MMAs with N rounded up to the 16 tokens that hold data
                const int n_valid = min(geo.N, (t.q - t.tt * geo.N + 15) / 16 * 16);
                const uint32_t idesc = idesc_bf16_f32(128, n_valid);
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (!mbar_wait_spin(&full_bar[stage], phase)) {
                        flag_error(a.err, kErrWaitTimeout);
                        s_abort = 1;
                        break;
                    }
                    if (kb == t.kb0) MOE_TRACE_TILE_FIRST(PHASE, ntile, t.e, t.tt, n_valid, t.rb);
                    if (kb == t.kb1 - 1) MOE_TRACE_TILE_LAST(PHASE, ntile);
                    tc_fence_after();
                    const uint32_t abase = smem_u32(a_slots + stage * kATileBytes);
                    const uint32_t bbase = smem_u32(b_slots + stage * geo.b_bytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = smem_desc(abase + (kk >> 1) * 512 + (kk & 1) * 32, 16, 1024,
                                                      kLayoutSw64);
                        const uint64_t bd = smem_desc(bbase + kk * 32, 16, 1024, kLayoutSw128);
                        tc_mma(d, ad, bd, idesc, (kb > t.kb0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit(&empty_bar[stage]);  // slot free once these MMAs have read it
                    if (++stage == geo.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                tc_commit(&tfull_bar[buf]);  // accumulator ready
            }
            tc_commit(&done_bar);  // every MMA this thread issued has completed
            if (!mbar_wait(&done_bar, 0)) flag_error(a.err, kErrWaitTimeout);
        }
    } else {
        // ======================= epilogue =======================================
        const int lq = warp & 3;            // TMEM lane quarter this warp may access
        const int row_in_tile = lq * 32 + lane;
        int ntile = 0;
        int cur = 0;  // expert of the last tile (a role's tiles come in order)
        for (long long u = blockIdx.x; u < total; u += gridDim.x, ++ntile) {
            // warp-uniform decisions: tcgen05.ld below needs the whole warp
            if (__any_sync(0xffffffffu, s_abort)) break;
            const TcTile t = tc_tile(u, s_prefix, s_act, s_off, s_q, nact, geo, cur);
            const int buf = ntile & 1;
            const uint32_t use_parity = (ntile >> 1) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(&tfull_bar[buf], use_parity))) {
                if (lane == 0) flag_error(a.err, kErrWaitTimeout);
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const int R = t.rb * 128 + row_in_tile;  // stored weight row of this thread
            const int tok0 = t.tt * geo.N;
            const int n_valid = min(geo.N, (t.q - tok0 + 15) / 16 * 16);
            if (PHASE == kDown) tc_stage_weights(a, t.off, tok0, t.q, n_valid, s_w[lq], lane);
            for (int c0 = 0; c0 < n_valid; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem_base + (static_cast<uint32_t>(lq * 32) << 16) +
                              static_cast<uint32_t>(buf * geo.N + c0),
                          v);
                tmem_ld_wait();
                if (PHASE == kUp && GATED) {
                    const int r16 = R & 15;
                    const int f = (R >> 4) * 8 + (r16 & 7);
                    if (geo.splits == 1) {
                        tc_swiglu_store16(v, 1.0f, r16 < 8, static_cast<__nv_bfloat16 *>(a.h), a.p, f, t.off,
                                          tok0 + c0, t.q);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float gv = __uint_as_float(v[j]);
                            const float uv = __shfl_down_sync(0xffffffffu, gv, 8);
                            const int tok = tok0 + c0 + j;
                            if (r16 < 8 && tok < t.q) {
                                const size_t o =
                                    (static_cast<size_t>(t.ks) * a.n_rows_cap + t.off + tok) * a.p + f;
                                a.gate_part[o] = gv;
                                a.up_part[o] = uv;
                            }
                        }
                    }
                } else if (PHASE == kUp) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tok = tok0 + c0 + j;
                        if (tok < t.q) {
                            const int pos = t.off + tok;
                            const float hv = __uint_as_float(v[j]);
                            if (geo.splits == 1)
                                static_cast<__nv_bfloat16 *>(a.h)[static_cast<size_t>(pos) * a.p + R] =
                                    __float2bfloat16_rn(fmaxf(hv, 0.0f));
                            else
                                a.gate_part[(static_cast<size_t>(t.ks) * a.n_rows_cap + pos) * a.p + R] = hv;
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tok = tok0 + c0 + j;
                        if (tok < t.q) {
                            const int pos = t.off + tok;
                            const size_t o = (static_cast<size_t>(t.ks) * a.n_rows_cap + pos) * a.m + R;
                            const float yv = s_w[lq][c0 + j] * __uint_as_float(v[j]);
                            if (a.ypart_bf16)
                                reinterpret_cast<__nv_bfloat16 *>(a.ypart)[o] = __float2bfloat16_rn(yv);
                            else
                                a.ypart[o] = yv;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty_bar[buf]);
        }
    }
    // one barrier for every role; then no copy may still be in flight and the
    // tensor memory is released
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0)
        for (int i = 0; i < geo.stages; ++i)
            if (used[i]) mbar_wait(&full_bar[i], last_parity[i]);
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, geo.tmem_cols);
    }
}

// x_perm[pos] = x[gather[pos] / k] for the permuted rows (16-byte vectors).
// HBM-bound: a block takes kR rows at a time, reads their gather indices once,
// and its threads stride over the 16-byte vectors of the rows with the kR
// rows' loads issued together before the stores.
constexpr int kGatherRows = 4;

__global__ void gather_rows_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ gather,
                                   int rows, int k, int m, uint16_t *__restrict__ xp, uint32_t *err) {
    pdl_wait();
    pdl_trigger();
    const int vec = m / 8;
    for (int r0 = blockIdx.x * kGatherRows; r0 < rows; r0 += gridDim.x * kGatherRows) {
        int fi[kGatherRows];
#pragma unroll
        for (int b = 0; b < kGatherRows; ++b) {
            fi[b] = -1;
            if (r0 + b < rows) {
                const int f = gather[r0 + b];
                if (f >= 0 && f < rows)
                    fi[b] = f;
                else if (threadIdx.x == 0)
                    flag_error(err, kErrGatherIndex);
            }
        }
        for (int v = threadIdx.x; v < vec; v += blockDim.x) {
            uint4 val[kGatherRows];
#pragma unroll
            for (int b = 0; b < kGatherRows; ++b)
                val[b] = fi[b] >= 0 ? ld_nc_v4(x + static_cast<size_t>(fi[b] / k) * m + v * 8)
                                    : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int b = 0; b < kGatherRows; ++b)
                if (r0 + b < rows)
                    *reinterpret_cast<uint4 *>(xp + static_cast<size_t>(r0 + b) * m + v * 8) = val[b];
        }
    }
}

template <int PHASE, bool GATED>
cudaError_t launch_tc_t(const ExpertArgs &a, const TcGeom &g, const CUtensorMap &bmap, int num_sms,
                        cudaStream_t s) {
    if (!tc_tiles_fit(a, g)) return cudaErrorInvalidValue;
    const size_t smem = 1024 + static_cast<size_t>(g.stages) * (kATileBytes + g.b_bytes);
    auto kern = tc_kernel<PHASE, GATED>;
    static int configured = 0;
    if (static_cast<int>(smem) > configured) {
        const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        configured = static_cast<int>(smem);
    }
    return launch_pdl(kern, dim3(num_sms), dim3(kTcThreads), smem, s, *a.tab, a, g, bmap);
}

TcGeom make_tc_geom(int K, int rows, int splits, int N) {
    TcGeom g;
    g.K = K;
    g.rg = rows / 16;
    g.n_rb = rows / 128;
    g.nkb = K / 64;
    g.splits = splits;
    g.N = N;
    g.b_bytes = N * 128;
    int st = kTcSmemBudget / (kATileBytes + g.b_bytes);
    g.stages = st > kMaxTcStages ? kMaxTcStages : st;
    int cols = 32;
    while (cols < 2 * N) cols <<= 1;
    g.tmem_cols = cols;
    g.idesc = idesc_bf16_f32(128, N);
    return g;
}

}  // namespace

cudaError_t launch_gather_rows(const void *x, const int32_t *gather, int rows, int k, int m,
                               void *x_perm, uint32_t *err, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    long long blocks = (rows + kGatherRows - 1) / kGatherRows;
    if (blocks > 152 * 8) blocks = 152 * 8;
    return launch_pdl(gather_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                      static_cast<const uint16_t *>(x), gather, rows, k, m,
                      static_cast<uint16_t *>(x_perm), err);
}

cudaError_t launch_tc_up(const ExpertArgs &a, bool gated, int splits, int N, const CUtensorMap &xmap,
                         int num_sms, cudaStream_t s) {
    const TcGeom g = make_tc_geom(a.m, gated ? 2 * a.p : a.p, splits, N);
    return gated ? launch_tc_t<kUp, true>(a, g, xmap, num_sms, s)
                 : launch_tc_t<kUp, false>(a, g, xmap, num_sms, s);
}

cudaError_t launch_tc_down(const ExpertArgs &a, int splits, int N, const CUtensorMap &hmap,
                           int num_sms, cudaStream_t s) {
    const TcGeom g = make_tc_geom(a.p, a.m, splits, N);
    return launch_tc_t<kDown, false>(a, g, hmap, num_sms, s);
}

}  // namespace moe

MOE_TRACE_READER(moe_tile_trace_tc)
