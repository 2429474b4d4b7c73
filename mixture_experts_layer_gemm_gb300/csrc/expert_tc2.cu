// expert_tc2.cu -- the grouped expert GEMM on CTA pairs (tcgen05 cta_group::2)
// for token tiles of 256, the batch regime's compute-bound case (used for the
// up projection; the down projection measured faster on one CTA per tile).
//
// Why pairs: with one CTA computing a 128 x 256 tile, every 64-deep step
// brings 16 KB of weights and 32 KB of tokens into shared memory and the MMAs
// read 48 KB back out, close to 190 bytes per clock per SM against a shared
// memory that serves about 128: the tensor pipe idles a third of the time.  A
// pair of CTAs on two SMs computes a 256 x 256 tile with one MMA stream: each
// CTA holds 128 weight rows and 128 of the 256 tokens, so per SM the fill
// halves for the tokens and the operand reads drop to 32 KB per step.
//
//   A (per CTA) = its 128 weight rows x 64 reduction elements: one contiguous
//       16 KB run of the packed layout (64-byte swizzle built in), fetched as
//       128 rows of 128 bytes through a tensor map over the weight buffer;
//   B (per CTA) = its 128 tokens x 64 elements of x_perm / h, one tensor-map
//       copy, 128-byte swizzle;
//   D = 128 lanes x 256 fp32 columns in each CTA's tensor memory (rows of its
//       own weight half, all 256 tokens), two buffers (512 columns);
//   the even CTA's MMA thread issues M = 256, N = 256 MMAs that read both
//       CTAs' operands at the same shared-memory offsets.
// Signalling (mbarriers, all waits bounded):
//   full[s]   (even CTA) both CTAs' copies of stage s landed: every copy of
//             the pair completes its bytes on this barrier (the pair form of
//             the tensor copy), and the even CTA's producer arms it with the
//             bytes of both;
//   empty[s]  both CTAs: the pair MMAs that read stage s completed (commit to
//             each CTA's barrier);
//   tfull[b]  both CTAs: accumulator buffer b complete (commit to each);
//   tempty[b] (even CTA) all eight epilogue warps of the pair read buffer b.
// Tiles: (expert, 256-row pair block, 256-token tile), token tile fastest;
// both CTAs of a pair walk the same tile sequence.
// Teardown: the even CTA's producer waits for the last phase of every stage
// it armed (both CTAs' bytes); the odd CTA's producer waits until its last
// stages were consumed by the MMAs (which implies they landed).  Every path reaches the
// final cluster barrier, so neither CTA leaves while the other may still read
// its shared memory or the MMAs may still write its tensor memory.
#include "common.cuh"
#include "kernels.cuh"
#include "packing.h"
#include "tc.cuh"
#include "tc_tiles.cuh"
#include "tile_trace.cuh"

namespace moe {

namespace {

constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kHalfA = 16384;  // 128 weight rows x 64 bf16 per CTA
constexpr int kHalfB = 16384;  // 128 tokens x 64 bf16 per CTA
constexpr int kStageBytes = kHalfA + kHalfB;
constexpr int kMaxStages = 6;
constexpr int kN = 256;               // tokens per pair tile
constexpr uint32_t kTmemCols = 512;   // two accumulators of 256 columns

// Up projection only: the down projection runs on one CTA per tile, which
// measured faster for it.
template <bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
    tc2_kernel(const ExpertTables tab, const ExpertArgs a, const TcGeom geo,
               const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
    __shared__ uint64_t tfull_bar[2], tempty_bar[2], done_bar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_act[kMaxExperts], s_off[kMaxExperts], s_q[kMaxExperts];
    __shared__ long long s_prefix[kMaxExperts + 1];
    __shared__ int s_nact;
    __shared__ volatile int s_abort;

    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const long long pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    MOE_TRACE_ENTRY(0);
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
                mbar_init(&tempty_bar[i], 2 * kEpiWarps);
            }
            mbar_init(&done_bar, 1);
            fence_barrier_init();
        }
    }
    if (warp == 1) tmem_alloc_pair(&s_tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA arrive
    tc_fence_after();
    const uint32_t tmem_base = s_tmem;
    const int nact = s_nact;
    const long long total = nact ? s_prefix[nact] : 0;

    uint32_t last_parity[kMaxStages];
    bool used[kMaxStages];
    for (int i = 0; i < kMaxStages; ++i) used[i] = false;
    if (warp == 0) {
        // ======================= producer (both CTAs) ===========================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            const uint8_t *wbase = static_cast<const uint8_t *>(a.wbase);
            int cur = 0;  // expert of the last tile (a role's tiles come in order)
            for (long long u = pair; u < total && !s_abort; u += npairs) {
                const TcTile t = tc_tile(u, s_prefix, s_act, s_off, s_q, nact, geo, cur);
                const uint8_t *w = static_cast<const uint8_t *>(tab.w1[t.e]);
                const int nv = min(kN, (t.q - t.tt * kN + 31) / 32 * 32);
                const int brow = t.off + t.tt * kN + static_cast<int>(rank) * (nv / 2);
                const int rb = 2 * t.rb + static_cast<int>(rank);  // this CTA's 128-row block
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (!mbar_wait_cluster(&empty_bar[stage], phase ^ 1u)) {
                        flag_error(a.err, kErrWaitTimeout);
                        s_abort = 1;
                        break;
                    }
                    uint8_t *st = smem + stage * kStageBytes;
                    const uint32_t fb = mapa_shared(smem_u32(&full_bar[stage]), 0);  // the even CTA's
                    if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * kStageBytes);
                    const size_t blk = static_cast<size_t>(kb) * geo.rg + 8 * rb;
                    const int arow = static_cast<int>(((w - wbase) + blk * kBlockBytes) >> 7);  // 128-byte rows
                    tma_load_2d_pair(st, &amap, 0, arow, fb);
                    tma_load_2d_pair(st + kHalfA, &bmap, kb * 64, brow, fb);
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
        if (lane == 0 && leader) {
            // =================== MMA issuer (even CTA) ==========================
            int stage = 0;
            uint32_t phase = 0;
            int ntile = 0;
            int cur = 0;  // expert of the last tile (a role's tiles come in order)
            for (long long u = pair; u < total && !s_abort; u += npairs, ++ntile) {
                const TcTile t = tc_tile(u, s_prefix, s_act, s_off, s_q, nact, geo, cur);
                const int buf = ntile & 1;
                const uint32_t use_parity = (ntile >> 1) & 1;
                if (!mbar_wait_cluster_spin(&tempty_bar[buf], use_parity ^ 1u)) {
                    flag_error(a.err, kErrWaitTimeout);
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(buf * kN);
                const int nv = min(kN, (t.q - t.tt * kN + 31) / 32 * 32);
                const uint32_t idesc = idesc_bf16_f32(256, nv);
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (!mbar_wait_cluster_spin(&full_bar[stage], phase)) {
                        flag_error(a.err, kErrWaitTimeout);
                        s_abort = 1;
                        break;
                    }
                    if (kb == t.kb0) MOE_TRACE_TILE_FIRST(0, ntile, t.e, t.tt, nv, t.rb);
                    if (kb == t.kb1 - 1) MOE_TRACE_TILE_LAST(0, ntile);
                    tc_fence_after();
                    const uint32_t abase = smem_u32(smem + stage * kStageBytes);
                    const uint32_t bbase = abase + kHalfA;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = smem_desc(abase + (kk >> 1) * 512 + (kk & 1) * 32, 16, 1024,
                                                      kLayoutSw64);
                        const uint64_t bd = smem_desc(bbase + kk * 32, 16, 1024, kLayoutSw128);
                        tc_mma_pair(d, ad, bd, idesc, (kb > t.kb0 || kk > 0) ? 1u : 0u);
                    }
                    const uint32_t eb = smem_u32(&empty_bar[stage]);
                    tc_commit_pair(eb);                   // this CTA's slot is free
                    tc_commit_pair(mapa_shared(eb, 1));   // and the odd CTA's
                    if (++stage == geo.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                const uint32_t tb = smem_u32(&tfull_bar[buf]);
                tc_commit_pair(tb);
                tc_commit_pair(mapa_shared(tb, 1));
            }
            tc_commit_pair(smem_u32(&done_bar));  // every pair MMA issued has completed
            if (!mbar_wait(&done_bar, 0)) flag_error(a.err, kErrWaitTimeout);
        }
    } else {
        // ======================= epilogue (both CTAs) ===========================
        const int lq = warp & 3;
        const int row_in_tile = lq * 32 + lane;
        int ntile = 0;
        int cur = 0;  // expert of the last tile (a role's tiles come in order)
        for (long long u = pair; u < total; u += npairs, ++ntile) {
            if (__any_sync(0xffffffffu, s_abort)) break;
            const TcTile t = tc_tile(u, s_prefix, s_act, s_off, s_q, nact, geo, cur);
            const int buf = ntile & 1;
            const uint32_t use_parity = (ntile >> 1) & 1;
            if (!__all_sync(0xffffffffu, mbar_wait_cluster(&tfull_bar[buf], use_parity))) {
                if (lane == 0) flag_error(a.err, kErrWaitTimeout);
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const int R = (2 * t.rb + static_cast<int>(rank)) * 128 + row_in_tile;  // stored weight row
            const int tok0 = t.tt * kN;
            const int nv = min(kN, (t.q - tok0 + 31) / 32 * 32);
            for (int c0 = 0; c0 < nv; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem_base + (static_cast<uint32_t>(lq * 32) << 16) +
                              static_cast<uint32_t>(buf * kN + c0),
                          v);
                tmem_ld_wait();
                if (GATED) {
                    const int r16 = R & 15;
                    tc_swiglu_store16(v, 1.0f, r16 < 8, static_cast<__nv_bfloat16 *>(a.h), a.p,
                                      (R >> 4) * 8 + (r16 & 7), t.off, tok0 + c0, t.q);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int tok = tok0 + c0 + j;
                        if (tok < t.q)
                            static_cast<__nv_bfloat16 *>(a.h)[static_cast<size_t>(t.off + tok) * a.p + R] =
                                __float2bfloat16_rn(fmaxf(__uint_as_float(v[j]), 0.0f));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[buf]), 0));
        }
    }
    // one barrier per CTA, the producer drains its copies, then one barrier of
    // the pair: after it no CTA touches the other's memory and the pair's
    // tensor memory is released together
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0)
        for (int i = 0; i < geo.stages; ++i)
            if (used[i]) {
                if (leader)
                    mbar_wait_cluster(&full_bar[i], last_parity[i]);
                else
                    mbar_wait_cluster(&empty_bar[i], last_parity[i]);
            }
    __syncwarp();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

template <bool GATED>
cudaError_t launch_t(const ExpertArgs &a, const TcGeom &g, const CUtensorMap &amap, const CUtensorMap &bmap,
                     int num_sms, cudaStream_t s) {
    if (!tc_tiles_fit(a, g)) return cudaErrorInvalidValue;
    const size_t smem = 1024 + static_cast<size_t>(g.stages) * kStageBytes;
    auto kern = tc2_kernel<GATED>;
    static int configured = 0, pairs = 0;
    if (static_cast<int>(smem) > configured) {
        const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        configured = static_cast<int>(smem);
        pairs = 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    if (pairs == 0) {  // pairs that can be resident at once: one persistent pair each
        cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1));
        cfg.numAttrs = 1;
        int n = 0;
        const cudaError_t err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (err != cudaSuccess) return err;
        pairs = n < 1 ? 1 : (n > num_sms / 2 ? num_sms / 2 : n);
    }
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, *a.tab, a, g, amap, bmap);
}

// K: reduction length (multiple of 64); rows: stored rows (multiple of 256).
TcGeom make_geom(int K, int rows) {
    TcGeom g;
    g.K = K;
    g.rg = rows / 16;
    g.n_rb = rows / 256;  // pair blocks
    g.nkb = K / 64;
    g.splits = 1;
    g.N = kN;
    g.b_bytes = kHalfB;
    g.stages = kMaxStages;
    g.tmem_cols = static_cast<int>(kTmemCols);
    g.idesc = idesc_bf16_f32(256, kN);
    return g;
}

}  // namespace

cudaError_t launch_tc2_up(const ExpertArgs &a, bool gated, const CUtensorMap &wmap, const CUtensorMap &xmap_half,
                          int num_sms, cudaStream_t s) {
    const TcGeom g = make_geom(a.m, gated ? 2 * a.p : a.p);
    return gated ? launch_t<true>(a, g, wmap, xmap_half, num_sms, s)
                 : launch_t<false>(a, g, wmap, xmap_half, num_sms, s);
}

}  // namespace moe

MOE_TRACE_READER(moe_tile_trace_tc2)
