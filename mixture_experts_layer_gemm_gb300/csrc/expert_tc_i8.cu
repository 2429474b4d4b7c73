// expert_tc_i8.cu -- grouped expert GEMM on the tensor cores with int8 weights
// (per-output-channel symmetric codes; DeepSpeed-Inference article, part 4:
// INT8 weights dequantised inside the kernel).
//
// Numerics.  Down projection: the codes q (|q| <= 127) are exact in bf16, so
// the tensor cores compute sum_k q[row, k] h[token, k] in fp32 from bf16
// operands, and the epilogue multiplies by the row's scale -- the same "scale
// after the dot product" as the int8 weight-streaming GEMV.  Up projection:
// the operands are fp16, which widens codes in a third of the instructions of
// bf16 (the converters bound this kernel at small token tiles): the A operand
// is 1152 + q (exact; fp16 bit pattern 0x6400 | (q + 128)), the B operand the
// token row times 2^-s (gather_rows_f16_kernel: exact for every value within a
// factor 2^31 of the row's largest), and the epilogue forms
// (acc - 1152 * sum_k x'[token, k]) * 2^s * scale[row], the row sum x' taken
// over the tile's reduction split.
//
// Shared-memory traffic, not the tensor pipe, bounds the bf16 grouped GEMM
// (TMA fill + operand reads).  Widening int8 to bf16 in shared memory would
// add a write and a read of twice the bytes, so the widened tile goes to
// tensor memory instead and the MMA takes its A operand from there:
//   stage (128 reduction elements): A8 = 128 weight rows x 128 int8 (one
//     contiguous 16 KB run of the packed layout, one bulk copy) and
//     B = N tokens x 128 bf16 (two tensor-map copies of 64 columns, 128-byte
//     swizzle);
//   converter warps (two per TMEM lane quarter; a thread takes one weight row
//     and one half of the stage's reduction range) widen 64 codes to 32
//     fp16x2 (up) or bf16x2 (down) words and store them to an A buffer in
//     tensor memory (buffers of 64 columns);
//   an MMA thread issues 8 MMAs of K = 16 per stage, A from tensor memory,
//     B from shared memory, D = 128 lanes x N fp32 columns (two buffers, one
//     accumulator per MMA issuer in each).
// Tensor memory: D buffers at columns [0, 2N) with one issuer (N <= 192) or
// [0, 4N) with two (N <= 96; buffer b, issuer i at (2b + i) N), A buffers of
// 64 columns from the next multiple of 64 up to column 512 (two at N = 192,
// six at N = 32); 512 columns allocated (one CTA per SM).
// Warp roles (480 threads): 0 producer, 1 tensor-memory owner + MMA issuer,
// 2-5 epilogue, 6-13 converters, 14 second MMA issuer.  A small-N MMA stream
// from one thread is paced by that thread's instructions, so where four
// accumulators fit below the A buffers (N <= 96) the K blocks of a tile
// alternate between the two issuers, each with its own accumulator, and the
// epilogue adds the two.  Every wait is bounded; a wait that gives up
// sets kErrWaitTimeout and the CTA drains and returns.
#include "common.cuh"
#include "kernels.cuh"
#include "packing.h"
#include "tc.cuh"
#include "tc_tiles.cuh"

namespace moe {

namespace {

constexpr int kThreads = 480;
constexpr int kMma2Warp = 14;  // second MMA issuer
constexpr int kEpiWarps = 4;
constexpr int kCvtWarps = 8;  // two per TMEM lane quarter, one K half each
constexpr int kA8Bytes = 16384;  // 128 rows x 128 int8
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 200 * 1024;
constexpr uint32_t kTmemCols = 512;
// A buffers (64 columns each) fill the columns above the accumulators, from
// the first multiple of 64 at or past them: two at N = 192, up to seven at
// N = 16, so that the converters can run ahead of the MMAs.
constexpr int kMaxABufs = 7;
constexpr uint32_t kTwoIssuerCols = 384;  // two issuers while their four D buffers fit here
static_assert(2 * kTcI8MaxN + 2 * 64 <= kTmemCols, "tensor-memory columns: two A buffers at N = max");

enum Phase { kUp = 0, kDown = 1 };

// The fp16 token rows of a tile (up projection): the scale of each row (into
// sc) and its sum over reduction split ks (into sm), one lane per token; zero
// for tokens past the segment.
__device__ __forceinline__ void stage_row_factors(const ExpertArgs &a, int off, int tok0, int q, int n, int ks,
                                                  float *sc, float *sm, int lane) {
    __syncwarp();  // every lane is past its reads of the previous tile's factors
    for (int c = lane; c < n; c += 32) {
        const int tok = tok0 + c;
        float f = 0.0f, sum = 0.0f;
        if (tok < q) {
            const int pos = off + tok;
            f = a.x_scale[pos];
            sum = a.x_sum[static_cast<size_t>(ks) * a.xsum_stride + pos];
        }
        sc[c] = f;
        sm[c] = sum;
    }
    __syncwarp();
}

template <int PHASE, bool GATED>
__global__ void __launch_bounds__(kThreads, 1)
    tc_i8_kernel(const ExpertTables tab, const ExpertArgs a, const TcGeom geo,
                 const __grid_constant__ CUtensorMap bmap) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
    __shared__ uint64_t afull_bar[kMaxABufs], aempty_bar[kMaxABufs];
    __shared__ uint64_t tfull_bar[2], tempty_bar[2], done_bar[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_act[kMaxExperts], s_off[kMaxExperts], s_q[kMaxExperts];
    __shared__ long long s_prefix[kMaxExperts + 1];
    __shared__ int s_nact;
    __shared__ volatile int s_abort;
    // down: routing weights of the tile's tokens; up: the scales of their fp16 rows
    __shared__ float s_w[kEpiWarps][kTcMaxTileTokens];
    __shared__ float s_xs[kEpiWarps][kTcMaxTileTokens];  // up: the rows' sums over the tile's split

    const uint32_t raw_s = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
    const int stage_bytes = kA8Bytes + 2 * geo.b_bytes;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // MMA issuers: two where both accumulator buffers of both fit below the A buffers
    const int nis = (4 * geo.N <= static_cast<int>(kTwoIssuerCols)) ? 2 : 1;
    const uint32_t a_col0 = static_cast<uint32_t>((2 * nis * geo.N + 63) / 64 * 64);
    const int nab = min(kMaxABufs, static_cast<int>((kTmemCols - a_col0) / 64));
    // The weight and scale pointers, copied from the launch parameters into
    // shared memory before the wait: the producer and the epilogue look them up
    // at every tile, and a dynamically indexed parameter read can miss the
    // constant cache.  Scales: gate rows s1, up rows s3 (SwiGLU); s1 (ReLU up);
    // s2 (down).
    __shared__ const void *s_wptr[kExpertTableMax];
    __shared__ const float *s_sptr[2][kExpertTableMax];
    if (warp == 2)
        for (int e = lane; e < kExpertTableMax; e += 32) {
            s_wptr[e] = PHASE == kUp ? tab.w1[e] : tab.w2[e];
            s_sptr[0][e] = PHASE == kUp ? tab.s1[e] : tab.s2[e];
            s_sptr[1][e] = tab.s3[e];
        }
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
                mbar_init(&empty_bar[i], 1 + kCvtWarps);  // MMA commit + converter warps
            }
            for (int i = 0; i < nab; ++i) {
                mbar_init(&afull_bar[i], kCvtWarps);
                mbar_init(&aempty_bar[i], 1);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(&tfull_bar[i], nis);  // one commit per issuer
                mbar_init(&tempty_bar[i], kEpiWarps);
                mbar_init(&done_bar[i], 1);
            }
            fence_barrier_init();
        }
    }
    if (warp == 1) tmem_alloc(&s_tmem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s_tmem;
    const int nact = s_nact;
    const long long total = nact ? s_prefix[nact] : 0;

    uint32_t last_parity[kMaxStages];
    bool used[kMaxStages];
    for (int i = 0; i < kMaxStages; ++i) used[i] = false;
    if (warp == 0) {
        // ======================= producer =======================================
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int cur = 0;  // expert of the last tile (a role's tiles come in order)
            for (long long u = blockIdx.x; u < total && !s_abort; u += gridDim.x) {
                const TcTile t = tc_tile(u, s_prefix, s_act, s_off, s_q, nact, geo, cur);
                const uint8_t *w = static_cast<const uint8_t *>(s_wptr[t.e]);
                const int brow = t.off + t.tt * geo.N;
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1u)) {
                        flag_error(a.err, kErrWaitTimeout);
                        s_abort = 1;
                        break;
                    }
                    uint8_t *st = smem + stage * stage_bytes;
                    mbar_arrive_expect_tx(&full_bar[stage], kA8Bytes + 2 * geo.b_bytes);
                    const size_t blk = static_cast<size_t>(kb) * geo.rg + 8 * t.rb;
                    bulk_g2s(st, w + blk * kBlockBytes, kA8Bytes, &full_bar[stage]);
                    tma_load_2d(st + kA8Bytes, &bmap, kb * 128, brow, &full_bar[stage]);
                    tma_load_2d(st + kA8Bytes + geo.b_bytes, &bmap, kb * 128 + 64, brow, &full_bar[stage]);
                    used[stage] = true;
                    last_parity[stage] = phase;
                    if (++stage == geo.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1 || warp == kMma2Warp) {
        // ======================= MMA issuers ====================================
        // issuer `me` takes the K blocks kb0 + me, kb0 + me + nis, ... of every
        // tile into its own accumulator; both walk every stage and A buffer so
        // that their ring positions and phases agree
        const int me = warp == 1 ? 0 : 1;
        if (lane == 0 && me < nis) {
            int stage = 0, abuf = 0;
            uint32_t phase = 0, aphase = 0;
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
                const uint32_t d = tmem_base + static_cast<uint32_t>((buf * nis + me) * geo.N);
                const int n_valid = min(geo.N, (t.q - t.tt * geo.N + 15) / 16 * 16);
                const uint32_t idesc = PHASE == kUp ? idesc_f16_f32(128, n_valid) : idesc_bf16_f32(128, n_valid);
                uint32_t accum = 0;  // this issuer's first block of the tile starts the sum
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (((kb - t.kb0) & (nis - 1)) != me) {  // the other issuer's block (nis is 1 or 2)
                        if (++stage == geo.stages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        if (++abuf == nab) {
                            abuf = 0;
                            aphase ^= 1u;
                        }
                        continue;
                    }
                    if (!mbar_wait_spin(&full_bar[stage], phase) || !mbar_wait_spin(&afull_bar[abuf], aphase)) {
                        flag_error(a.err, kErrWaitTimeout);
                        s_abort = 1;
                        break;
                    }
                    tc_fence_after();
                    // the stage's two 64-column token halves; a half's K slices are
                    // 32 bytes apart, +2 in the descriptor's address field (the
                    // shared-memory addresses stay far below its 256 KB range, so
                    // the field never carries).  One MMA thread issues every MMA,
                    // so its loop is kept to an add per MMA.
                    const uint32_t bbase = smem_u32(smem + stage * stage_bytes + kA8Bytes);
                    const uint64_t bd0 = smem_desc(bbase, 16, 1024, kLayoutSw128);
                    const uint64_t bd1 = smem_desc(bbase + geo.b_bytes, 16, 1024, kLayoutSw128);
                    const uint32_t acol = tmem_base + a_col0 + static_cast<uint32_t>(abuf * 64);
                    tc_mma_tmem_a(d, acol, bd0, idesc, accum);
                    accum = 1;
#pragma unroll
                    for (int kk = 1; kk < 8; ++kk)
                        tc_mma_tmem_a(d, acol + kk * 8, (kk < 4 ? bd0 : bd1) + 2u * (kk & 3), idesc, 1u);
                    tc_commit(&empty_bar[stage]);   // B slot read
                    tc_commit(&aempty_bar[abuf]);   // A buffer read
                    if (++stage == geo.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (++abuf == nab) {
                        abuf = 0;
                        aphase ^= 1u;
                    }
                }
                tc_commit(&tfull_bar[buf]);
            }
            tc_commit(&done_bar[me]);
            if (!mbar_wait(&done_bar[me], 0)) flag_error(a.err, kErrWaitTimeout);
        }
    } else if (warp < 2 + kEpiWarps) {
        // ======================= epilogue =======================================
        const int lq = warp & 3;
        const int row_in_tile = lq * 32 + lane;
        int ntile = 0;
        int cur = 0;  // expert of the last tile (a role's tiles come in order)
        for (long long u = blockIdx.x; u < total; u += gridDim.x, ++ntile) {
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
            // per-row scale: SwiGLU gate rows use s1, up rows s3 (feature f);
            // ReLU rows s1[R]; down-projection rows s2[R]
            const int r16 = R & 15;
            const int f = (R >> 4) * 8 + (r16 & 7);
            float scale;
            if (PHASE == kUp && GATED)
                scale = s_sptr[r16 < 8 ? 0 : 1][t.e][f];
            else
                scale = s_sptr[0][t.e][R];
            const int tok0 = t.tt * geo.N;
            const int n_valid = min(geo.N, (t.q - tok0 + 15) / 16 * 16);
            if (PHASE == kDown)
                tc_stage_weights(a, t.off, tok0, t.q, n_valid, s_w[lq], lane);
            else
                stage_row_factors(a, t.off, tok0, t.q, n_valid, t.ks, s_w[lq], s_xs[lq], lane);
            // the tile's accumulators: the second issuer's holds a partial sum
            // when the tile has two or more K blocks (a warp-uniform choice)
            const uint32_t dcol = (static_cast<uint32_t>(lq * 32) << 16) + static_cast<uint32_t>(buf * nis * geo.N);
            const bool two = nis == 2 && t.kb1 - t.kb0 >= 2;
            for (int c0 = 0; c0 < n_valid; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem_base + dcol + static_cast<uint32_t>(c0), v);
                if (two) {
                    uint32_t v1[16];
                    tmem_ld16(tmem_base + dcol + static_cast<uint32_t>(geo.N + c0), v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + __uint_as_float(v1[j]));
                } else {
                    tmem_ld_wait();
                }
                if (PHASE == kUp) {  // fp16 operands: take out the code bias, undo the token scales
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[j] = __float_as_uint((__uint_as_float(v[j]) - kI8F16Bias * s_xs[lq][c0 + j]) *
                                               s_w[lq][c0 + j]);
                }
                if (PHASE == kUp && GATED) {
                    if (geo.splits == 1) {
                        tc_swiglu_store16(v, scale, r16 < 8, static_cast<__nv_bfloat16 *>(a.h), a.p, f, t.off,
                                          tok0 + c0, t.q);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float gv = __uint_as_float(v[j]) * scale;
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
                            const float hv = __uint_as_float(v[j]) * scale;
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
                            const float yv = s_w[lq][c0 + j] * (__uint_as_float(v[j]) * scale);
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
    } else {
        // ======================= converters =====================================
        // thread = one weight row r of the 128-row block and one K half hk of
        // the stage: row group r / 16, atom half G = (r % 16) / 8, row g = r % 8
        // inside the 512-byte atoms; codes 64 hk .. 64 hk + 63 are atom hk
        const int lq = warp & 3;
        const int hk = (warp - 2 - kEpiWarps) >> 2;
        const int r = lq * 32 + lane;
        const int rgl = r >> 4, G = (r >> 3) & 1, g = r & 7;
        const uint32_t row_off = static_cast<uint32_t>(rgl * kBlockBytes + G * 1024 + hk * 512);
        int stage = 0, abuf = 0;
        uint32_t phase = 0, aphase = 0;
        int cur = 0;  // expert of the last tile (a role's tiles come in order)
        for (long long u = blockIdx.x; u < total; u += gridDim.x) {
            if (__any_sync(0xffffffffu, s_abort)) break;
            const TcTile t = tc_tile(u, s_prefix, s_act, s_off, s_q, nact, geo, cur);
            bool ok = true;
            for (int kb = t.kb0; kb < t.kb1; ++kb) {
                // warp-uniform waits: tcgen05.st below needs the whole warp
                if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[stage], phase)) ||
                    !__all_sync(0xffffffffu, mbar_wait(&aempty_bar[abuf], aphase ^ 1u))) {
                    if (lane == 0) flag_error(a.err, kErrWaitTimeout);
                    s_abort = 1;
                    ok = false;
                    break;
                }
                const uint32_t a8_s = smem_u32(smem + stage * stage_bytes) + row_off;
                uint32_t wv[32];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 q = lds_v4(a8_s + atom_chunk_offset(g, c));
                    // codes 16c .. 16c + 15 of this half -> columns 8c .. 8c + 7
                    if (PHASE == kUp) {  // fp16 1152 + code, three instructions per four codes
                        i8x4_to_f16x2x2_biased(q.x, wv[c * 8 + 0], wv[c * 8 + 1]);
                        i8x4_to_f16x2x2_biased(q.y, wv[c * 8 + 2], wv[c * 8 + 3]);
                        i8x4_to_f16x2x2_biased(q.z, wv[c * 8 + 4], wv[c * 8 + 5]);
                        i8x4_to_f16x2x2_biased(q.w, wv[c * 8 + 6], wv[c * 8 + 7]);
                    } else {
                        i8x4_to_bf16x2x2(q.x, wv[c * 8 + 0], wv[c * 8 + 1]);
                        i8x4_to_bf16x2x2(q.y, wv[c * 8 + 2], wv[c * 8 + 3]);
                        i8x4_to_bf16x2x2(q.z, wv[c * 8 + 4], wv[c * 8 + 5]);
                        i8x4_to_bf16x2x2(q.w, wv[c * 8 + 6], wv[c * 8 + 7]);
                    }
                }
                tc_fence_after();
                tmem_st32(tmem_base + (static_cast<uint32_t>(lq * 32) << 16) + a_col0 +
                              static_cast<uint32_t>(abuf * 64 + hk * 32),
                          wv);
                tmem_st_wait();
                tc_fence_before();
                fence_proxy_async_smem();  // our reads of the A8 slot precede its next copy
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&afull_bar[abuf]);
                    mbar_arrive(&empty_bar[stage]);
                }
                if (++stage == geo.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
                if (++abuf == nab) {
                    abuf = 0;
                    aphase ^= 1u;
                }
            }
            if (!ok) break;
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
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

constexpr int kGatherThreads = 128;
constexpr int kMaxSumSplits = 4;  // reduction splits of an int8 tensor-core up projection

// One CTA per permuted row (grid-stride): the row's largest magnitude, then
// the fp16 row under the power-of-two scale that puts it in [2^14, 2^15), the
// scale, and the scaled row's sum over each reduction split (fixed order: each
// thread in element order, the warps' sums in warp order).
__global__ void __launch_bounds__(kGatherThreads)
    gather_rows_f16_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ gather, int rows, int k,
                           int m, int splits, uint16_t *__restrict__ xp, float *__restrict__ x_scale,
                           float *__restrict__ x_sum, int xsum_stride, uint32_t *err) {
    pdl_wait();
    pdl_trigger();
    __shared__ float s_red[kGatherThreads / 32][kMaxSumSplits];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int vec = m / 8;     // 16-byte chunks of a row
    const int nkb = m / 128;   // reduction blocks of 128 elements
    for (int r = blockIdx.x; r < rows; r += gridDim.x) {
        const int f = gather[r];
        const bool ok = f >= 0 && f < rows;
        if (!ok && tid == 0) flag_error(err, kErrGatherIndex);
        const uint16_t *src = x + static_cast<size_t>(ok ? f / k : 0) * m;  // a valid row stands in
        float mx = 0.0f;
        for (int v = tid; v < vec; v += kGatherThreads) {
            const uint4 q = ld_nc_v4(src + v * 8);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fmaxf(fabsf(bf16lo(w[i])), fabsf(bf16hi(w[i]))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) s_red[warp][0] = mx;
        __syncthreads();
#pragma unroll
        for (int w = 0; w < kGatherThreads / 32; ++w) mx = fmaxf(mx, s_red[w][0]);
        const int sh = f16_row_shift(mx);
        const float down = pow2f(-sh);
        __syncthreads();  // s_red is reused for the sums
        float sum[kMaxSumSplits];
#pragma unroll
        for (int sp = 0; sp < kMaxSumSplits; ++sp) sum[sp] = 0.0f;
        for (int v = tid; v < vec; v += kGatherThreads) {
            const int kb = v / 16;  // 16 chunks of 8 elements per reduction block
            int sp = 0;
            while (sp + 1 < splits && kb >= (nkb * (sp + 1)) / splits) ++sp;
            const uint4 q = ld_nc_v4(src + v * 8);
            uint32_t w[4] = {q.x, q.y, q.z, q.w};
            float part = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __half2 hv = __floats2half2_rn(bf16lo(w[i]) * down, bf16hi(w[i]) * down);
                part += __low2float(hv) + __high2float(hv);
                w[i] = *reinterpret_cast<const uint32_t *>(&hv);
            }
#pragma unroll
            for (int i = 0; i < kMaxSumSplits; ++i)
                if (i == sp) sum[i] += part;
            *reinterpret_cast<uint4 *>(xp + static_cast<size_t>(r) * m + v * 8) = make_uint4(w[0], w[1], w[2], w[3]);
        }
#pragma unroll
        for (int sp = 0; sp < kMaxSumSplits; ++sp) {
            const float v = warp_sum(sum[sp]);
            if (lane == 0) s_red[warp][sp] = v;
        }
        __syncthreads();
        if (tid < splits) {
            float tot = 0.0f;
#pragma unroll
            for (int w = 0; w < kGatherThreads / 32; ++w) tot += s_red[w][tid];
            x_sum[static_cast<size_t>(tid) * xsum_stride + r] = tot;
        }
        if (tid == 0) x_scale[r] = pow2f(sh);
        __syncthreads();
    }
}

template <int PHASE, bool GATED>
cudaError_t launch_t(const ExpertArgs &a, const TcGeom &g, const CUtensorMap &bmap, int num_sms,
                     cudaStream_t s) {
    if (!tc_tiles_fit(a, g)) return cudaErrorInvalidValue;
    const size_t smem = 1024 + static_cast<size_t>(g.stages) * (kA8Bytes + 2 * g.b_bytes);
    auto kern = tc_i8_kernel<PHASE, GATED>;
    static int configured = 0;
    if (static_cast<int>(smem) > configured) {
        const cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        configured = static_cast<int>(smem);
    }
    return launch_pdl(kern, dim3(num_sms), dim3(kThreads), smem, s, *a.tab, a, g, bmap);
}

// K: reduction length (multiple of 128); rows: stored rows (multiple of 128);
// N: token tile, 16 .. 128 in steps of 16.
TcGeom make_geom(int K, int rows, int splits, int N) {
    TcGeom g;
    g.K = K;
    g.rg = rows / 16;
    g.n_rb = rows / 128;
    g.nkb = K / 128;
    g.splits = splits;
    g.N = N;
    g.b_bytes = N * 128;
    const int st = kSmemBudget / (kA8Bytes + 2 * g.b_bytes);
    g.stages = st > kMaxStages ? kMaxStages : st;
    g.tmem_cols = static_cast<int>(kTmemCols);
    g.idesc = idesc_bf16_f32(128, N);
    return g;
}

}  // namespace

cudaError_t launch_gather_rows_f16(const void *x, const int32_t *gather, int rows, int k, int m, int splits,
                                   void *x_perm, float *x_scale, float *x_sum, int xsum_stride, uint32_t *err,
                                   cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    if (splits < 1 || splits > kMaxSumSplits || m % 128) return cudaErrorInvalidValue;
    const int blocks = rows < 8192 ? rows : 8192;
    return launch_pdl(gather_rows_f16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kGatherThreads), 0, s,
                      static_cast<const uint16_t *>(x), gather, rows, k, m, splits, static_cast<uint16_t *>(x_perm),
                      x_scale, x_sum, xsum_stride, err);
}

cudaError_t launch_tc_i8_up(const ExpertArgs &a, bool gated, int splits, int N, const CUtensorMap &xmap,
                            int num_sms, cudaStream_t s) {
    if (N < 16 || N > kTcI8MaxN || N % 16) return cudaErrorInvalidValue;
    const TcGeom g = make_geom(a.m, gated ? 2 * a.p : a.p, splits, N);
    return gated ? launch_t<kUp, true>(a, g, xmap, num_sms, s) : launch_t<kUp, false>(a, g, xmap, num_sms, s);
}

cudaError_t launch_tc_i8_down(const ExpertArgs &a, int splits, int N, const CUtensorMap &hmap,
                              int num_sms, cudaStream_t s) {
    if (N < 16 || N > kTcI8MaxN || N % 16) return cudaErrorInvalidValue;
    const TcGeom g = make_geom(a.p, a.m, splits, N);
    return launch_t<kDown, false>(a, g, hmap, num_sms, s);
}

}  // namespace moe
