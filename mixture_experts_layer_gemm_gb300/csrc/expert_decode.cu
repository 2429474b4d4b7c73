// expert_decode.cu -- decode-regime expert MLP: a weight-streaming skinny GEMM.
//
// At decode batch sizes each expert sees a handful of tokens, so the expert
// matmuls are bound by reading the weights once from HBM (DeepSpeed-Inference
// article, part 1: small-batch inference is limited by the bandwidth of
// reading the weights; the expert-cache article, section 1: a Mixtral expert
// takes 0.3 ms on an RTX 4090, one pass over its ~340 MB).  The kernel follows
// SBI-GeMM (DeepSpeed-Inference article, part 3):
//   1. tiling along the outputs: a work unit is 128 stored weight rows of one
//      expert (8 row-groups of 16, one per consumer warp), so the reduction
//      stays inside the unit; where the outputs alone would not give every SM
//      enough units, the reduction range is split across units too (the
//      two-kernel variant) and a later pass adds the partial sums in a fixed
//      order (the up-projection finish kernel, or the combine);
//   2. reduction: inside a warp the tensor-core MMA reduces across lanes, and
//      each warp owns its 16 rows, so no cross-warp reduction is needed;
//   3. full cache lines: weights are stored transposed and tiled at create
//      time (packing.h), so the 8 row-groups of one reduction block are one
//      contiguous 16 KB run, and a warp's 16-byte-per-lane shared-memory read
//      covers one 512-byte atom without bank conflicts.
// GB300-specific design:
//   - one producer thread streams each unit's 16 KB weight stages from HBM
//     with bulk asynchronous copies (the TMA engine) into an 8-stage
//     shared-memory ring guarded by mbarriers, so up to 128 KB per SM are in
//     flight whatever the register budget;
//   - the per-warp dot products run on the warp-level tensor-core MMA
//     (m16n8k16, bf16 in, fp32 accumulate) with the tokens on the N side:
//     from about four tokens per expert on, CUDA-core FMAs cannot keep pace
//     with HBM.  A dot product does not depend on the order of its terms, so
//     lane (g, t) takes the 16-byte run t of weight rows g and g+8 and the
//     16-byte run t of its token row, and feeds them to two (bf16) or four
//     (int8) MMAs under one shared permutation of the reduction index;
//   - the token rows of the current expert and split are staged once in
//     shared memory and reused by every unit of that expert;
//   - int8 weights run the MMAs in fp16: one XOR and two byte permutes turn
//     four codes b into the exact fp16 values 1152 + b (a third of the
//     instructions of widening to bf16), the staged token rows are converted
//     to fp16 under a power-of-two scale per row (exact for every value in
//     fp16's normal range), and the epilogue takes out 1152 times the row sum
//     of the scaled activations, undoes the row scale and applies the
//     per-output weight scale.
// Every wait is bounded; a wait that gives up sets kErrWaitTimeout in the
// layer's error word and the CTA drains its copies in flight and returns.
#include <cmath>

#include "common.cuh"
#include "kernels.cuh"
#include "packing.h"

namespace moe {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kStages = 8;  // 128 KB of weights in flight per SM
constexpr int kBlocksPerStage = 8;
constexpr int kStageBytes = kBlocksPerStage * kBlockBytes;  // 16 KB
constexpr int kRowsPerUnit = 16;
constexpr uint32_t kBarConsumers = 1;  // named barrier id for the consumer warps

template <WeightType WT>
struct WTraits;
template <>
struct WTraits<WeightType::kBF16> {
    static constexpr int kBK = 64;      // reduction elements per 2 KB block
    static constexpr int kPad = 64;     // staged token-row padding: conflict-free B reads
};
template <>
struct WTraits<WeightType::kI8> {
    static constexpr int kBK = 128;
    static constexpr int kPad = 16;
};

enum Phase { kUp = 0, kDown = 1 };

struct DecodeGeom {
    int K;          // reduction length (m for up, p for down)
    int rg;         // row-groups of 16 stored rows
    int rg8;        // units along the rows: ceil(rg / 8)
    int splits;     // split of the K-blocks across units
    int nkb;        // K / BK
    int row_bytes;  // smem stride of one staged token row
    int bstage_bytes;
};

// n * ks < 2^31: n <= K / 64 reduction blocks, ks <= 16 splits
__device__ __forceinline__ int split_begin(int n, int splits, int ks) {
    return static_cast<int>(static_cast<unsigned>(n * ks) / static_cast<unsigned>(splits));
}

// int8 weights: convert the staged bf16 token rows 0 .. nrows-1 to fp16 in
// place.  The row's largest magnitude sets a power-of-two scale 2^-s that puts
// it in [2^14, 2^15): every bf16 value whose scaled magnitude is at least
// 2^-14 is then an exact fp16 value (only values below the row maximum by a
// factor of 2^28 or more round).  Records 2^s and the sum of the converted
// values for the epilogue.  A row of zeros, or one holding an infinity or NaN,
// keeps scale 1.
//
// A pass of a few rows (one or two at the smallest batches) is latency-bound:
// each row goes to wpr warps, the largest power of two with nrows * wpr <= 8
// (1 from five rows on), whose partial maxima and sums meet in s_red / s_red2
// and are combined in warp order, so the sums are deterministic.
// Rows past nrows are not touched: their MMA columns belong to no token.
__device__ __forceinline__ void stage_rows_f16(uint8_t *bstage, int row_bytes, int vec_per_row, int nrows,
                                               int warp, int lane, float *s_red, float *s_red2, float *s_xscale,
                                               float *s_xsum) {
    const int wpr = nrows >= 5 ? 1 : (nrows >= 3 ? 2 : (nrows == 2 ? 4 : 8));  // nrows * wpr <= 8 below 8 rows
    const int ngroups = kConsumerWarps / wpr;
    const int grp = warp / wpr, sub = warp % wpr;
    const int j0 = sub * 32 + lane, stride = wpr * 32;
    for (int r = grp; r < nrows; r += ngroups) {
        const uint4 *row = reinterpret_cast<const uint4 *>(bstage + static_cast<size_t>(r) * row_bytes);
        float m0 = 0.0f, m1 = 0.0f;
        int v = j0;
        for (; v + stride < vec_per_row; v += 2 * stride) {
            const uint4 q0 = row[v], q1 = row[v + stride];
            const uint32_t w0[4] = {q0.x, q0.y, q0.z, q0.w}, w1[4] = {q1.x, q1.y, q1.z, q1.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                m0 = fmaxf(m0, fmaxf(fabsf(bf16lo(w0[i])), fabsf(bf16hi(w0[i]))));
                m1 = fmaxf(m1, fmaxf(fabsf(bf16lo(w1[i])), fabsf(bf16hi(w1[i]))));
            }
        }
        if (v < vec_per_row) {
            const uint4 q0 = row[v];
            const uint32_t w0[4] = {q0.x, q0.y, q0.z, q0.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) m0 = fmaxf(m0, fmaxf(fabsf(bf16lo(w0[i])), fabsf(bf16hi(w0[i]))));
        }
        float mx = fmaxf(m0, m1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) s_red[r * wpr + sub] = mx;
    }
    if (wpr > 1)
        named_sync(kBarConsumers, kConsumers);
    else
        __syncwarp();
    for (int r = grp; r < nrows; r += ngroups) {
        float mx = s_red[r * wpr];
        for (int w = 1; w < wpr; ++w) mx = fmaxf(mx, s_red[r * wpr + w]);
        const int sh = f16_row_shift(mx);
        const float down = pow2f(-sh);
        uint4 *row = reinterpret_cast<uint4 *>(bstage + static_cast<size_t>(r) * row_bytes);
        float s0 = 0.0f, s1 = 0.0f;
        for (int v = j0; v < vec_per_row; v += stride) {
            const uint4 q = row[v];
            uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __half2 hv = __floats2half2_rn(bf16lo(w[i]) * down, bf16hi(w[i]) * down);
                s0 += __low2float(hv);
                s1 += __high2float(hv);
                w[i] = *reinterpret_cast<const uint32_t *>(&hv);
            }
            row[v] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        const float sum = warp_sum(s0 + s1);
        if (lane == 0) {
            s_red2[r * wpr + sub] = sum;
            if (sub == 0) s_xscale[r] = pow2f(sh);
        }
    }
    if (wpr > 1)
        named_sync(kBarConsumers, kConsumers);
    else
        __syncwarp();
    if (sub == 0 && lane == 0)
        for (int r = grp; r < nrows; r += ngroups) {
            float sum = s_red2[r * wpr];
            for (int w = 1; w < wpr; ++w) sum += s_red2[r * wpr + w];
            s_xsum[r] = sum;
        }
}

// Work entries are (expert, token pass) pairs: an expert with more tokens
// than one pass holds gets one entry per pass, so that the units of a pass
// are consecutive and a CTA stages each (pass, split) of token rows once.
// Passes per expert are at most q / kTok + 1, so at most E + (T k) / 8 entries
// (T k <= 512 on this path).
constexpr int kMaxPassEntries = kMaxExperts + 512 / 8;

struct Unit {
    int e, tp, ks, g8, nrg, off, end, kb0, kb1;
    bool ok;
};

// Unit indices are 32-bit (the launcher checks the count fits): this runs on
// the path to each CTA's first weight copy, where 64-bit divisions (a software
// sequence each) cost about a microsecond.
__device__ __forceinline__ Unit decode_unit(unsigned u, const int *s_act, const int *s_tp, const int *s_off,
                                            const int *s_end, const DecodeGeom &geo, int rows_total) {
    Unit U;
    const unsigned rg8 = static_cast<unsigned>(geo.rg8), sp = static_cast<unsigned>(geo.splits);
    const unsigned q = u / rg8;
    U.g8 = static_cast<int>(u - q * rg8);
    const unsigned entry_u = q / sp;
    U.ks = static_cast<int>(q - entry_u * sp);
    const int entry = static_cast<int>(entry_u);
    U.e = s_act[entry];
    U.tp = s_tp[entry];
    U.nrg = min(8, geo.rg - 8 * U.g8);
    U.off = s_off[entry];
    U.end = s_end[entry];
    U.ok = !(U.off < 0 || U.end > rows_total || U.end < U.off);
    U.kb0 = split_begin(geo.nkb, geo.splits, U.ks);
    U.kb1 = split_begin(geo.nkb, geo.splits, U.ks + 1);
    return U;
}

template <WeightType WT, int PHASE, bool GATED, int NT>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const ExpertTables tab, const ExpertArgs a, const DecodeGeom geo) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int kTok = 8 * NT;  // tokens per pass
    constexpr int kBK = WTraits<WT>::kBK;
    __shared__ uint64_t full_bar[kStages], empty_bar[kStages];
    __shared__ uint64_t rows_bar;  // token rows of the current (expert, split, pass) staged
    __shared__ int s_act[kMaxPassEntries], s_tp[kMaxPassEntries];  // (expert, pass) entries
    __shared__ int s_off[kMaxPassEntries], s_end[kMaxPassEntries];  // the entry's expert segment
    __shared__ int s_nact;
    __shared__ volatile int s_abort;
    __shared__ float s_xscale[kTok], s_xsum[kTok];  // int8: per staged row, 2^s and sum of x 2^-s
    __shared__ float s_red[kTok], s_red2[kTok];       // int8: per-warp partial maxima and sums

    uint8_t *ring = smem;
    uint8_t *bstage = smem + kStages * kStageBytes;
    const uint32_t bsm = smem_u32(bstage);
    const uint32_t ring_sm = smem_u32(ring);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rows_total = a.T * a.k;
    // The producer's weight pointers, copied from the launch parameters into
    // shared memory before anything waits: parameters are not written by the
    // predecessor, and their first reads in a CTA are slow (measured: the
    // CTA's first weight copy about a microsecond earlier).
    __shared__ const void *s_wptr[kExpertTableMax];
    if (warp == kConsumerWarps)
        for (int e = lane; e < kExpertTableMax; e += 32) s_wptr[e] = PHASE == kUp ? tab.w1[e] : tab.w2[e];
    if (tid == 0)
        touch_params(a.offsets, a.only[0], a.n_only, a.E, a.T, a.k, a.gather, a.x, a.h, a.topk_w, a.ypart, a.err);
    // The up projection reads the routing its predecessor (the router) wrote.
    // The down projection's predecessor is the up projection: the routing is
    // two launches back and complete, so the weight stream starts at once and
    // only the consumers wait, before they read the hidden rows.
    if (PHASE == kUp) {
        pdl_wait();
        pdl_trigger();
    }

    if (warp == 0) {
        // One warp lists the (expert, token pass) entries: lane l takes the
        // candidate experts l, l + 32 (all experts, or those of a.only, in
        // order), so their offsets are read in one round trip; each entry
        // keeps its expert's segment, so the producer and the consumers find
        // it in shared memory instead of another global read before their
        // first copy.  A malformed segment keeps one entry, whose unit then
        // reports it.
        const bool only = a.n_only > 0;
        const int ncand = only ? min(a.n_only, kMaxExperts) : a.E;
        int n = 0;
        for (int c0 = 0; c0 < ncand; c0 += 32) {
            const int ci = c0 + lane;
            int e = -1, np = 0, off = 0, end = 0;
            if (ci < ncand) {
                e = only ? a.only[ci] : ci;
                off = a.offsets[e];
                end = a.offsets[e + 1];
                const bool bad = off < 0 || end > rows_total || end < off;
                if (only || end > off) np = ((bad ? 1 : end - off) + kTok - 1) / kTok;
            }
            int incl = np;  // inclusive prefix sum of the pass counts over lanes
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            const int base = n + incl - np;
            for (int tp = 0; tp < np; ++tp) {
                if (base + tp >= kMaxPassEntries) {
                    flag_error(a.err, kErrOffsets);
                    break;
                }
                s_act[base + tp] = e;
                s_tp[base + tp] = tp;
                s_off[base + tp] = off;
                s_end[base + tp] = end;
            }
            n += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            s_nact = min(n, kMaxPassEntries);
            s_abort = 0;
            for (int i = 0; i < kStages; ++i) {
                mbar_init(&full_bar[i], 1);
                mbar_init(&empty_bar[i], kConsumers);  // every consumer lane releases
            }
            mbar_init(&rows_bar, 1);
            fence_barrier_init();
        }
    }
    __syncthreads();
    const unsigned units = static_cast<unsigned>(s_nact) * geo.splits * geo.rg8;
    // each CTA takes a contiguous range of units, so that consecutive units
    // share the expert and split and reuse the staged token rows: CTA b takes
    // [floor(units b / grid), floor(units (b + 1) / grid)), the longer ranges
    // spread evenly, computed in 32 bits as b u_per + floor(b u_rem / grid)
    const unsigned u_per = units / gridDim.x, u_rem = units - u_per * gridDim.x;
    const unsigned u_begin = blockIdx.x * u_per + (blockIdx.x * u_rem) / gridDim.x;
    const unsigned u_end = (blockIdx.x + 1) * u_per + ((blockIdx.x + 1) * u_rem) / gridDim.x;

    // A slot is re-armed only after all consumer warps released it, which they
    // do only after seeing its copy land; so at any time each slot has at most
    // one phase in flight, the last one issued.
    uint32_t last_parity[kStages];
    bool used[kStages];
    uint32_t rows_phase = 0, rows_last = 0;  // token-row staging: next and last issued parity
    bool rows_issued = false;
    for (int i = 0; i < kStages; ++i) used[i] = false;
    if (warp == kConsumerWarps) {
        // ================= producer: stream weight stages into the ring ==========
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (unsigned u = u_begin; u < u_end && !s_abort; ++u) {
                const Unit U = decode_unit(u, s_act, s_tp, s_off, s_end, geo, rows_total);
                if (!U.ok) continue;
                const uint8_t *w = static_cast<const uint8_t *>(s_wptr[U.e]);
                const uint32_t bytes = static_cast<uint32_t>(U.nrg) * kBlockBytes;
                const int q = U.end - U.off;
                {  // this unit's pass
                    for (int kb = U.kb0; kb < U.kb1; ++kb) {
                        if (!mbar_wait(&empty_bar[stage], phase ^ 1u)) {
                            flag_error(a.err, kErrWaitTimeout);
                            s_abort = 1;
                            break;
                        }
                        mbar_arrive_expect_tx(&full_bar[stage], bytes);
                        const size_t blk = static_cast<size_t>(kb) * geo.rg + 8 * U.g8;
                        if (q <= kTok)  // one token pass: each weight byte is read once
                            bulk_g2s_once(ring + stage * kStageBytes, w + blk * kBlockBytes, bytes,
                                          &full_bar[stage]);
                        else
                            bulk_g2s(ring + stage * kStageBytes, w + blk * kBlockBytes, bytes,
                                     &full_bar[stage]);
                        used[stage] = true;
                        last_parity[stage] = phase;
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
        }
    } else {
    // ================= consumers: warp w owns row-group 8*g8 + w of each unit ======
    if (PHASE == kDown) {
        pdl_wait();
        pdl_trigger();
    }
    const int g = lane >> 2, t = lane & 3;
    int stage = 0;
    uint32_t phase = 0;
    int staged_e = -1, staged_ks = -1, staged_tp = -1;
    for (unsigned u = u_begin; u < u_end; ++u) {
        // one decision for all consumer warps: the named barriers need all of them
        if (named_sync_or(kBarConsumers, kConsumers, s_abort)) break;
        const Unit U = decode_unit(u, s_act, s_tp, s_off, s_end, geo, rows_total);
        if (!U.ok) {
            if (tid == 0) flag_error(a.err, kErrOffsets);
            continue;
        }
        const int kbase = U.kb0 * kBK;                 // first reduction element of the split
        const int kcount = (U.kb1 - U.kb0) * kBK;
        const bool mine = warp < U.nrg;
        const int rg = 8 * U.g8 + warp;
        {
            const int tp = U.tp;  // this unit's token pass
            // ---- stage this pass's token rows (bf16) in shared memory: one
            // bulk copy per row (the copy engine, a single round trip), issued
            // by the lanes of consumer warp 0.  Rows past the segment are not
            // copied: their MMA columns are tokens whose results are never
            // stored.
            if (staged_e != U.e || staged_ks != U.ks || staged_tp != tp) {
                // every consumer is past its reads (and the int8 in-place
                // conversion) of the previous rows before the copy engine
                // overwrites them
                fence_proxy_async_smem();
                named_sync(kBarConsumers, kConsumers);
                if (warp == 0) {
                    const int pos = U.off + tp * kTok + lane;
                    const bool row = lane < kTok && pos < U.end;
                    const uint16_t *src = nullptr;
                    if (row) {
                        if (PHASE == kUp) {
                            int fi = a.gather[pos];
                            if (fi < 0 || fi >= rows_total) {  // reported; a valid row stands in
                                flag_error(a.err, kErrGatherIndex);
                                fi = 0;
                            }
                            src = static_cast<const uint16_t *>(a.x) + static_cast<size_t>(fi / a.k) * geo.K + kbase;
                        } else {
                            src = static_cast<const uint16_t *>(a.h) + static_cast<size_t>(pos) * geo.K + kbase;
                        }
                    }
                    const uint32_t nrows = __popc(__ballot_sync(0xffffffffu, row));
                    if (lane == 0) mbar_arrive_expect_tx(&rows_bar, nrows * static_cast<uint32_t>(kcount) * 2u);
                    __syncwarp();
                    if (row)
                        bulk_g2s(bstage + static_cast<size_t>(lane) * geo.row_bytes, src,
                                 static_cast<uint32_t>(kcount) * 2u, &rows_bar);
                }
                rows_issued = true;
                rows_last = rows_phase;
                const bool landed = mbar_wait(&rows_bar, rows_phase);
                if (named_sync_or(kBarConsumers, kConsumers, !landed)) {
                    if (tid == 0) flag_error(a.err, kErrWaitTimeout);
                    s_abort = 1;
                    break;
                }
                rows_phase ^= 1u;
                staged_e = U.e;
                staged_ks = U.ks;
                staged_tp = tp;
                if constexpr (WT == WeightType::kI8) {
                    const int nrows = min(kTok, U.end - (U.off + tp * kTok));
                    stage_rows_f16(bstage, geo.row_bytes, kcount / 8, nrows, warp, lane, s_red, s_red2, s_xscale,
                                   s_xsum);
                    named_sync(kBarConsumers, kConsumers);
                }
            }
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;

            // ---- consume the unit's weight stages: block `warp` of each stage
            for (int kb = U.kb0; kb < U.kb1; ++kb) {
                // warp-uniform: the MMAs below need the whole warp
                bool have = false;
                if (!__any_sync(0xffffffffu, s_abort)) {
                    have = __all_sync(0xffffffffu, mbar_wait(&full_bar[stage], phase));
                    if (!have) {
                        if (lane == 0) flag_error(a.err, kErrWaitTimeout);
                        s_abort = 1;
                    }
                }
                if (have) {
                    // This warp's weight fragments of the stage into registers,
                    // then the slot goes back to the producer at once (each
                    // lane's arrive releases its own reads), so the copy
                    // engine refills it while the MMAs below run.  The token
                    // operands live in the staged rows, outside the ring.
                    uint4 ra[2], rb[2];
                    if (mine) {
                        const uint32_t blk = ring_sm + stage * kStageBytes + warp * kBlockBytes;
#pragma unroll
                        for (int sh = 0; sh < 2; ++sh) {
                            const uint32_t atom = blk + sh * 512 + atom_chunk_offset(g, t);
                            ra[sh] = lds_v4(atom);         // row g
                            rb[sh] = lds_v4(atom + 1024);  // row g + 8
                        }
                    }
                    mbar_arrive(&empty_bar[stage]);
                    if (mine) {
#pragma unroll
                        for (int sh = 0; sh < 2; ++sh) {
                            const int kcol = (kb - U.kb0) * kBK + sh * (kBK / 2);  // in the staged rows
                            if constexpr (WT == WeightType::kBF16) {
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    const uint4 xb =
                                        lds_v4(bsm + (nt * 8 + g) * geo.row_bytes + (kcol + 8 * t) * 2);
                                    mma_bf16_16816(acc[nt], ra[sh].x, rb[sh].x, ra[sh].y, rb[sh].y, xb.x, xb.y);
                                    mma_bf16_16816(acc[nt], ra[sh].z, rb[sh].z, ra[sh].w, rb[sh].w, xb.z, xb.w);
                                }
                            } else {
                                uint32_t al[4], ah[4], bl[4], bh[4];
                                const uint32_t va[4] = {ra[sh].x, ra[sh].y, ra[sh].z, ra[sh].w};
                                const uint32_t vb[4] = {rb[sh].x, rb[sh].y, rb[sh].z, rb[sh].w};
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    i8x4_to_f16x2x2_biased(va[i], al[i], ah[i]);
                                    i8x4_to_f16x2x2_biased(vb[i], bl[i], bh[i]);
                                }
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    const uint32_t xa = bsm + (nt * 8 + g) * geo.row_bytes + (kcol + 16 * t) * 2;
                                    const uint4 x0 = lds_v4(xa);
                                    const uint4 x1 = lds_v4(xa + 16);
                                    mma_f16_16816(acc[nt], al[0], bl[0], ah[0], bh[0], x0.x, x0.y);
                                    mma_f16_16816(acc[nt], al[1], bl[1], ah[1], bh[1], x0.z, x0.w);
                                    mma_f16_16816(acc[nt], al[2], bl[2], ah[2], bh[2], x1.x, x1.y);
                                    mma_f16_16816(acc[nt], al[3], bl[3], ah[3], bh[3], x1.z, x1.w);
                                }
                            }
                        }
                    }
                }
                if (++stage == kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            // ---- epilogue straight from the MMA fragments of this warp's 16 rows:
            // acc[nt][0..1] = (row g, tokens nt*8+2t, +1), acc[nt][2..3] = row g + 8
            if (mine && !s_abort) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int tk = nt * 8 + 2 * t + h2;  // token of the pass
                        const int pos = U.off + tp * kTok + tk;
                        if (pos >= U.end) continue;
                        float v0 = acc[nt][h2], v8 = acc[nt][2 + h2];
                        if (WT == WeightType::kI8) {  // take out the code bias, undo the row scale
                            v0 = fmaf(-kI8F16Bias, s_xsum[tk], v0) * s_xscale[tk];
                            v8 = fmaf(-kI8F16Bias, s_xsum[tk], v8) * s_xscale[tk];
                        }
                        if (PHASE == kUp && GATED) {
                            const int n = rg * 8 + g;  // feature: gate row g, up row g + 8
                            if (WT == WeightType::kI8) {
                                v0 *= tab.s1[U.e][n];
                                v8 *= tab.s3[U.e][n];
                            }
                            if (geo.splits == 1) {
                                static_cast<__nv_bfloat16 *>(a.h)[static_cast<size_t>(pos) * a.p + n] =
                                    __float2bfloat16_rn(silu(v0) * v8);
                            } else {
                                const size_t o = (static_cast<size_t>(U.ks) * a.n_rows_cap + pos) * a.p + n;
                                a.gate_part[o] = v0;
                                a.up_part[o] = v8;
                            }
                        } else if (PHASE == kUp) {
                            const int n0 = rg * 16 + g, n8 = n0 + 8;
                            if (WT == WeightType::kI8) {
                                v0 *= tab.s1[U.e][n0];
                                v8 *= tab.s1[U.e][n8];
                            }
                            if (geo.splits == 1) {
                                __nv_bfloat16 *hr = static_cast<__nv_bfloat16 *>(a.h) + static_cast<size_t>(pos) * a.p;
                                hr[n0] = __float2bfloat16_rn(fmaxf(v0, 0.0f));
                                hr[n8] = __float2bfloat16_rn(fmaxf(v8, 0.0f));
                            } else {
                                float *gp = a.gate_part + (static_cast<size_t>(U.ks) * a.n_rows_cap + pos) * a.p;
                                gp[n0] = v0;
                                gp[n8] = v8;
                            }
                        } else {
                            const int n0 = rg * 16 + g, n8 = n0 + 8;
                            if (WT == WeightType::kI8) {
                                v0 *= tab.s2[U.e][n0];
                                v8 *= tab.s2[U.e][n8];
                            }
                            const int fi = a.gather[pos];
                            const float wgt = (fi >= 0 && fi < rows_total) ? a.topk_w[fi] : 0.0f;
                            float *yr = a.ypart + (static_cast<size_t>(U.ks) * a.n_rows_cap + pos) * a.m;
                            yr[n0] = wgt * v0;
                            yr[n8] = wgt * v8;
                        }
                    }
                }
            }
        }
    }
    }
    // one barrier for producer and consumers; then no copy may still be in
    // flight when the CTA exits (matters on the abort path)
    __syncwarp();
    __syncthreads();
    if (warp == kConsumerWarps && lane == 0)
        for (int i = 0; i < kStages; ++i)
            if (used[i]) mbar_wait(&full_bar[i], last_parity[i]);
    // a token-row staging whose wait gave up may still be landing
    if (tid == 0 && rows_issued) mbar_wait(&rows_bar, rows_last);
}

// h = act(sum_s gate_part[s]) [* sum_s up_part[s]] for split-K up projections.
template <bool GATED>
__global__ void up_finish_kernel(const ExpertArgs a, int splits) {
    pdl_wait();
    pdl_trigger();
    const size_t rows = static_cast<size_t>(a.T) * a.k;
    const size_t n = rows * a.p;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        float gv = 0.0f, uv = 0.0f;
        for (int s = 0; s < splits; ++s) {
            const size_t o = static_cast<size_t>(s) * a.n_rows_cap * a.p + i;
            gv += a.gate_part[o];
            if (GATED) uv += a.up_part[o];
        }
        const float hv = GATED ? silu(gv) * uv : fmaxf(gv, 0.0f);
        static_cast<__nv_bfloat16 *>(a.h)[i] = __float2bfloat16_rn(hv);
    }
}

template <WeightType WT>
DecodeGeom make_geom(int K, int rows, int splits, int nt) {
    DecodeGeom g;
    g.K = K;
    g.rg = rows / kRowsPerUnit;
    g.rg8 = (g.rg + 7) / 8;
    g.splits = splits;
    g.nkb = K / WTraits<WT>::kBK;
    const int max_kb = (g.nkb + splits - 1) / splits;
    const int kr = max_kb * WTraits<WT>::kBK;
    const int kr64 = (kr + 63) / 64 * 64;
    g.row_bytes = kr64 * 2 + WTraits<WT>::kPad;
    g.bstage_bytes = (8 * nt * g.row_bytes + 15) / 16 * 16;
    return g;
}

template <WeightType WT, int PHASE, bool GATED, int NT>
cudaError_t launch_one(const ExpertArgs &a, int K, int rows, int splits, int num_sms,
                       cudaStream_t s) {
    const DecodeGeom geo = make_geom<WT>(K, rows, splits, NT);
    // the kernel counts units (and splits of the reduction blocks) in 32 bits
    if (static_cast<long long>(kMaxPassEntries) * splits * geo.rg8 >= (1LL << 31) ||
        static_cast<long long>(geo.nkb) * splits >= (1LL << 31))
        return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(kStages) * kStageBytes + geo.bstage_bytes;
    auto kern = decode_kernel<WT, PHASE, GATED, NT>;
    static int configured_smem = 0;  // per instantiation
    if (static_cast<int>(smem) > configured_smem) {
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        configured_smem = static_cast<int>(smem);
    }
    return launch_pdl(kern, dim3(num_sms), dim3(kThreads), smem, s, *a.tab, a, geo);
}

template <WeightType WT, int PHASE, bool GATED>
cudaError_t dispatch_nt(const ExpertArgs &a, int nt, int K, int rows, int splits, int num_sms,
                        cudaStream_t s) {
    switch (nt) {
    case 1: return launch_one<WT, PHASE, GATED, 1>(a, K, rows, splits, num_sms, s);
    case 2: return launch_one<WT, PHASE, GATED, 2>(a, K, rows, splits, num_sms, s);
    case 3: return launch_one<WT, PHASE, GATED, 3>(a, K, rows, splits, num_sms, s);
    default: return launch_one<WT, PHASE, GATED, 4>(a, K, rows, splits, num_sms, s);
    }
}

}  // namespace

// Token tiles per pass.  An expert with more tokens than one pass holds
// streams its weights once per pass, so the pass is sized for the busier
// experts, not the mean: under uniform routing an expert's count has mean
// T k / E and variance T k (1/E)(1 - 1/E), and the pass covers the mean plus
// 1.5 standard deviations.  Every tile adds MMAs per widened weight and
// staged rows, so the smallest pass that covers them is taken (Mixtral shape,
// int8, T = 64: 24-token passes 456 us per layer, 32-token passes 513 us).  An
// expert with more tokens still takes further passes (its own work entries),
// each streaming its weights again.
int decode_token_tiles(int T, int k, int E) {
    const double mean = static_cast<double>(T) * k / E;
    const double hi = mean + 1.5 * std::sqrt(mean * (1.0 - 1.0 / E)) + 0.5;
    if (hi <= 8.0) return 1;
    if (hi <= 18.0) return 2;
    if (hi <= 24.0) return 3;
    return 4;
}

cudaError_t launch_decode_up(const ExpertArgs &a, WeightType wt, bool gated, int splits,
                             int num_sms, cudaStream_t s) {
    const int nt = decode_token_tiles(a.T, a.k, a.E);
    const int rows = gated ? 2 * a.p : a.p;
    if (wt == WeightType::kBF16)
        return gated ? dispatch_nt<WeightType::kBF16, kUp, true>(a, nt, a.m, rows, splits, num_sms, s)
                     : dispatch_nt<WeightType::kBF16, kUp, false>(a, nt, a.m, rows, splits, num_sms, s);
    return gated ? dispatch_nt<WeightType::kI8, kUp, true>(a, nt, a.m, rows, splits, num_sms, s)
                 : dispatch_nt<WeightType::kI8, kUp, false>(a, nt, a.m, rows, splits, num_sms, s);
}

cudaError_t launch_decode_down(const ExpertArgs &a, WeightType wt, int splits, int num_sms,
                               cudaStream_t s) {
    const int nt = decode_token_tiles(a.T, a.k, a.E);
    if (wt == WeightType::kBF16)
        return dispatch_nt<WeightType::kBF16, kDown, false>(a, nt, a.p, a.m, splits, num_sms, s);
    return dispatch_nt<WeightType::kI8, kDown, false>(a, nt, a.p, a.m, splits, num_sms, s);
}

cudaError_t launch_decode_up_finish(const ExpertArgs &a, bool gated, int splits, cudaStream_t s) {
    const size_t n = static_cast<size_t>(a.T) * a.k * a.p;
    if (n == 0) return cudaSuccess;
    const int blocks = static_cast<int>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    if (gated)
        return launch_pdl(up_finish_kernel<true>, dim3(blocks), dim3(256), 0, s, a, splits);
    else
        return launch_pdl(up_finish_kernel<false>, dim3(blocks), dim3(256), 0, s, a, splits);
}

}  // namespace moe
