// expert_decode.cu -- decode-regime expert MLP: a weight-streaming skinny GEMM.
//
// At decode batch sizes each expert sees a handful of tokens, so the expert
// matmuls are bound by reading the weights once from HBM (DeepSpeed-Inference
// article, part 1: small-batch inference is limited by the bandwidth of
// reading the weights; the expert-cache article, section 1: a Mixtral expert
// takes 0.3 ms on an RTX 4090, i.e. one pass over its ~340 MB).  The kernel
// follows the three parts of SBI-GeMM (DeepSpeed-Inference article, part 3):
//   1. tiling: a work unit is 16 weight rows (outputs) of one expert, so the
//      reduction stays inside the unit; where the outputs alone would not give
//      every SM enough units, the reduction dimension is split across units too
//      (the two-kernel variant) and a second pass adds the partial sums;
//   2. reduction: the 8 warps of a CTA each reduce one slice of the unit's
//      reduction range; their partial tiles are written to shared memory in a
//      transposed layout that puts the 8 partials of one output next to each
//      other, and one thread per output adds them;
//   3. full cache lines: weights are stored transposed at create time (each
//      output's reduction run is contiguous), and every lane reads 16 bytes
//      per load -- 8 bf16 or 16 int8 values -- so each warp load covers whole
//      32-byte sectors.
// Different from the pages: the per-warp dot products run on the warp-level
// tensor-core MMA (m16n8k16, bf16 in, fp32 accumulate) with the tokens on the
// N side, because from about four tokens per expert on, CUDA-core FMAs cannot
// keep pace with GB300's HBM.  Since a dot product does not depend on the
// order of its terms, each lane's 16-byte run of weights and the matching
// 16-byte run of the token row are assigned to the fragment slots of two
// (bf16) or four (int8) MMAs with the same permutation of the reduction
// index, so both operands come from contiguous vector loads.
// int8 weights are widened to bf16 in registers (exact) and the per-output
// scale is applied after the dot product.
#include "common.cuh"
#include "kernels.cuh"

namespace moe {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerUnit = 16;
constexpr int kUnroll = 8;

template <WeightType WT>
struct WTraits;
template <>
struct WTraits<WeightType::kBF16> {
    static constexpr int kStep = 32;    // reduction elements per warp step
    static constexpr int kPad = 64;     // smem row padding (bank-conflict-free B reads)
    static constexpr int kElem = 2;
};
template <>
struct WTraits<WeightType::kI8> {
    static constexpr int kStep = 64;
    static constexpr int kPad = 16;
    static constexpr int kElem = 1;
};

enum Phase { kUp = 0, kDown = 1 };

struct DecodeGeom {
    int K;          // reduction length (m for up, p for down)
    int splits;     // split of the reduction across units
    int nsteps;     // K / kStep
    int kr_max;     // largest split in elements, rounded up to 64
    int row_bytes;  // smem stride of one staged token row
    int rg;         // row groups (units along the output) per expert
};

__device__ __forceinline__ int split_begin(int nsteps, int splits, int ks) {
    return static_cast<int>((static_cast<long long>(nsteps) * ks) / splits);
}

// Load one step of A (weights) for rows g and g+8 of the unit.
template <WeightType WT>
__device__ __forceinline__ void load_a(const uint8_t *row_g, const uint8_t *row_g8, int kelem,
                                       uint4 &ra, uint4 &rb) {
    ra = ld_stream_v4(row_g + static_cast<size_t>(kelem) * WTraits<WT>::kElem);
    rb = ld_stream_v4(row_g8 + static_cast<size_t>(kelem) * WTraits<WT>::kElem);
}

// One warp step: A fragments from the loaded weight runs, B fragments from the
// staged token rows (smem), MMAs into acc.
template <WeightType WT, int NT>
__device__ __forceinline__ void mma_step(float (&acc)[NT][4], const uint4 &ra, const uint4 &rb,
                                         uint32_t bsm, int row_bytes, int g, int t, int kcol) {
    if constexpr (WT == WeightType::kBF16) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint4 xb = lds_v4(bsm + (nt * 8 + g) * row_bytes + (kcol + 8 * t) * 2);
            mma_bf16_16816(acc[nt], ra.x, rb.x, ra.y, rb.y, xb.x, xb.y);
            mma_bf16_16816(acc[nt], ra.z, rb.z, ra.w, rb.w, xb.z, xb.w);
        }
    } else {
        uint32_t al[4], ah[4], bl[4], bh[4];
        const uint32_t va[4] = {ra.x, ra.y, ra.z, ra.w};
        const uint32_t vb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            i8x4_to_bf16x2x2(va[i], al[i], ah[i]);
            i8x4_to_bf16x2x2(vb[i], bl[i], bh[i]);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint32_t base = bsm + (nt * 8 + g) * row_bytes + (kcol + 16 * t) * 2;
            const uint4 x0 = lds_v4(base);
            const uint4 x1 = lds_v4(base + 16);
            mma_bf16_16816(acc[nt], al[0], bl[0], ah[0], bh[0], x0.x, x0.y);
            mma_bf16_16816(acc[nt], al[1], bl[1], ah[1], bh[1], x0.z, x0.w);
            mma_bf16_16816(acc[nt], al[2], bl[2], ah[2], bh[2], x1.x, x1.y);
            mma_bf16_16816(acc[nt], al[3], bl[3], ah[3], bh[3], x1.z, x1.w);
        }
    }
}

template <WeightType WT, int PHASE, bool GATED, int NT>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const ExpertTables tab, const ExpertArgs a, const DecodeGeom geo) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kTok = 8 * NT;                  // tokens per pass
    constexpr int kOut = kRowsPerUnit * kTok;     // outputs of one unit-pass
    constexpr int kStep = WTraits<WT>::kStep;
    __shared__ int s_act[kMaxExperts];
    __shared__ int s_nact;

    uint8_t *bstage = smem;
    float *red = reinterpret_cast<float *>(smem + static_cast<size_t>(kTok) * geo.row_bytes);
    const uint32_t bsm = smem_u32(bstage);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int rows_total = a.T * a.k;

    // active expert list (in expert order)
    if (tid == 0) {
        int n = 0;
        if (a.n_only > 0) {
            for (int i = 0; i < a.n_only && i < kMaxExperts; ++i) s_act[n++] = a.only[i];
        } else {
            for (int e = 0; e < a.E; ++e)
                if (a.offsets[e + 1] > a.offsets[e]) s_act[n++] = e;
        }
        s_nact = n;
    }
    __syncthreads();
    const int nact = s_nact;
    const long long units = static_cast<long long>(nact) * geo.splits * geo.rg;

    int staged_e = -1, staged_ks = -1, staged_tp = -1;
    for (long long u = blockIdx.x; u < units; u += gridDim.x) {
        const int rg = static_cast<int>(u % geo.rg);
        const int ks = static_cast<int>((u / geo.rg) % geo.splits);
        const int e = s_act[static_cast<int>(u / (static_cast<long long>(geo.rg) * geo.splits))];
        int off = a.offsets[e], end = a.offsets[e + 1];
        if (off < 0 || end > rows_total || end < off) {  // corrupt tables: skip the expert
            if (tid == 0) flag_error(a.err, kErrOffsets);
            continue;
        }
        const int q = end - off;
        const int s0 = split_begin(geo.nsteps, geo.splits, ks);
        const int s1 = split_begin(geo.nsteps, geo.splits, ks + 1);
        const int kbase = s0 * kStep;                    // first reduction element of the split
        const int kcount = (s1 - s0) * kStep;
        // weight rows of this unit
        const uint8_t *row_g, *row_g8;
        {
            const size_t K = static_cast<size_t>(geo.K) * WTraits<WT>::kElem;
            if (PHASE == kUp) {
                const uint8_t *w1 = static_cast<const uint8_t *>(tab.w1[e]);
                if (GATED) {
                    const uint8_t *w3 = static_cast<const uint8_t *>(tab.w3[e]);
                    row_g = w1 + static_cast<size_t>(rg * 8 + g) * K;
                    row_g8 = w3 + static_cast<size_t>(rg * 8 + g) * K;
                } else {
                    row_g = w1 + static_cast<size_t>(rg * 16 + g) * K;
                    row_g8 = w1 + static_cast<size_t>(rg * 16 + 8 + g) * K;
                }
            } else {
                const uint8_t *w2 = static_cast<const uint8_t *>(tab.w2[e]);
                row_g = w2 + static_cast<size_t>(rg * 16 + g) * K;
                row_g8 = w2 + static_cast<size_t>(rg * 16 + 8 + g) * K;
            }
            row_g += static_cast<size_t>(kbase) * WTraits<WT>::kElem;
            row_g8 += static_cast<size_t>(kbase) * WTraits<WT>::kElem;
        }
        const int lane_k = (WT == WeightType::kBF16) ? 8 * t : 16 * t;
        // this warp's slice of the split's steps
        const int nst = s1 - s0;
        const int w0 = s0 + (nst * warp) / kWarps, w1e = s0 + (nst * (warp + 1)) / kWarps;

        for (int tp = 0; tp * kTok < q; ++tp) {
            // ---- stage the token rows of this pass (bf16) into shared memory
            if (staged_e != e || staged_ks != ks || staged_tp != tp) {
                __syncthreads();
                const int vec_per_row = kcount / 8;  // 16-byte vectors
                for (int idx = tid; idx < kTok * vec_per_row; idx += kThreads) {
                    const int r = idx / vec_per_row, v = idx - r * vec_per_row;
                    const int pos = off + tp * kTok + r;
                    uint4 val = make_uint4(0, 0, 0, 0);
                    if (pos < end) {
                        const uint16_t *src;
                        if (PHASE == kUp) {
                            const int fi = a.gather[pos];
                            if (fi >= 0 && fi < rows_total) {
                                src = static_cast<const uint16_t *>(a.x) +
                                      static_cast<size_t>(fi / a.k) * geo.K;
                                val = ld_nc_v4(src + kbase + v * 8);
                            } else if (v == 0) {
                                flag_error(a.err, kErrGatherIndex);
                            }
                        } else {
                            src = static_cast<const uint16_t *>(a.h) + static_cast<size_t>(pos) * geo.K;
                            val = ld_nc_v4(src + kbase + v * 8);
                        }
                    }
                    *reinterpret_cast<uint4 *>(bstage + static_cast<size_t>(r) * geo.row_bytes + v * 16) = val;
                }
                staged_e = e;
                staged_ks = ks;
                staged_tp = tp;
                __syncthreads();
            }
            // ---- stream this warp's weight slice
            float acc[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[nt][i] = 0.0f;
            for (int s = w0; s < w1e; s += kUnroll) {
                uint4 ra[kUnroll], rb[kUnroll];
#pragma unroll
                for (int i = 0; i < kUnroll; ++i)
                    if (s + i < w1e) load_a<WT>(row_g, row_g8, (s + i - s0) * kStep + lane_k, ra[i], rb[i]);
#pragma unroll
                for (int i = 0; i < kUnroll; ++i)
                    if (s + i < w1e)
                        mma_step<WT, NT>(acc, ra[i], rb[i], bsm, geo.row_bytes, g, t, (s + i - s0) * kStep);
            }
            // ---- transposed partial tile: red[out * 8 + warp]
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int c0 = nt * 8 + 2 * t;
                red[((g)*kTok + c0) * kWarps + warp] = acc[nt][0];
                red[((g)*kTok + c0 + 1) * kWarps + warp] = acc[nt][1];
                red[((g + 8) * kTok + c0) * kWarps + warp] = acc[nt][2];
                red[((g + 8) * kTok + c0 + 1) * kWarps + warp] = acc[nt][3];
            }
            __syncthreads();
            // ---- one thread per output adds the 8 partials, then the epilogue
            auto rsum = [&](int o) {
                const float4 p0 = *reinterpret_cast<const float4 *>(red + o * kWarps);
                const float4 p1 = *reinterpret_cast<const float4 *>(red + o * kWarps + 4);
                return ((p0.x + p0.y) + (p0.z + p0.w)) + ((p1.x + p1.y) + (p1.z + p1.w));
            };
            if (PHASE == kUp && GATED) {
                for (int o = tid; o < 8 * kTok; o += kThreads) {
                    const int tok = o >> 3, r = o & 7;
                    const int pos = off + tp * kTok + tok;
                    if (pos < end) {
                        const int n = rg * 8 + r;
                        float gv = rsum(r * kTok + tok), uv = rsum((r + 8) * kTok + tok);
                        if (WT == WeightType::kI8) {
                            gv *= tab.s1[e][n];
                            uv *= tab.s3[e][n];
                        }
                        if (geo.splits == 1) {
                            static_cast<__nv_bfloat16 *>(a.h)[static_cast<size_t>(pos) * a.p + n] =
                                __float2bfloat16_rn(silu(gv) * uv);
                        } else {
                            const size_t o2 = (static_cast<size_t>(ks) * a.n_rows_cap + pos) * a.p + n;
                            a.gate_part[o2] = gv;
                            a.up_part[o2] = uv;
                        }
                    }
                }
            } else {
                for (int o = tid; o < kRowsPerUnit * kTok; o += kThreads) {
                    const int tok = o >> 4, r = o & 15;
                    const int pos = off + tp * kTok + tok;
                    if (pos < end) {
                        float v = rsum(r * kTok + tok);
                        const int n = rg * 16 + r;
                        if (PHASE == kUp) {
                            if (WT == WeightType::kI8) v *= tab.s1[e][n];
                            if (geo.splits == 1) {
                                static_cast<__nv_bfloat16 *>(a.h)[static_cast<size_t>(pos) * a.p + n] =
                                    __float2bfloat16_rn(fmaxf(v, 0.0f));
                            } else {
                                a.gate_part[(static_cast<size_t>(ks) * a.n_rows_cap + pos) * a.p + n] = v;
                            }
                        } else {
                            if (WT == WeightType::kI8) v *= tab.s2[e][n];
                            const int fi = a.gather[pos];
                            const float wgt = (fi >= 0 && fi < rows_total) ? a.topk_w[fi] : 0.0f;
                            a.ypart[(static_cast<size_t>(ks) * a.n_rows_cap + pos) * a.m + n] = wgt * v;
                        }
                    }
                }
            }
            __syncthreads();
        }
    }
}

// h = act(sum_s gate_part[s]) [* sum_s up_part[s]] for split-K up projections.
template <bool GATED>
__global__ void up_finish_kernel(const ExpertArgs a, int splits) {
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
DecodeGeom make_geom(int K, int splits, int nt, int rg) {
    DecodeGeom g;
    g.K = K;
    g.splits = splits;
    g.nsteps = K / WTraits<WT>::kStep;
    const int max_steps = (g.nsteps + splits - 1) / splits;
    const int kr = max_steps * WTraits<WT>::kStep;
    g.kr_max = (kr + 63) / 64 * 64;
    g.row_bytes = g.kr_max * 2 + WTraits<WT>::kPad;
    g.rg = rg;
    (void)nt;
    return g;
}

template <WeightType WT, int PHASE, bool GATED, int NT>
cudaError_t launch_one(const ExpertArgs &a, int K, int splits, int rg, int num_sms,
                       cudaStream_t s) {
    const DecodeGeom geo = make_geom<WT>(K, splits, NT, rg);
    const size_t smem = static_cast<size_t>(8 * NT) * geo.row_bytes +
                        static_cast<size_t>(kRowsPerUnit * 8 * NT) * kWarps * sizeof(float);
    auto kern = decode_kernel<WT, PHASE, GATED, NT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    kern<<<num_sms * per_sm, kThreads, smem, s>>>(*a.tab, a, geo);
    return cudaGetLastError();
}

template <WeightType WT, int PHASE, bool GATED>
cudaError_t dispatch_nt(const ExpertArgs &a, int nt, int K, int splits, int rg, int num_sms,
                        cudaStream_t s) {
    switch (nt) {
    case 1: return launch_one<WT, PHASE, GATED, 1>(a, K, splits, rg, num_sms, s);
    case 2: return launch_one<WT, PHASE, GATED, 2>(a, K, splits, rg, num_sms, s);
    default: return launch_one<WT, PHASE, GATED, 4>(a, K, splits, rg, num_sms, s);
    }
}

}  // namespace

// Token tiles per pass, from the mean tokens per expert (T*k/E); experts with
// more tokens than one pass holds take further passes over their weights.
int decode_token_tiles(int T, int k, int E) {
    const int mean_q = (T * k + E - 1) / E;
    if (mean_q <= 6) return 1;
    if (mean_q <= 12) return 2;
    return 4;
}

cudaError_t launch_decode_up(const ExpertArgs &a, WeightType wt, bool gated, int splits,
                             int num_sms, cudaStream_t s) {
    const int nt = decode_token_tiles(a.T, a.k, a.E);
    const int rg = gated ? a.p / 8 : a.p / 16;
    if (wt == WeightType::kBF16)
        return gated ? dispatch_nt<WeightType::kBF16, kUp, true>(a, nt, a.m, splits, rg, num_sms, s)
                     : dispatch_nt<WeightType::kBF16, kUp, false>(a, nt, a.m, splits, rg, num_sms, s);
    return gated ? dispatch_nt<WeightType::kI8, kUp, true>(a, nt, a.m, splits, rg, num_sms, s)
                 : dispatch_nt<WeightType::kI8, kUp, false>(a, nt, a.m, splits, rg, num_sms, s);
}

cudaError_t launch_decode_down(const ExpertArgs &a, WeightType wt, int splits, int num_sms,
                               cudaStream_t s) {
    const int nt = decode_token_tiles(a.T, a.k, a.E);
    const int rg = a.m / 16;
    if (wt == WeightType::kBF16)
        return dispatch_nt<WeightType::kBF16, kDown, false>(a, nt, a.p, splits, rg, num_sms, s);
    return dispatch_nt<WeightType::kI8, kDown, false>(a, nt, a.p, splits, rg, num_sms, s);
}

cudaError_t launch_decode_up_finish(const ExpertArgs &a, bool gated, int splits, cudaStream_t s) {
    const size_t n = static_cast<size_t>(a.T) * a.k * a.p;
    if (n == 0) return cudaSuccess;
    const int blocks = static_cast<int>((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
    if (gated)
        up_finish_kernel<true><<<blocks, 256, 0, s>>>(a, splits);
    else
        up_finish_kernel<false><<<blocks, 256, 0, s>>>(a, splits);
    return cudaGetLastError();
}

}  // namespace moe
