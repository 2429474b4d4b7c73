// kernels.cuh -- argument blocks and host launchers of the library's kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Launch a forward-path kernel with programmatic stream serialisation allowed
// (see pdl_wait / pdl_trigger in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

constexpr int kExpertTableMax = 64;

// ---- routing -------------------------------------------------------------------
struct RouterArgs {
    const void *x;       // [T x m] act type
    const float *wrt;    // [E x m] router weights, transposed, fp32
    const void *wra;     // [E x m] the same, in the activation type (exact)
    const float *bias;   // [E] or nullptr
    int T, m, E, k;
    int32_t *ids;        // [T*k]
    float *w;            // [T*k]
    float *logits;       // [T*E] or nullptr
    unsigned *ticket;    // device counter, 0 between launches (fused permute)
    uint32_t *err;
};

struct PermuteArgs {
    const int32_t *ids;  // [T*k]
    int T, k, E;
    int32_t *counts, *offsets, *gather, *scatter;
    // per-CTA expert counts of a multi-CTA fused router permute
    // ([ceil(T / 16) x E], overwritten by their prefix over CTAs), or nullptr
    int32_t *cta_count;
};

// Router + top-k with the permute fused in (the launch's last CTA runs it).
cudaError_t launch_router_topk(const RouterArgs &a, const PermuteArgs &pa, bool act_bf16,
                               cudaStream_t s);
cudaError_t launch_topk_from_logits(const float *logits, int T, int E, int k, int32_t *ids,
                                    float *w, cudaStream_t s);
cudaError_t launch_topk_copy_validate(const int32_t *ids_in, const float *w_in, int T, int E,
                                      int k, int32_t *ids_out, float *w_out, uint32_t *err,
                                      cudaStream_t s);
cudaError_t launch_permute(const PermuteArgs &a, cudaStream_t s);

// ---- expert weights as stored ---------------------------------------------------
// fp32 layers: w1/w3[e] = W1^T/W3^T [p x m], w2[e] = W2^T [m x p], row-major.
// bf16 / int8 layers: packed (packing.h): w1[e] = U (gate and up rows
// interleaved for SwiGLU), w2[e] = D = W2^T; w3 unused.
// For int8 weights, s1/s3[e] hold p fp32 scales and s2[e] holds m scales.
struct ExpertTables {
    const void *w1[kExpertTableMax];
    const void *w3[kExpertTableMax];
    const void *w2[kExpertTableMax];
    const float *s1[kExpertTableMax];
    const float *s3[kExpertTableMax];
    const float *s2[kExpertTableMax];
};

// Which experts a launch covers: the experts listed in `only` (n_only > 0,
// paged layers launch per resident expert) or every expert with tokens.
struct ExpertArgs {
    const ExpertTables *tab;     // host copy, passed by value to the kernel
    const void *x;               // [T x m] act type (tokens in token order)
    const int32_t *gather;       // [T*k]
    const int32_t *offsets;      // [E+1]
    const float *topk_w;         // [T*k]
    int T, k, E, m, p;
    void *h;                     // [T*k x p] act type (permuted order)
    float *ypart;                // [splits x T*k x m] fp32 (permuted order); bf16 where ypart_bf16
    int ypart_bf16;              // batch regime: the down projection writes its rows rounded to bf16
    int n_rows_cap;              // T*k capacity of one ypart split
    float *gate_part;            // [splits_up x T*k x p] fp32 (decode split-K up only)
    float *up_part;              // same
    uint32_t *err;
    int only[kExpertTableMax];
    int n_only;
    const void *wbase;           // start of the resident weight buffer (CTA-pair kernels)
    // int8 weights, tensor-core up projection: x_perm holds the permuted token
    // rows in fp16 under a power-of-two scale per row; x_scale[pos] is that
    // scale and x_sum[s * xsum_stride + pos] the row's sum over reduction split s
    const float *x_scale;
    const float *x_sum;
    int xsum_stride;
};

enum class WeightType { kF32, kBF16, kI8 };

// Decode regime: weight-streaming expert GEMV on the legacy tensor path.
// Token tiles of 8 per pass chosen from the mean tokens per expert.
int decode_token_tiles(int T, int k, int E);
cudaError_t launch_decode_up(const ExpertArgs &a, WeightType wt, bool gated, int splits,
                             int num_sms, cudaStream_t s);
cudaError_t launch_decode_down(const ExpertArgs &a, WeightType wt, int splits, int num_sms,
                               cudaStream_t s);
// finish a split-K up projection: h = act(sum_s gate_part) [* sum_s up_part]
cudaError_t launch_decode_up_finish(const ExpertArgs &a, bool gated, int splits,
                                    cudaStream_t s);

// Tensor-core (tcgen05) grouped GEMM: weights on the M side (128-row blocks),
// N tokens per tile (16..256, multiple of 16); the tensor map fetches the
// permuted activations (x_perm for up, h for down) in N x 64 boxes.
cudaError_t launch_gather_rows(const void *x, const int32_t *gather, int rows, int k, int m,
                               void *x_perm, uint32_t *err, cudaStream_t s);
cudaError_t launch_tc_up(const ExpertArgs &a, bool gated, int splits, int N, const CUtensorMap &xmap,
                         int num_sms, cudaStream_t s);
cudaError_t launch_tc_down(const ExpertArgs &a, int splits, int N, const CUtensorMap &hmap,
                           int num_sms, cudaStream_t s);
// The same on CTA pairs (cta_group::2) for 256-token tiles, bf16 weights,
// stored rows a multiple of 256, no reduction split; the tensor map fetches
// 128-token halves (the N = 128 map).
// wmap: the packed weights (a.wbase on) as 128-byte rows, 128-row boxes.
cudaError_t launch_tc2_up(const ExpertArgs &a, bool gated, const CUtensorMap &wmap, const CUtensorMap &xmap_half,
                          int num_sms, cudaStream_t s);

// The same with int8 weights (K a multiple of 128): codes widened exactly in
// tensor memory -- to fp16 (1152 + code) against the fp16 token rows of
// launch_gather_rows_f16 in the up projection, to bf16 against the bf16 hidden
// rows in the down projection -- with the bias, the token scales and the
// per-row weight scale taken out in the epilogue; N tokens per tile, 16..192.
constexpr int kTcI8MaxN = 192;
// x_perm[pos] = x[gather[pos] / k] in fp16 times 2^-s (s from the row's largest
// magnitude, f16_row_shift), x_scale[pos] = 2^s, and the sums of the scaled
// row over each of `splits` reduction splits (K blocks of 128) into x_sum.
cudaError_t launch_gather_rows_f16(const void *x, const int32_t *gather, int rows, int k, int m, int splits,
                                   void *x_perm, float *x_scale, float *x_sum, int xsum_stride, uint32_t *err,
                                   cudaStream_t s);
cudaError_t launch_tc_i8_up(const ExpertArgs &a, bool gated, int splits, int N, const CUtensorMap &xmap,
                            int num_sms, cudaStream_t s);
cudaError_t launch_tc_i8_down(const ExpertArgs &a, int splits, int N, const CUtensorMap &hmap,
                              int num_sms, cudaStream_t s);

// fp32 path (SIMT, warp-shuffle reductions)
cudaError_t launch_simt_up(const ExpertArgs &a, bool gated, cudaStream_t s);
cudaError_t launch_simt_down(const ExpertArgs &a, cudaStream_t s);

// Combine: y[t] = sum_j sum_s ypart[s][scatter[t*k+j]] in fp32, rounded once.
// The partial rows are fp32, or bf16 where the batch regime's down projection
// wrote them rounded (part_bf16).
struct CombineArgs {
    const void *ypart;
    int splits;
    size_t split_stride;         // elements between splits
    const int32_t *scatter;
    int T, k, m;
    void *y;
    uint32_t *err;
    bool part_bf16;
};
cudaError_t launch_combine(const CombineArgs &a, bool act_bf16, cudaStream_t s);

// ---- weight ingestion ------------------------------------------------------------
// dst[c][r] = src[r][c] for a rows x cols matrix; element size 2 or 4 bytes.
cudaError_t launch_transpose(const void *src, void *dst, int rows, int cols, int elem_bytes,
                             cudaStream_t s);
// Per-row symmetric int8 of a bf16 nrows x len matrix (rows of the transposed
// weight = columns of the user's matrix): codes [nrows x len], scales [nrows].
cudaError_t launch_quantize_rows(const void *wt_bf16, int nrows, int len, int8_t *codes,
                                 float *scales, cudaStream_t s);
// Pack transposed rows into the blocked layout of packing.h (src3: SwiGLU up).
cudaError_t launch_pack(const void *src1, const void *src3, int rows, int K, int elem_bytes,
                        void *dst, cudaStream_t s);
// widen router weights to fp32 and transpose: dst[e][c] = src[c][e]
cudaError_t launch_router_prep(const void *src, bool bf16, int m, int E, float *dst,
                               cudaStream_t s);

}  // namespace moe
