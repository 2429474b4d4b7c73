// tc_tiles.cuh -- the tile space of the grouped expert GEMMs on the tensor
// cores: (expert, reduction split, 128-row block, token tile), token tile
// fastest, so that CTAs working at the same time share a weight block
// through L2.  Each CTA of a persistent launch takes tiles blockIdx.x,
// blockIdx.x + gridDim.x, ...; the active experts and the prefix sums of their
// tile counts sit in shared memory.
#pragma once

#include <stdint.h>

#include "common.cuh"
#include "kernels.cuh"

namespace moe {

struct TcGeom {
    int K;          // reduction length
    int rg;         // row-groups of 16 stored rows
    int n_rb;       // 128-row blocks
    int nkb;        // K / (reduction elements per pipeline stage)
    int splits;     // reduction splits
    int N;          // token tile
    int stages;
    int b_bytes;    // N * 128
    int tmem_cols;  // columns allocated
    uint32_t idesc;
};

struct TcTile {
    int e, ks, rb, tt, off, q, kb0, kb1;
};

// Tile u of the launch.  `cur` is the caller's cursor into the expert list:
// a role walks its tiles in increasing order, so the search for u's expert
// starts where the last one ended (a scan from the first expert costs a chain
// of dependent shared-memory loads per tile with many experts).  The index
// arithmetic is 32-bit (the launchers check that one expert's tiles fit): a
// role's single thread runs it between two tiles, where 64-bit divisions
// (software sequences) held the MMAs back about a microsecond per tile.
__device__ __forceinline__ TcTile tc_tile(long long u, const long long *prefix, const int *act,
                                          const int *offs, const int *qs, int nact, const TcGeom &g, int &cur) {
    int i = cur;
    while (i + 1 < nact && u >= prefix[i + 1]) ++i;
    cur = i;
    const unsigned local = static_cast<unsigned>(u - prefix[i]);
    const unsigned ntt = static_cast<unsigned>((qs[i] + g.N - 1) / g.N);
    const unsigned nrb = static_cast<unsigned>(g.n_rb);
    TcTile t;
    t.e = act[i];
    t.off = offs[i];
    t.q = qs[i];
    const unsigned rest = local / ntt;
    t.tt = static_cast<int>(local - rest * ntt);
    const unsigned ks = rest / nrb;
    t.rb = static_cast<int>(rest - ks * nrb);
    t.ks = static_cast<int>(ks);
    const unsigned nkb = static_cast<unsigned>(g.nkb), sp = static_cast<unsigned>(g.splits);
    t.kb0 = static_cast<int>((nkb * ks) / sp);
    t.kb1 = static_cast<int>((nkb * (ks + 1)) / sp);
    return t;
}

// Host side: whether tc_tile's 32-bit arithmetic holds for a launch (one
// expert's tiles, at most ceil(T k / N) token tiles, and nkb x splits below
// 2^31); the launchers refuse a launch for which it does not.
inline bool tc_tiles_fit(const ExpertArgs &a, const TcGeom &g) {
    const long long ntt = (static_cast<long long>(a.T) * a.k + g.N - 1) / g.N;
    return static_cast<long long>(g.splits) * g.n_rb * ntt < (1LL << 31) &&
           static_cast<long long>(g.nkb) * (g.splits + 1) < (1LL << 31);
}

// One warp (all 32 lanes): list the experts this launch covers (all with
// tokens, or those in a.only), in ascending expert order, their segments, and
// the prefix sums of their tile counts.  Lane l examines experts l and l + 32,
// so every offset is read in one round trip; a ballot compacts the list and a
// shuffle scan sums the tiles.  Returns the number of experts listed (in
// every lane).
__device__ __forceinline__ int tc_list_tiles(const ExpertArgs &a, const TcGeom &geo, int *act,
                                             int *offs, int *qs, long long *prefix, int lane) {
    const int rows_total = a.T * a.k;
    int n = 0;
    long long acc = 0;
    if (lane == 0) prefix[0] = 0;
    for (int e0 = 0; e0 < a.E; e0 += 32) {
        const int e = e0 + lane;
        bool take = false;
        int off = 0, q = 0;
        if (e < a.E) {
            off = a.offsets[e];
            const int end = a.offsets[e + 1];
            if (off < 0 || end > rows_total || end < off) {
                flag_error(a.err, kErrOffsets);
            } else {
                q = end - off;
                take = q > 0;
                if (take && a.n_only > 0) {
                    bool listed = false;
                    for (int i = 0; i < a.n_only; ++i) listed |= a.only[i] == e;
                    take = listed;
                }
            }
        }
        const unsigned mask = __ballot_sync(0xffffffffu, take);
        const int idx = n + __popc(mask & ((1u << lane) - 1u));
        long long incl = take ? static_cast<long long>(geo.splits) * geo.n_rb * ((q + geo.N - 1) / geo.N) : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        if (take) {
            act[idx] = e;
            offs[idx] = off;
            qs[idx] = q;
            prefix[idx + 1] = acc + incl;
        }
        acc += __shfl_sync(0xffffffffu, incl, 31);
        n += __popc(mask);
    }
    return n;
}

// Routing weights of a tile's tokens tok0 .. tok0 + n - 1 (n <= 256) of the
// segment at `off`, read by one warp with independent loads (eight per lane)
// into that warp's shared-memory row, so that the down projection's store loop
// does not wait on two dependent global loads per token.  Tokens past the
// segment, or whose gather index is out of range, get weight 0.
constexpr int kTcMaxTileTokens = 256;

// SiLU from the hardware exp2 and reciprocal approximations (the __expf and
// __fdividef intrinsics): a few instructions instead of the IEEE-accurate
// sequences, with an error far below the bf16 rounding of h.  For z -> -inf
// the denominator overflows to +inf and the quotient is 0.
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// SwiGLU epilogue of 16 accumulator columns, the tokens tok .. tok + 15 of the
// segment at `off`.  Stored rows interleave 8 gate and 8 up rows, so a lane
// whose row has bit 3 clear holds gate values and the lane 8 away the matching
// up values of the same feature f.  The pair swaps half its columns with one
// shuffle per column pair, after which the gate lane finishes tokens 0..7 and
// the up lane tokens 8..15: every lane does useful work and each SiLU is
// evaluated once.  `scale` multiplies this lane's own values (int8 row scales;
// 1 for bf16 weights).  Tokens at or past q are not stored.
__device__ __forceinline__ void tc_swiglu_store16(const uint32_t (&v)[16], float scale, bool gate_lane,
                                                  __nv_bfloat16 *h, int p, int f, int off, int tok,
                                                  int q) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float lo = __uint_as_float(v[j]) * scale, hi = __uint_as_float(v[j + 8]) * scale;
        const float recv = __shfl_xor_sync(0xffffffffu, gate_lane ? hi : lo, 8);
        const float g = gate_lane ? lo : recv;
        const float u = gate_lane ? recv : hi;
        const int tk = tok + j + (gate_lane ? 0 : 8);
        if (tk < q) h[static_cast<size_t>(off + tk) * p + f] = __float2bfloat16_rn(silu_fast(g) * u);
    }
}

__device__ __forceinline__ void tc_stage_weights(const ExpertArgs &a, int off, int tok0, int q, int n,
                                                 float *s_w, int lane) {
    const int rows_total = a.T * a.k;
    int fi[kTcMaxTileTokens / 32];
#pragma unroll
    for (int ci = 0; ci < kTcMaxTileTokens / 32; ++ci) {
        const int c = ci * 32 + lane;
        fi[ci] = (c < n && tok0 + c < q) ? a.gather[off + tok0 + c] : -1;
    }
    float wv[kTcMaxTileTokens / 32];
#pragma unroll
    for (int ci = 0; ci < kTcMaxTileTokens / 32; ++ci)
        wv[ci] = (fi[ci] >= 0 && fi[ci] < rows_total) ? a.topk_w[fi[ci]] : 0.0f;
    __syncwarp();  // every lane is past its reads of the previous tile's row
#pragma unroll
    for (int ci = 0; ci < kTcMaxTileTokens / 32; ++ci) s_w[ci * 32 + lane] = wv[ci];
    __syncwarp();
}

}  // namespace moe
