// packing.h -- the stored layout of bf16 and int8 expert weights.
//
// Each expert matrix is stored transposed (one row per output, the reduction
// index K along the row; SBI-GeMM's init-time weight transpose) and tiled
// into 2 KB blocks of 16 rows x BK reduction elements (BK = 64 for bf16,
// 128 for int8).  Blocks are ordered K-block-major: block (kb, rg) sits at
// byte (kb * RG + rg) * 2048, RG = rows / 16.  A block holds four 512-byte
// atoms, atom (G, s) = rows 8G..8G+7 x the s-th half of the block's K range,
// at G * 1024 + s * 512.  Inside an atom, row g (0..7) takes 64 bytes and its
// 16-byte chunk c (0..3) is stored at chunk position c ^ ((g / 2) % 4): the
// 64-byte swizzle of the tensor cores' K-major operand layout.
// Two consumers read it:
//   - the decode GEMV: lane (g, t) of a warp reads chunk t of row g of one
//     atom, so each warp load covers one 512-byte atom and, thanks to the
//     swizzle, every 8-lane phase of the shared-memory read hits 8 different
//     banks groups;
//   - the tensor-core GEMM (bf16): 8 consecutive row-groups of one K-block
//     form a 16 KB contiguous tile in the canonical 64-byte-swizzled K-major
//     layout: atoms 1024 bytes apart along the rows, 512 bytes apart along K.
// For the SwiGLU up-projection the stored matrix U interleaves the gate and
// up rows per 8: rows 16q..16q+7 are W1^T[8q..8q+7] and rows 16q+8..16q+15 are
// W3^T[8q..8q+7]; for the ReLU form U is W1^T.  The down-projection matrix D
// is W2^T.
#pragma once

#include <stddef.h>
#include <stdint.h>

#ifdef __CUDACC__
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

namespace moe {

constexpr int kBlockBytes = 2048;
constexpr int kBlockRows = 16;

MOE_HD int block_k(int elem_bytes) { return elem_bytes == 1 ? 128 : 64; }

// Byte offset, inside a 512-byte atom, of 16-byte chunk t of row g.
MOE_HD int atom_chunk_offset(int g, int t) { return g * 64 + ((t ^ (g >> 1)) & 3) * 16; }

// Byte offset of element (row, k) in a packed matrix with `rows` rows.
MOE_HD size_t packed_offset(int row, int k, int rows, int elem_bytes) {
    const int BK = block_k(elem_bytes);
    const int per16 = 16 / elem_bytes;  // elements per 16-byte run
    const int half = BK / 2;
    const int rg = row / 16, r = row % 16;
    const int kb = k / BK, c = k % BK;
    const int G = r / 8, g = r % 8;
    const int s = c / half, t = (c % half) / per16, e = c % per16;
    const size_t block = static_cast<size_t>(kb) * (rows / 16) + rg;
    return block * kBlockBytes + G * 1024 + s * 512 + atom_chunk_offset(g, t) + e * elem_bytes;
}

// Stored row of SwiGLU up-projection feature n (gate: W1, up: W3).
MOE_HD int up_row_gate(int n) { return (n / 8) * 16 + (n % 8); }
MOE_HD int up_row_up(int n) { return (n / 8) * 16 + 8 + (n % 8); }

}  // namespace moe
