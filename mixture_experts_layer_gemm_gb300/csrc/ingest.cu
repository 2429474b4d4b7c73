// ingest.cu -- weight ingestion at layer creation: transpose each expert
// matrix so that every output's reduction run is contiguous (the init-time
// weight transpose of SBI-GeMM, DeepSpeed-Inference article, part 3.3), widen
// the router to fp32, and quantise to per-column symmetric int8.
#include "common.cuh"
#include "kernels.cuh"
#include "packing.h"

namespace moe {

namespace {

template <typename T>
__global__ void transpose_kernel(const T *__restrict__ src, T *__restrict__ dst, int rows, int cols) {
    __shared__ T tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int r = r0 + i, c = c0 + threadIdx.x;
        if (r < rows && c < cols) tile[i][threadIdx.x] = src[static_cast<size_t>(r) * cols + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, r = r0 + threadIdx.x;
        if (r < rows && c < cols) dst[static_cast<size_t>(c) * rows + r] = tile[threadIdx.x][i];
    }
}

// One warp per row of the transposed bf16 matrix (= one column of the
// original): scale = max|w| / 127 (fp32), code = rint(w / scale) clamped to
// [-127, 127]; an all-zero column gets scale 1 and codes 0.
__global__ void quantize_rows_kernel(const uint16_t *__restrict__ wt, int nrows, int len,
                                     int8_t *__restrict__ codes, float *__restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (row >= nrows) return;
    const uint16_t *src = wt + static_cast<size_t>(row) * len;
    float amax = 0.0f;
    for (int i = lane; i < len; i += 32) amax = fmaxf(amax, fabsf(__uint_as_float(uint32_t(src[i]) << 16)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 127.0f);
    if (lane == 0) scales[row] = scale;
    int8_t *dst = codes + static_cast<size_t>(row) * len;
    for (int i = lane; i < len; i += 32) {
        const float w = __uint_as_float(uint32_t(src[i]) << 16);
        float c = rintf(__fdiv_rn(w, scale));
        c = fminf(fmaxf(c, -127.0f), 127.0f);
        dst[i] = static_cast<int8_t>(c);
    }
}

// Pack a transposed matrix (rows x K, K contiguous; elem_bytes 1 or 2) into
// the blocked layout of packing.h.  With src3 given (SwiGLU up-projection),
// stored row 16q + r takes row 8q + r of src1 for r < 8 and row 8q + r - 8 of
// src3 otherwise.  One thread moves one 16-byte run.
__global__ void pack_kernel(const uint8_t *__restrict__ src1, const uint8_t *__restrict__ src3,
                            int rows, int K, int elem_bytes, uint8_t *__restrict__ dst) {
    const int per16 = 16 / elem_bytes;
    const long long runs_per_row = K / per16;
    const long long n = static_cast<long long>(rows) * runs_per_row;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(i / runs_per_row);
        const int k = static_cast<int>(i % runs_per_row) * per16;
        const uint8_t *src;
        if (src3) {
            const int q = r / 16, rr = r % 16;
            src = (rr < 8 ? src1 + static_cast<size_t>(q * 8 + rr) * K * elem_bytes
                          : src3 + static_cast<size_t>(q * 8 + rr - 8) * K * elem_bytes);
        } else {
            src = src1 + static_cast<size_t>(r) * K * elem_bytes;
        }
        const uint4 v = *reinterpret_cast<const uint4 *>(src + static_cast<size_t>(k) * elem_bytes);
        *reinterpret_cast<uint4 *>(dst + packed_offset(r, k, rows, elem_bytes)) = v;
    }
}

template <typename T>
__global__ void router_prep_kernel(const T *src, int m, int E, float *dst) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= m * E) return;
    const int c = i / E, e = i % E;
    float v;
    if constexpr (sizeof(T) == 2)
        v = __uint_as_float(uint32_t(src[i]) << 16);
    else
        v = src[i];
    dst[static_cast<size_t>(e) * m + c] = v;
}

}  // namespace

cudaError_t launch_transpose(const void *src, void *dst, int rows, int cols, int elem_bytes,
                             cudaStream_t s) {
    dim3 grid((cols + 31) / 32, (rows + 31) / 32), block(32, 8);
    if (elem_bytes == 2)
        transpose_kernel<uint16_t><<<grid, block, 0, s>>>(static_cast<const uint16_t *>(src),
                                                          static_cast<uint16_t *>(dst), rows, cols);
    else
        transpose_kernel<float><<<grid, block, 0, s>>>(static_cast<const float *>(src),
                                                       static_cast<float *>(dst), rows, cols);
    return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const void *wt_bf16, int nrows, int len, int8_t *codes,
                                 float *scales, cudaStream_t s) {
    const int warps = 8;
    quantize_rows_kernel<<<(nrows + warps - 1) / warps, 32 * warps, 0, s>>>(
        static_cast<const uint16_t *>(wt_bf16), nrows, len, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_pack(const void *src1, const void *src3, int rows, int K, int elem_bytes,
                        void *dst, cudaStream_t s) {
    const long long n = static_cast<long long>(rows) * K * elem_bytes / 16;
    long long blocks = (n + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    pack_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<const uint8_t *>(src1), static_cast<const uint8_t *>(src3), rows, K, elem_bytes,
        static_cast<uint8_t *>(dst));
    return cudaGetLastError();
}

cudaError_t launch_router_prep(const void *src, bool bf16, int m, int E, float *dst,
                               cudaStream_t s) {
    const int n = m * E;
    if (bf16)
        router_prep_kernel<uint16_t><<<(n + 255) / 256, 256, 0, s>>>(static_cast<const uint16_t *>(src),
                                                                     m, E, dst);
    else
        router_prep_kernel<float><<<(n + 255) / 256, 256, 0, s>>>(static_cast<const float *>(src), m,
                                                                  E, dst);
    return cudaGetLastError();
}

}  // namespace moe
