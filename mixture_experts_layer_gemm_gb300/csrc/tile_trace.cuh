// tile_trace.cuh -- per-tile timeline of the tensor-core grouped GEMM kernels,
// compiled in only when MOE_TILE_TRACE is defined (a separate build of the
// library, made by the tile-trace tool; the default build defines nothing
// here and every macro below expands to an empty statement).
//
// Each CTA below trace::kCtas records the globaltimer (ns) at its entry and,
// for each of its first trace::kTiles tiles, the time its MMA thread found the
// tile's first stage landed and the time it issued the tile's last stage,
// with the tile's expert, token tile, width in tokens and row block, into one
// of two slots (the kernel's phase: 0 up projection, 1 down projection).  A
// CTA pair records on its even CTA.  The buffers live in the translation unit
// that includes this header (no relocatable device code): each kernel file
// exports its own reader, named by MOE_TRACE_READER.
#pragma once

#ifdef MOE_TILE_TRACE

#include <cuda_runtime.h>

namespace moe {
namespace trace {

constexpr int kCtas = 160;
constexpr int kTiles = 128;

static __device__ unsigned long long g_t[2][kCtas][kTiles][2];  // first stage landed, last stage issued
static __device__ unsigned long long g_t0[2][kCtas];             // CTA entry
static __device__ int g_info[2][kCtas][kTiles][4];               // expert, token tile, width, row block
static __device__ int g_on;

__device__ __forceinline__ unsigned long long now() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace trace
}  // namespace moe

#define MOE_TRACE_ENTRY(slot)                                                             \
    do {                                                                                  \
        if (threadIdx.x == 0 && moe::trace::g_on && blockIdx.x < moe::trace::kCtas)       \
            moe::trace::g_t0[slot][blockIdx.x] = moe::trace::now();                       \
    } while (0)

#define MOE_TRACE_TILE_FIRST(slot, ti, e, tt, n, rb)                                     \
    do {                                                                                  \
        if (moe::trace::g_on && blockIdx.x < moe::trace::kCtas && (ti) < moe::trace::kTiles) { \
            moe::trace::g_t[slot][blockIdx.x][ti][0] = moe::trace::now();                 \
            int *inf_ = moe::trace::g_info[slot][blockIdx.x][ti];                         \
            inf_[0] = (e);                                                                \
            inf_[1] = (tt);                                                               \
            inf_[2] = (n);                                                                \
            inf_[3] = (rb);                                                               \
        }                                                                                 \
    } while (0)

#define MOE_TRACE_TILE_LAST(slot, ti)                                                     \
    do {                                                                                  \
        if (moe::trace::g_on && blockIdx.x < moe::trace::kCtas && (ti) < moe::trace::kTiles) \
            moe::trace::g_t[slot][blockIdx.x][ti][1] = moe::trace::now();                 \
    } while (0)

// extern "C" int name(t, t0, info, on): copies the buffers out (each pointer
// may be null: t [2][kCtas][kTiles][2] u64, t0 [2][kCtas] u64,
// info [2][kCtas][kTiles][4] int), then clears them and sets recording on
// (on != 0) or off.  Returns a cudaError_t.
#define MOE_TRACE_READER(name)                                                            \
    extern "C" int name(unsigned long long *t, unsigned long long *t0, int *info, int on) { \
        cudaError_t e = cudaSuccess;                                                      \
        if (t && e == cudaSuccess) e = cudaMemcpyFromSymbol(t, moe::trace::g_t, sizeof(moe::trace::g_t)); \
        if (t0 && e == cudaSuccess) e = cudaMemcpyFromSymbol(t0, moe::trace::g_t0, sizeof(moe::trace::g_t0)); \
        if (info && e == cudaSuccess)                                                     \
            e = cudaMemcpyFromSymbol(info, moe::trace::g_info, sizeof(moe::trace::g_info)); \
        void *p = nullptr;                                                                \
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&p, moe::trace::g_t);              \
        if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(moe::trace::g_t));              \
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&p, moe::trace::g_t0);             \
        if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(moe::trace::g_t0));             \
        if (e == cudaSuccess) e = cudaGetSymbolAddress(&p, moe::trace::g_info);           \
        if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(moe::trace::g_info));           \
        if (e == cudaSuccess) e = cudaMemcpyToSymbol(moe::trace::g_on, &on, sizeof(int)); \
        if (e == cudaSuccess) e = cudaDeviceSynchronize();                                \
        return static_cast<int>(e);                                                       \
    }

#else

#define MOE_TRACE_ENTRY(slot) \
    do {                      \
    } while (0)
#define MOE_TRACE_TILE_FIRST(slot, ti, e, tt, n, rb) \
    do {                                             \
    } while (0)
#define MOE_TRACE_TILE_LAST(slot, ti) \
    do {                              \
    } while (0)
#define MOE_TRACE_READER(name)

#endif
