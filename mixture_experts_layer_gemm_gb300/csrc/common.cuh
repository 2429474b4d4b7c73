// common.cuh -- device helpers shared by the library's kernels (not by the
// oracle, which has none of this code).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kMaxExperts = 64;
constexpr int kMaxTopK = 8;

// Bits of the layer's device error word.
enum : uint32_t {
    kErrExpertId = 1u << 0,     // expert id outside [0, E): routed to expert 0
    kErrDuplicateId = 1u << 1,  // the same expert twice in one token's top-k
    kErrGatherIndex = 1u << 2,  // gather index outside [0, T*k): access skipped
    kErrOffsets = 1u << 3,      // offsets not monotone / out of range: clamped
    kErrWaitTimeout = 1u << 4,  // a bounded device wait gave up
    kErrTmemAlloc = 1u << 5,    // tensor-memory allocation did not succeed
};

__device__ __forceinline__ void flag_error(uint32_t *err, uint32_t bits) {
    if (err) atomicOr(err, bits);
}

// ---- element conversions --------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&r);
}

// ---- memory access ----------------------------------------------------------
// 16-byte load through the read-only path (data no kernel of the launch writes).
__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

// ---- legacy warp-level tensor-core MMA -----------------------------------
// D[16x8] += A[16x16] * B[16x8], bf16 inputs, fp32 accumulate.
// Fragment ownership (g = lane/4, t = lane%4):
//   a0 = A[g][2t..2t+1]   a1 = A[g+8][2t..2t+1]
//   a2 = A[g][2t+8..+9]   a3 = A[g+8][2t+8..+9]
//   b0 = B[2t..2t+1][g]   b1 = B[2t+8..+9][g]
//   d0,d1 = D[g][2t..2t+1]  d2,d3 = D[g+8][2t..2t+1]
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same with fp16 inputs (same fragment ownership).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four signed int8 values b (one word, byte 0 first) -> two fp16x2 words
// holding 1152 + b for bytes (0,1) and (2,3), exactly: flipping the sign bit
// gives the byte u = b + 128 in [0, 255], and the fp16 bit pattern 0x6400 | u
// is 1024 + u (exponent 2^10, u in the low bits of the ten-bit mantissa).
// Three instructions per word; the constant 1152 is taken out after the dot
// product (1152 times the sum of the activations).
__device__ __forceinline__ void i8x4_to_f16x2x2_biased(uint32_t v, uint32_t &lo, uint32_t &hi) {
    const uint32_t u = v ^ 0x80808080u;
    lo = __byte_perm(u, 0x64646464u, 0x4140);  // {u0, 0x64, u1, 0x64}
    hi = __byte_perm(u, 0x64646464u, 0x4342);  // {u2, 0x64, u3, 0x64}
}
constexpr float kI8F16Bias = 1152.0f;

// Power-of-two scaling of a row of bf16 activations into fp16 for the int8
// paths whose MMAs run in fp16: the shift s puts the row's largest magnitude mx
// in [2^14, 2^15), so every bf16 value of the row whose scaled magnitude is at
// least 2^-17 (all within a factor 2^31 of mx) is an exact fp16 value.  A row of
// zeros, or one holding an infinity or NaN, keeps s = 0.
__device__ __forceinline__ int f16_row_shift(float mx) {
    const int eb = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu);
    const int sh = (eb == 0 || eb == 255) ? 0 : eb - 127 - 14;
    return sh < -100 ? -100 : (sh > 113 ? 113 : sh);
}
__device__ __forceinline__ float pow2f(int e) {  // 2^e for e in [-126, 127]
    return __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
}

// Four signed int8 values (one 32-bit word, byte 0 first) -> two bf16x2 words
// holding bytes (0,1) and (2,3), exactly, with byte permutes and one packed
// bf16 FMA per pair (no int-to-float or float-to-bf16 conversions).
// A two's-complement byte b with low seven bits l and sign bit s is
// l - 128 s.  The bf16 bit pattern 0x4300 | l is 128 + l (exponent 2^7, l in
// the seven mantissa bits), and 0x4300 | (s << 7) is 128 + 128 s (0x4380 is
// 2^8).  Their difference, l - 128 s, lies in [-128, 127], so the packed
// subtraction (an FMA by -1) is exact.
__device__ __forceinline__ void i8x4_to_bf16x2x2(uint32_t v, uint32_t &lo, uint32_t &hi) {
    const uint32_t mag = v & 0x7F7F7F7Fu;
    const uint32_t sgn = v & 0x80808080u;
    const uint32_t x_lo = __byte_perm(mag, 0x43434343u, 0x4140);  // {b0, 0x43, b1, 0x43}
    const uint32_t x_hi = __byte_perm(mag, 0x43434343u, 0x4342);  // {b2, 0x43, b3, 0x43}
    const uint32_t y_lo = __byte_perm(sgn, 0x43434343u, 0x4140);
    const uint32_t y_hi = __byte_perm(sgn, 0x43434343u, 0x4342);
    const uint32_t minus_one = 0xBF80BF80u;  // bf16x2 (-1, -1)
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(lo) : "r"(y_lo), "r"(minus_one), "r"(x_lo));
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(hi) : "r"(y_hi), "r"(minus_one), "r"(x_hi));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// ---- mbarrier and bulk asynchronous copies (TMA engine) -------------------------
// Waits are bounded: after kWaitLimit polls the caller gives up and reports.
constexpr uint32_t kWaitLimit = 1u << 22;

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async proxy before first use.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy, tensor core) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of a phase.  A try_wait on a phase that has already
// completed returns at once in isolation (~23 cycles), but costs ~235 cycles
// when issued by a thread with tensor-core MMAs or commits in flight, which
// is exactly what the MMA-issuing threads do between stages; test_wait stays
// at ~23 cycles there (measured: an int8 MMA issuer's stage, two ready waits
// plus 8 MMAs and 2 commits, 919 cycles with try_wait, 526 with test_wait).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// true when the phase with the given parity completed, false after the limit.
// A completed phase is caught by the cheap test; otherwise the thread polls
// with try_wait, which may suspend it and so leaves issue slots to the
// other warps.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_test_wait(bar, parity)) return true;
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// The same wait by spinning on test_wait, for a single thread on the critical
// path (an MMA issuer) that should notice the phase as soon as it completes.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t *bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_test_wait(bar, parity)) return true;
    return false;
}

// Global -> shared bulk copy (no tensor map); both addresses 16-byte aligned,
// size a multiple of 16.  Completion is counted on `bar` in bytes.
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gsrc, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// The same copy for data read once per launch (streamed expert weights): the
// lines are marked first to go from L2, so that what the neighbouring
// launches reuse (activations, partial sums) stays resident.
__device__ __forceinline__ void bulk_g2s_once(void *smem_dst, const void *gsrc, uint32_t bytes,
                                              uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .b64 pol;\n\t"
        "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "pol;\n\t}" ::"r"(smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// ---- programmatic dependent launch -----------------------------------------------
// Kernels on the forward path are launched so that each may start while its
// predecessor in the stream finishes.  Protocol: a kernel calls pdl_wait()
// before it reads anything its predecessor writes or writes anything its
// predecessor reads, and calls pdl_trigger() only after that wait.  Then a
// kernel can overlap only its immediate predecessor, and everything issued
// two kernels back has completed when it starts.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch parameters are never written by a predecessor, but a CTA's first
// reads of them go to memory (measured: about a microsecond).  A kernel names
// the parameters it needs soon after its dependency wait in touch_params()
// before that wait, so those reads are issued, and overlap the predecessor's
// tail, instead of starting after it.
__device__ __forceinline__ void touch_one(const void *p) { asm volatile("" ::"l"(p)); }
__device__ __forceinline__ void touch_one(int v) { asm volatile("" ::"r"(v)); }
__device__ __forceinline__ void touch_one(unsigned v) { asm volatile("" ::"r"(v)); }
__device__ __forceinline__ void touch_one(size_t v) { asm volatile("" ::"l"(v)); }
template <typename... Ts>
__device__ __forceinline__ void touch_params(const Ts &...v) {
    (touch_one(v), ...);
}

// Starts [p, p + bytes) on its way from global memory into L2, in 16 KB bulk
// prefetches (no destination and nothing to wait for).  p 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void *p, size_t bytes) {
    const char *c = static_cast<const char *>(p);
    for (size_t o = 0; o < bytes; o += 16384) {
        const uint32_t n = static_cast<uint32_t>(bytes - o < 16384 ? bytes - o : 16384);
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c + o), "r"(n) : "memory");
    }
}
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier over a subset of the CTA's warps.
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads, so
// that every participant takes the same decision.
__device__ __forceinline__ int named_sync_or(uint32_t id, uint32_t threads, int pred) {
    int out;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.s32 pi, %1, 0;\n\t"
        "barrier.cta.red.or.pred po, %2, %3, pi;\n\t"
        "selp.s32 %0, 1, 0, po;\n\t}"
        : "=r"(out)
        : "r"(pred), "r"(id), "r"(threads)
        : "memory");
    return out;
}

}  // namespace moe
