// Device helpers shared by the library's kernels: the summation tree, the
// binary32 exponential, mbarrier / bulk-copy / programmatic-dependent-launch
// wrappers in inline PTX, and the device status word.
//
// Every floating-point step that must match the tree-order definition is a
// single correctly rounded operation (__fadd_rn / __fmul_rn / __fdiv_rn /
// __fsqrt_rn or a packed .rn f32x2 op), so the compiler cannot contract or
// reorder it.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace abg {

// Device status word (bit 0: a bounded wait timed out).  Kernels only OR
// bits into it.  Each translation unit has its own word (the library is built
// without relocatable device code) and exports a host function that reads it;
// abg_device_status() combines them.
static __device__ unsigned int g_status;
constexpr unsigned kStatusTimeout = 1u;
// A bounded wait gives up after this many nanoseconds of %globaltimer (no
// legitimate wait here lasts more than microseconds).
constexpr unsigned long long kWaitLimitNs = 500000000ull;

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- PDL ------
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before its predecessor finishes; grid_dep_wait()
// blocks until the predecessor grid has completed and its writes are
// visible; grid_dep_launch() lets the next launch start.  Every kernel here
// calls grid_dep_launch() only after its own grid_dep_wait() has returned, so
// a chain of launches never has more than two grids resident and waiting
// (signalling at kernel start let a long chain fill the GPU with grids all
// waiting on their predecessors, which hung).  Both are no-ops for a kernel
// launched without the attribute.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------ mbarrier -----
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
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
// try_wait that may suspend the thread until the phase completes or
// `hint_ns` nanoseconds pass, so a waiting warp does not spin on issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
constexpr uint32_t kSleepHintNs = 100000;

// Waits for the phase with the given parity to complete.  Returns false (and
// sets the timeout bit) if it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
        if (globaltimer() - t0 > kWaitLimitNs) {
            atomicOr(&g_status, kStatusTimeout | (1u << 7));
            return false;
        }
    }
}

// ------------------------------------------------------------ bulk copy ----
// One-dimensional bulk copy global -> shared, completing on an mbarrier's
// transaction count.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// L2 policy for data read once (packed weights): evict first.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Named barrier over `threads` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_bar(unsigned id, unsigned threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------- packed f32x2 ------
// Two independent binary32 operations, each rounded to nearest even (no
// flush to zero); element-wise identical to the scalar __f*_rn intrinsics.
// Unlike the scalar intrinsics, a packed multiply followed by a packed add
// may be fused into one packed FMA by the compiler, so exact code never
// feeds mul2's result into add2.
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)));
    return *reinterpret_cast<float2 *>(&d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)));
    return *reinterpret_cast<float2 *>(&d);
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)),
          "l"(*reinterpret_cast<unsigned long long *>(&c)));
    return *reinterpret_cast<float2 *>(&d);
}

// ------------------------------------------------------------- the tree ----
// The summation order is a balanced pairwise tree in index order with an odd
// last element carried up.  Carrying an element unchanged is the same as
// adding -0.0 to it (x + -0 == x for every x, including -0 and NaN), so the
// tree over m leaves equals the full power-of-two tree over the leaves padded
// with -0.0 to the next power of two.  The warp butterfly below realizes the
// power-of-two tree across lanes: after the step with distance d, lane i holds
// the sum of the aligned block of 2d lanes that contains i.
constexpr float kNegZero = -0.0f;

template <int kWidth>
__device__ __forceinline__ float warp_tree(float v) {
#pragma unroll
    for (int d = 1; d < kWidth; d <<= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, d));
    return v;
}

// Tree over buf[0..m) in shared memory by ONE warp, in place (buf must hold
// next_pow2(m) slots; slots m.. are overwritten with -0).  Returns the sum to
// every lane of that warp.
__device__ __forceinline__ float warp_tree_smem(float *buf, int m) {
    const int lane = threadIdx.x & 31;
    int p = 1;
    while (p < m) p <<= 1;
    for (int i = m + lane; i < p; i += 32) buf[i] = kNegZero;
    __syncwarp();
    for (int h = 1; h < p; h <<= 1) {
        for (int i = lane * 2 * h; i < p; i += 64 * h) buf[i] = __fadd_rn(buf[i], buf[i + h]);
        __syncwarp();
    }
    const float s = buf[0];
    __syncwarp();
    return s;
}

// ------------------------------------------------------------------ EXP ----
// The library's binary32 exponential (ABG_TREE mode), from its written
// definition: NaN -> NaN; v > 89 -> +inf; v < -104 -> +0; otherwise
//   k  = round-half-even(v * L2E)
//   rr = (v + (-k)*LN2HI) + (-k)*LN2LO
//   p  = Horner(rr; RN(1/0!), ..., RN(1/7!))   (multiply, then add)
//   result = p * 2^k, scaled in two exact-then-rounded steps outside
//            the normal exponent range so it is rounded once.
// L2E = RN(log2 e); LN2HI = RN(ln 2) with its low 12 significand bits cleared
// (so k*LN2HI is exact); LN2LO = RN(ln 2 - LN2HI).
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((e + 127) << 23); }

__device__ __forceinline__ float exp_tree(float v) {
    if (v != v) return v;
    if (v > 89.0f) return __int_as_float(0x7f800000);
    if (v < -104.0f) return 0.0f;
    const float kL2E = __int_as_float(0x3FB8AA3B);
    const float kLn2Hi = __int_as_float(0x3F317000);
    const float kLn2Lo = __int_as_float(0x3805FDF4);
    const float kf = rintf(__fmul_rn(v, kL2E));
    const int k = static_cast<int>(kf);
    const float nk = -kf;
    const float rr = __fadd_rn(__fadd_rn(v, __fmul_rn(nk, kLn2Hi)), __fmul_rn(nk, kLn2Lo));
    float p = __int_as_float(0x39500D01);                  // 1/7!
    p = __fadd_rn(__fmul_rn(p, rr), __int_as_float(0x3AB60B61));  // 1/6!
    p = __fadd_rn(__fmul_rn(p, rr), __int_as_float(0x3C088889));  // 1/5!
    p = __fadd_rn(__fmul_rn(p, rr), __int_as_float(0x3D2AAAAB));  // 1/4!
    p = __fadd_rn(__fmul_rn(p, rr), __int_as_float(0x3E2AAAAB));  // 1/3!
    p = __fadd_rn(__fmul_rn(p, rr), __int_as_float(0x3F000000));  // 1/2!
    p = __fadd_rn(__fmul_rn(p, rr), 1.0f);                         // 1/1!
    p = __fadd_rn(__fmul_rn(p, rr), 1.0f);                         // 1/0!
    if (k > 127) return __fmul_rn(__fmul_rn(p, pow2i(127)), pow2i(k - 127));
    if (k < -126) return __fmul_rn(__fmul_rn(p, pow2i(k + 126)), pow2i(-126));
    return __fmul_rn(p, pow2i(k));
}

// SwiGLU element: silu(g) * u with silu(g) = g / (1 + exp(-g)).
template <bool kTree>
__device__ __forceinline__ float swiglu(float g, float u) {
    if (kTree) {
        const float e = exp_tree(-g);
        return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, e)), u);
    }
    return g / (1.0f + __expf(-g)) * u;
}

}  // namespace abg
